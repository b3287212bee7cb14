"""The allocation-free sampling entry point (sv_verify_sample_noalloc).

Some callers cannot allocate device memory while they enqueue work: a
framework hook or plugin interface that forbids allocation at enqueue time, or
a serving loop that must not risk a cudaMalloc that synchronises the device or
fails under memory pressure.  For them the library offers a sampling call
that uses a fixed 4 MiB scratch array compiled into the library instead of a
caller workspace.  This file checks, through the C ABI, that two calls in a
row give the results of the regular sv_verify_sample call and of the oracle
(same tolerance as the other parity tests: decisions exact, drawn tokens up
to counted boundary cases), on device rows (the single-launch kernel) and on
rows in page-locked host memory (the three-launch chain, which uses more of
the shared array); that a call with preallocated outputs changes neither
torch's allocations nor the device's free memory; and that sizes beyond the
array are refused.

It is collected last on purpose and builds what it needs, so it also runs on
its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_08_gb300 as sv
from oracle.compare import compare
from speculative_decoding_verification_08_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.build()
    return sv.load()


def _P(x):
    return ctypes.c_void_p(0 if x is None else x.data_ptr())


def _noalloc(lib, bt, n, nx, p=None, q=None):
    p = bt.p if p is None else p
    q = bt.q if q is None else q
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.sv_verify_sample_noalloc(_P(p), bt.V, _P(q), bt.V, _P(bt.t), _P(bt.u_acc),
                                        _P(bt.u_res), bt.B, bt.K, bt.V, _P(n), _P(nx), stream)


def _regular(lib, bt):
    n = torch.empty(bt.B, dtype=torch.int32, device="cuda")
    nx = torch.empty(bt.B, dtype=torch.int32, device="cuda")
    ws = sv.Workspace(bt.B, bt.K, bt.V)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.sv_verify_sample(_P(bt.p), bt.V, _P(bt.q), bt.V, _P(bt.t), _P(bt.u_acc),
                              _P(bt.u_res), bt.B, bt.K, bt.V, _P(n), _P(nx), ws.ptr, ws.nbytes,
                              stream)
    assert rc == 0
    return n.cpu().numpy(), nx.cpu().numpy()


def _outputs(B):
    return (torch.full((B,), -7, dtype=torch.int32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda"))


def _check(lib, bt, n, nx, label):
    """Against the workspace entry point and against the oracle."""
    p, q, t, ua, ur, md = bt.numpy()
    n_gpu, nx_gpu = n.cpu().numpy(), nx.cpu().numpy()
    n_ref, nx_ref = _regular(lib, bt)
    compare(p, q, ur, 1, bt.K, n_ref, nx_ref, n_gpu, nx_gpu, label=f"{label} vs workspace call")
    n0, x0, s0 = oracle.verify_sample(p, q, t, ua, ur, nthreads=8)
    assert s0 == 0
    compare(p, q, ur, 1, bt.K, n0, x0, n_gpu, nx_gpu, label=f"{label} vs oracle")
    assert np.all(n_gpu >= 0) and np.all(nx_gpu >= 0)


def test_two_calls_match_the_workspace_entry_point_and_the_oracle(lib):
    # two different batches back to back: the second call must not be disturbed
    # by what the first left in the shared scratch array
    batches = [make_inputs(3, "cuda", seed=9001, B=256, V=128256, K=5),
               make_inputs(5, "cuda", seed=9002, B=40, V=70001, K=9)]
    outs = [_outputs(bt.B) for bt in batches]
    for bt, (n, nx) in zip(batches, outs):
        assert _noalloc(lib, bt, n, nx) == 0
    torch.cuda.synchronize()
    for i, (bt, (n, nx)) in enumerate(zip(batches, outs)):
        _check(lib, bt, n, nx, f"no-alloc call {i}")


def test_rows_in_host_memory_take_the_chain_through_the_array(lib):
    # page-locked rows: the scan / stream / decide chain, whose per-sequence
    # state and block sums also live in the shared array; two calls in a row
    batches = [make_inputs(3, "cuda", seed=9101, B=24, V=50000, K=5),
               make_inputs(4, "cuda", seed=9102, B=16, V=30011, K=7)]
    outs = [_outputs(bt.B) for bt in batches]
    pinned = [(bt.p.cpu().pin_memory(), bt.q.cpu().pin_memory()) for bt in batches]
    for bt, (n, nx), (hp, hq) in zip(batches, outs, pinned):
        assert _noalloc(lib, bt, n, nx, hp, hq) == 0
        assert sv.last_kernel_count() == 3, "expected the three-launch chain"
    torch.cuda.synchronize()
    for i, (bt, (n, nx)) in enumerate(zip(batches, outs)):
        _check(lib, bt, n, nx, f"no-alloc host rows {i}")


def test_a_call_allocates_nothing(lib):
    bt = make_inputs(3, "cuda", seed=9201, B=128, V=128256, K=5)
    n, nx = _outputs(bt.B)
    assert _noalloc(lib, bt, n, nx) == 0   # loads the device code if nothing has yet
    torch.cuda.synchronize()
    before = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(),
              torch.cuda.mem_get_info()[0])
    for _ in range(3):
        assert _noalloc(lib, bt, n, nx) == 0
    torch.cuda.synchronize()
    after = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved(),
             torch.cuda.mem_get_info()[0])
    assert after == before
    _check(lib, bt, n, nx, "no-alloc repeated")


def test_sizes_beyond_the_scratch_are_refused(lib):
    B, K, V = 8192, 5, 128256
    assert sv.workspace_size(B, K, V) > sv.NOALLOC_SCRATCH_BYTES
    dummy = ctypes.c_void_p(4096)   # never dereferenced: the size check comes first
    rc = lib.sv_verify_sample_noalloc(dummy, V, dummy, V, dummy, dummy, dummy, B, K, V, dummy,
                                      dummy, None)
    assert rc == sv.SV_ETOOLARGE
    assert "4 MiB" in sv.status_string(rc)
