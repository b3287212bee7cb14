"""The allocation-free sampling entry point (sv_verify_sample_noalloc).

Some callers cannot allocate device memory while they enqueue work: a
framework hook or plugin interface that forbids allocation at enqueue time, or
a serving loop that must not risk a cudaMalloc that synchronises the device or
fails under memory pressure.  For them the library offers a sampling call
that uses a fixed 4 MiB scratch array compiled into the library instead of a
caller workspace.  This file checks, through the C ABI, that two calls in a
row give the results of the regular sv_verify_sample call (same tolerance as
the other parity tests), and that sizes beyond the array are refused.

It is collected last on purpose and builds what it needs, so it also runs on
its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

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


def _noalloc(lib, bt, n, nx):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.sv_verify_sample_noalloc(_P(bt.p), bt.V, _P(bt.q), bt.V, _P(bt.t), _P(bt.u_acc),
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


def test_two_calls_match_the_workspace_entry_point(lib):
    # two different batches back to back: the second call must not be disturbed
    # by what the first left in the shared scratch array
    batches = [make_inputs(3, "cuda", seed=9001, B=256, V=128256, K=5),
               make_inputs(5, "cuda", seed=9002, B=40, V=70001, K=9)]
    outs = [(torch.full((bt.B,), -7, dtype=torch.int32, device="cuda"),
             torch.full((bt.B,), -7, dtype=torch.int32, device="cuda")) for bt in batches]
    for bt, (n, nx) in zip(batches, outs):
        assert _noalloc(lib, bt, n, nx) == 0
    torch.cuda.synchronize()
    for bt, (n, nx) in zip(batches, outs):
        n_ref, nx_ref = _regular(lib, bt)
        p, q, t, ua, ur, md = bt.numpy()
        compare(p, q, ur, 1, bt.K, n_ref, nx_ref, n.cpu().numpy(), nx.cpu().numpy())
        assert np.all(n.cpu().numpy() >= 0)


def test_sizes_beyond_the_scratch_are_refused(lib):
    B, K, V = 8192, 5, 128256
    assert sv.workspace_size(B, K, V) > sv.NOALLOC_SCRATCH_BYTES
    dummy = ctypes.c_void_p(4096)   # never dereferenced: the size check comes first
    rc = lib.sv_verify_sample_noalloc(dummy, V, dummy, V, dummy, dummy, dummy, B, K, V, dummy,
                                      dummy, None)
    assert rc == sv.SV_ETOOLARGE
    assert "4 MiB" in sv.status_string(rc)
