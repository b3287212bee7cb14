"""The timeline build (SV_TRACE=1) on the GPU: its outputs equal the default
build's, and its records obey what every launch must show -- each CTA placed,
started and gone once per launch; the sampling item kernel retires each
sequence's items and writes one decision per sequence; the logits workers
record one mass decision per sequence (every sequence ends in one draw), at
least one normaliser decision per sequence, and one or two per group.  Tracing is a diagnostic build:
these tests check that it records what happened, not how fast."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import speculative_decoding_verification_08_gb300 as sv
from speculative_decoding_verification_08_gb300 import _build
from speculative_decoding_verification_08_gb300 import trace as T
from speculative_decoding_verification_08_gb300.inputs import make_inputs

EV = {n: i for i, n in enumerate(T.TRACE_EVENTS)}
B, K, V = 64, 4, 32000


@pytest.fixture(scope="module")
def libs(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    path = tmp_path_factory.mktemp("trace") / "libspecverify_trace.so"
    return sv.load(), sv._declare(ctypes.CDLL(_build.build_trace(str(path))))


def _fields(records):
    _, t, ev, cta, arg = T._fields(records)
    return t, ev, cta, arg


def _run(lib, fn, stream, bt, zp=None, zq=None):
    dev = bt.p.device
    P = lambda x: ctypes.c_void_p(0 if x is None else x.data_ptr())
    sh = ctypes.c_void_p(stream.cuda_stream)
    nb = lib.sv_workspace_size(B, K, V)
    ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
    assert lib.sv_workspace_init(P(ws), nb, sh) == 0
    n = torch.full((B,), -7, dtype=torch.int32, device=dev)
    nx = torch.full((B,), -7, dtype=torch.int32, device=dev)
    if fn == "sample":
        rc = lib.sv_verify_sample(P(bt.p), V, P(bt.q), V, P(bt.t), P(bt.u_acc), P(bt.u_res), B, K, V,
                                  P(n), P(nx), P(ws), nb, sh)
    else:
        rc = lib.sv_verify_sample_logits(P(zp), V, P(zq), V, P(bt.t), P(bt.u_acc), P(bt.u_res), B, K, V,
                                         ctypes.c_float(1.0), P(n), P(nx), P(ws), nb, sh)
    assert rc == 0
    st = ctypes.c_uint32(0)
    assert lib.sv_get_status(P(ws), sh, ctypes.byref(st)) == 0
    stream.synchronize()
    assert st.value == 0
    return n.cpu().numpy(), nx.cpu().numpy()


def _per_launch_ctas(records, launches):
    parts = T.split_launches(records)
    assert len(parts) == launches
    for r in parts:
        _, ev, cta, _ = _fields(r)
        ctas = np.unique(cta)
        for name in ("cta_placed", "cta_begin", "cta_end"):
            m = ev == EV[name]
            assert np.array_equal(np.sort(cta[m]), ctas), name  # once per CTA
    return parts


def test_sampling_timeline_of_two_launches(libs):
    base, tr = libs
    dev = torch.device("cuda", 0)
    bt = make_inputs(3, dev, seed=515, B=B, K=K, V=V)
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    want = _run(base, "sample", stream, bt)
    sv.trace_reset(stream, tr)
    got = [_run(tr, "sample", stream, bt) for _ in range(2)]
    rec = sv.trace_read(stream, tr)
    for g in got:
        assert np.array_equal(g[0], want[0]) and np.array_equal(g[1], want[1])
    for r in _per_launch_ctas(rec, 2):
        _, ev, cta, arg = _fields(r)
        dec = np.sort(arg[ev == EV["decide_end"]])
        assert np.array_equal(dec, np.arange(B)), "one decision per sequence"
        assert set(arg[ev == EV["item_retired"]]) == set(range(B))
    tl = sv.trace_timeline(rec)
    assert len(tl["launches"]) == 2 and len(tl["between"]) == 1


def test_logits_timeline(libs):
    base, tr = libs
    dev = torch.device("cuda", 0)
    bt = make_inputs(3, dev, seed=516, B=B, K=K, V=V)
    zp, zq = torch.log(bt.p), torch.log(bt.q)
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    want = _run(base, "logits", stream, bt, zp, zq)
    sv.trace_reset(stream, tr)
    got = _run(tr, "logits", stream, bt, zp, zq)
    rec = sv.trace_read(stream, tr)
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
    (r,) = _per_launch_ctas(rec, 1)
    _, ev, cta, arg = _fields(r)
    dec = ev == EV["lg_decide"]
    seq, pos, kind = arg & 0xFFFF, (arg >> 16) & 0xFF, (arg >> 24) & 0xFF
    mass = dec & (kind == 2)
    assert np.array_equal(np.sort(seq[mass]), np.arange(B)), "one draw per sequence"
    # the draw is at the position where the sequence stopped: n, or K after all accepted
    assert np.array_equal(pos[mass][np.argsort(seq[mass])], want[0])
    norm = dec & (kind == 1)
    assert set(seq[norm]) == set(range(B))
    # a normaliser group's last arrival is recorded, then its merge, then one
    # decision per position it covers (one or two)
    last = int((ev == EV["lg_last"]).sum())
    assert last <= int(norm.sum()) <= 2 * last
    assert (ev == EV["lg_merged"]).sum() == last
    assert (ev == EV["lg_claim"]).sum() >= (ev == EV["lg_issued"]).sum() > 0
