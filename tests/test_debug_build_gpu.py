"""The debug build of the library (compiled with SV_DEBUG=1).

It checks every input row before a call's kernels and raises
SV_STATUS_BAD_VALUE for a probability that is negative, NaN or infinite (for
logits: NaN or infinite).  On valid inputs it must verify exactly as the
oracle does, with no status bit.  The invalid values are planted only in rows
the rule never reads for that sequence (the bonus row of a sequence that
rejected a draft, a draft row past the first rejection away from its draft
token), so the outputs stay those of the clean inputs while the check still
has to find them.  Needs a GPU (-m gpu)."""
import ctypes
import os
import tempfile

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_08_gb300 as sv
from oracle.compare import compare
from speculative_decoding_verification_08_gb300 import _build
from speculative_decoding_verification_08_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

BAD = sv.STATUS_BAD_VALUE


@pytest.fixture(scope="module")
def dbg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.build()
    sv.load()
    out = os.path.join(tempfile.mkdtemp(prefix="specverify_debug"), "libspecverify_debug.so")
    return sv._declare(ctypes.CDLL(_build.build_debug(out)))


def _P(x):
    return ctypes.c_void_p(0 if x is None else x.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _outs(B):
    n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    return n, torch.full((B,), -7, dtype=torch.int32, device="cuda")


def _sample(lib, p, q, t, ua, ur, ws):
    B, K, V = t.shape[0], t.shape[1], p.shape[2]
    n, nx = _outs(B)
    assert lib.sv_verify_sample(_P(p), V, _P(q), V, _P(t), _P(ua), _P(ur), B, K, V, _P(n),
                                _P(nx), ws.ptr, ws.nbytes, _stream()) == 0
    return n.cpu().numpy(), nx.cpu().numpy(), ws.status()


def _greedy(lib, p, t, ws):
    B, K, V = t.shape[0], t.shape[1], p.shape[2]
    n, nx = _outs(B)
    assert lib.sv_verify_greedy(_P(p), V, _P(t), B, K, V, _P(n), _P(nx), ws.ptr, ws.nbytes,
                                _stream()) == 0
    return n.cpu().numpy(), nx.cpu().numpy(), ws.status()


def _logits(lib, zp, zq, t, ua, ur, ws, tau=1.0):
    B, K, V = t.shape[0], t.shape[1], zp.shape[2]
    n, nx = _outs(B)
    assert lib.sv_verify_sample_logits(_P(zp), V, _P(zq), V, _P(t), _P(ua), _P(ur), B, K, V,
                                       ctypes.c_float(tau), _P(n), _P(nx), ws.ptr, ws.nbytes,
                                       _stream()) == 0
    return n.cpu().numpy(), nx.cpu().numpy(), ws.status()


def _far_from(t, V):
    """An index of the row other than the draft token t."""
    return (int(t) + V // 2) % V


def test_valid_inputs_verify_as_the_oracle_with_no_flag(dbg):
    bt = make_inputs(3, "cuda", seed=4242, B=24, V=5000, K=4)
    ws = sv.Workspace(bt.B, bt.K, bt.V)
    p, q, t, ua, ur, md = bt.numpy()
    n, nx, st = _sample(dbg, bt.p, bt.q, bt.t, bt.u_acc, bt.u_res, ws)
    n0, x0, s0 = oracle.verify_sample(p, q, t, ua, ur)
    compare(p, q, ur, 1, bt.K, n0, x0, n, nx, s0, st)
    n, nx, st = _greedy(dbg, bt.p, bt.t, ws)
    n0, x0, s0 = oracle.verify_greedy(p, t)
    compare(p, q, ur, 0, bt.K, n0, x0, n, nx, s0, st)


@pytest.mark.parametrize("what", ["p_nan", "p_negative", "p_inf", "q_nan"])
def test_bad_values_are_flagged_and_change_nothing_read(dbg, what):
    bt = make_inputs(3, "cuda", seed=5151, B=24, V=5000, K=4)
    B, K, V = bt.B, bt.K, bt.V
    ws = sv.Workspace(B, K, V)
    n_clean, x_clean, st = _sample(dbg, bt.p, bt.q, bt.t, bt.u_acc, bt.u_res, ws)
    assert st == 0
    t = bt.t.cpu().numpy()
    p, q = bt.p.clone(), bt.q.clone()
    if what == "q_nan":
        # a draft row past the first rejection, away from its draft token
        b = int(np.nonzero(n_clean < K - 1)[0][0])
        q[b, K - 1, _far_from(t[b, K - 1], V)] = float("nan")
    else:
        # the bonus row of a sequence that rejected a draft
        b = int(np.nonzero(n_clean < K)[0][0])
        val = {"p_nan": float("nan"), "p_negative": -1e-3, "p_inf": float("inf")}[what]
        p[b, K, V - 1] = val
    n, x, st = _sample(dbg, p, q, bt.t, bt.u_acc, bt.u_res, ws)
    assert st & BAD, (what, st)
    assert np.array_equal(n, n_clean) and np.array_equal(x, x_clean)
    if what != "q_nan":
        # greedy reads p only, and never the bonus row of a sequence that missed
        n_g, x_g, st = _greedy(dbg, bt.p, bt.t, ws)
        assert st == 0
        b = int(np.nonzero(n_g < K)[0][0])
        pg = bt.p.clone()
        pg[b, K, 0] = p[int(np.nonzero(n_clean < K)[0][0]), K, V - 1]
        n2, x2, st = _greedy(dbg, pg, bt.t, ws)
        assert st & BAD, (what, st)
        assert np.array_equal(n2, n_g) and np.array_equal(x2, x_g)


def test_logits_may_be_negative_but_not_nan_or_infinite(dbg):
    bt = make_inputs(3, "cuda", seed=6161, B=16, V=4000, K=3)
    B, K, V = bt.B, bt.K, bt.V
    zp, zq = torch.log(bt.p), torch.log(bt.q)          # every logit is negative
    ws = sv.Workspace(B, K, V)
    n_clean, x_clean, st = _logits(dbg, zp, zq, bt.t, bt.u_acc, bt.u_res, ws)
    assert st == 0
    b = int(np.nonzero(n_clean < K)[0][0])
    for val in (float("nan"), float("inf"), -float("inf")):
        zp2 = zp.clone()
        zp2[b, K, 1] = val                              # a bonus row this sequence never reads
        n, x, st = _logits(dbg, zp2, zq, bt.t, bt.u_acc, bt.u_res, ws)
        assert st & BAD, (val, st)
        assert np.array_equal(n, n_clean) and np.array_equal(x, x_clean)
