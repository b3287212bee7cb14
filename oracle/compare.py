"""Comparison helpers shared by the GPU parity tests, smoke() and the bench.

Greedy outputs and every accept decision (n_accepted) must match the oracle
bit for bit.  A drawn token (resample or bonus) may differ from the oracle's
only when the oracle's threshold T = u * R lies within BOUNDARY_TOL * R of the
running mass C_k at a boundary between the two answers: the CUDA path sums
masses in double-fp32 arithmetic, the oracle in fp64, and the two sums can
order T differently only inside that band.  Such cases are counted.
"""
from __future__ import annotations

import numpy as np

from . import get as _get_oracle

BOUNDARY_TOL = 1e-9


def draw_distribution(p, q, mode, K, b, n):
    """Running masses C and total R of the distribution the oracle draws from
    for sequence b stopped at n (residual of row n, its p row if that residual
    has no mass, or the bonus row p_K)."""
    if mode == 1 and n < K:
        C, R = _get_oracle().residual_cumsum(p[b, n], q[b, n])
        if R > 0:
            return C, R
        return _get_oracle().residual_cumsum(p[b, n])
    return _get_oracle().residual_cumsum(p[b, K])


def explained(C, R, T, j_oracle, j_gpu, tol=BOUNDARY_TOL):
    """True if the GPU's token j_gpu differs from j_oracle only because T sits
    within tol*R of a CDF boundary between them (and j_gpu has mass)."""
    if j_gpu < 0 or j_gpu >= len(C) or j_oracle < 0:
        return False
    prev = C[j_gpu - 1] if j_gpu > 0 else 0.0
    if not C[j_gpu] > prev:
        return False
    if j_gpu > j_oracle:
        return C[j_gpu - 1] - T <= tol * R
    return T - C[j_gpu] <= tol * R


def compare(p, q, u_res, mode, K, n_ref, next_ref, n_gpu, next_gpu, st_ref=None, st_gpu=None):
    """Checks GPU outputs against the oracle's; returns the list of
    boundary-explained resample mismatches [(b, j_oracle, j_gpu)].  Raises
    AssertionError for any other difference."""
    n_ref, next_ref = np.asarray(n_ref), np.asarray(next_ref)
    n_gpu, next_gpu = np.asarray(n_gpu), np.asarray(next_gpu)
    bad_n = np.nonzero(n_ref != n_gpu)[0]
    assert bad_n.size == 0, (f"n_accepted differs at {bad_n[:10].tolist()}: oracle "
                             f"{n_ref[bad_n[:10]].tolist()} gpu {n_gpu[bad_n[:10]].tolist()}")
    if st_ref is not None and st_gpu is not None:
        assert st_ref == st_gpu, f"status oracle {st_ref} gpu {st_gpu}"
    boundary = []
    mism = np.nonzero(next_ref != next_gpu)[0]
    for b in mism.tolist():
        m = int(mode[b]) if np.ndim(mode) else int(mode)
        assert m == 1, f"greedy next_token differs at seq {b}: {next_ref[b]} vs {next_gpu[b]}"
        C, R = draw_distribution(p, q, m, K, b, int(n_ref[b]))
        T = float(u_res[b]) * R
        ok = explained(C, R, T, int(next_ref[b]), int(next_gpu[b]))
        assert ok, (f"seq {b}: next_token oracle {next_ref[b]} gpu {next_gpu[b]} is not a "
                    f"boundary case (T={T!r}, R={R!r})")
        boundary.append((b, int(next_ref[b]), int(next_gpu[b])))
    return boundary


# Sampling from logits: the kernels warp with fp32 exp2.approx, the oracle with
# an fp64 softmax.  Each mass then carries ~1e-6 relative error at most
# (exp2.approx ~2^-22, the fp32 argument (z - max)/T, the fp32 normaliser), so
# an accept decision may differ only where |u*q - p| <= ACCEPT_TOL_LOGITS * p,
# and a drawn token only where u*R lies within DRAW_TOL_LOGITS (normalised
# mass) of a boundary between the two answers.
ACCEPT_TOL_LOGITS = 1e-5
DRAW_TOL_LOGITS = 2e-6


def compare_logits(zp, zq, tau, t, u_acc, u_res, n_ref, next_ref, n_gpu, next_gpu):
    """Checks GPU outputs of sampling-from-logits against the oracle's; returns
    the explained differences [(b, kind)]: 'accept' near-threshold decisions and
    'draw' near-boundary tokens.  Raises AssertionError on any other."""
    import oracle
    explained = []
    K = t.shape[1]
    for b in np.nonzero((n_ref != n_gpu) | (next_ref != next_gpu))[0]:
        if n_ref[b] != n_gpu[b]:
            i = int(min(n_ref[b], n_gpu[b]))
            x = int(t[b, i])
            p = oracle.softmax(zp[b, i], tau)[x]
            q = oracle.softmax(zq[b, i], tau)[x]
            margin = abs(float(u_acc[b, i]) * q - p)
            assert margin <= ACCEPT_TOL_LOGITS * p, (
                f"seq {b}: n oracle {n_ref[b]} gpu {n_gpu[b]}, accept margin {margin / p:.3e}")
            explained.append((int(b), "accept"))
            continue
        n = int(n_ref[b])
        if n < K:
            r = np.maximum(oracle.softmax(zp[b, n], tau) - oracle.softmax(zq[b, n], tau), 0.0)
        else:
            r = oracle.softmax(zp[b, K], tau)
        C = np.cumsum(r)
        T = float(u_res[b]) * C[-1]
        j = int(next_gpu[b])
        assert 0 <= j < r.shape[0] and r[j] > 0, f"seq {b}: gpu token {j} has no mass"
        lo, hi = sorted((int(next_ref[b]), j))
        assert np.abs(C[lo:hi] - T).min() <= DRAW_TOL_LOGITS, (
            f"seq {b}: token oracle {next_ref[b]} gpu {j} not at a boundary")
        explained.append((int(b), "draw"))
    return explained
