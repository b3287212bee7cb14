"""Comparison helpers shared by the GPU parity tests, smoke() and the bench's
CPU-baseline leg (test infrastructure, like the rest of the oracle).

Greedy outputs and every accept decision (n_accepted) must match the oracle
bit for bit.  A drawn token (resample or bonus) may differ from the oracle's
only when the oracle's threshold T = u * R lies within BOUNDARY_TOL * R of the
running mass C_k at a boundary between the two answers: the CUDA path sums
masses in double-fp32 arithmetic, the oracle in fp64, and the two sums can
order T differently only inside that band.  Such cases are counted: every
comparison adds to TALLY (sequences compared, sampled draws among them, and
the boundary cases with their labels), which the test session prints at its
end and smoke() and the bench report.
"""
from __future__ import annotations

import numpy as np

from . import get as _get_oracle

BOUNDARY_TOL = 1e-9

# Running totals over every compare()/compare_logits() call of this process.
TALLY = {"sequences": 0, "draws": 0, "boundary": 0, "logits_accept": 0, "logits_draw": 0,
         "cases": []}


def reset_tally():
    TALLY.update(sequences=0, draws=0, boundary=0, logits_accept=0, logits_draw=0, cases=[])


def tally_line() -> str:
    """One line for a report: sequences compared, sampled draws, boundary cases."""
    t = TALLY
    s = (f"oracle comparisons: {t['sequences']} sequences, {t['draws']} sampled draws; "
         f"boundary-explained draw mismatches (|T - C_k| <= {BOUNDARY_TOL:g} R): {t['boundary']}")
    if t["logits_accept"] or t["logits_draw"]:
        s += (f"; from logits: {t['logits_accept']} near-threshold accept decisions, "
              f"{t['logits_draw']} near-boundary draws")
    return s


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


def classify(p, q, u_res, mode, K, n_ref, next_ref, n_gpu, next_gpu):
    """Sorts every difference between GPU and oracle outputs without raising:
    {"n": sequences whose n_accepted differs, "greedy": greedy sequences whose
    next_token differs, "boundary": [(b, j_oracle, j_gpu)] draws explained by
    the boundary band, "unexplained": [(b, j_oracle, j_gpu, T, R)] other draw
    differences}.  Only "boundary" is allowed."""
    n_ref, next_ref = np.asarray(n_ref), np.asarray(next_ref)
    n_gpu, next_gpu = np.asarray(n_gpu), np.asarray(next_gpu)
    out = {"n": np.nonzero(n_ref != n_gpu)[0].tolist(), "greedy": [], "boundary": [],
           "unexplained": []}
    for b in np.nonzero((next_ref != next_gpu) & (n_ref == n_gpu))[0].tolist():
        m = int(mode[b]) if np.ndim(mode) else int(mode)
        if m != 1:
            out["greedy"].append(b)
            continue
        C, R = draw_distribution(p, q, m, K, b, int(n_ref[b]))
        T = float(u_res[b]) * R
        if explained(C, R, T, int(next_ref[b]), int(next_gpu[b])):
            out["boundary"].append((b, int(next_ref[b]), int(next_gpu[b])))
        else:
            out["unexplained"].append((b, int(next_ref[b]), int(next_gpu[b]), T, R))
    return out


def count(mode, n_seqs, boundary, label=None):
    """Adds one comparison of n_seqs sequences (mode: one rule for all, or per
    sequence) and its boundary cases to TALLY."""
    m = np.asarray(mode)
    draws = (int(n_seqs) if int(m) == 1 else 0) if m.ndim == 0 else int((m == 1).sum())
    TALLY["sequences"] += int(n_seqs)
    TALLY["draws"] += draws
    TALLY["boundary"] += len(boundary)
    if boundary:
        TALLY["cases"].append((label, list(boundary)))


def compare(p, q, u_res, mode, K, n_ref, next_ref, n_gpu, next_gpu, st_ref=None, st_gpu=None,
            label=None):
    """Checks GPU outputs against the oracle's; returns the list of
    boundary-explained resample mismatches [(b, j_oracle, j_gpu)] and adds them
    to TALLY.  Raises AssertionError for any other difference."""
    n_ref, next_ref = np.asarray(n_ref), np.asarray(next_ref)
    n_gpu, next_gpu = np.asarray(n_gpu), np.asarray(next_gpu)
    bad_n = np.nonzero(n_ref != n_gpu)[0]
    assert bad_n.size == 0, (f"n_accepted differs at {bad_n[:10].tolist()}: oracle "
                             f"{n_ref[bad_n[:10]].tolist()} gpu {n_gpu[bad_n[:10]].tolist()}")
    if st_ref is not None and st_gpu is not None:
        assert st_ref == st_gpu, f"status oracle {st_ref} gpu {st_gpu}"
    c = classify(p, q, u_res, mode, K, n_ref, next_ref, n_gpu, next_gpu)
    if c["greedy"]:
        b = c["greedy"][0]
        raise AssertionError(f"greedy next_token differs at seq {b}: {next_ref[b]} vs {next_gpu[b]}")
    if c["unexplained"]:
        b, j0, j1, T, R = c["unexplained"][0]
        raise AssertionError(f"seq {b}: next_token oracle {j0} gpu {j1} is not a boundary case "
                             f"(T={T!r}, R={R!r})")
    count(mode, n_ref.shape[0], c["boundary"], label)
    return c["boundary"]


# Sampling from logits: the kernels warp with fp32 exp2.approx, the oracle with
# an fp64 softmax.  An accept test whose fp32 margin is inside the fast path's
# error bound is made again by the kernels in fp64 from the same formula, so
# an accept decision may differ from the oracle's only where the two fp64
# computations (summed in different orders) can round to different sides:
# |u*q - p| <= ACCEPT_BAND_LOGITS * p.  The masses of a draw are fp32 (~1e-6
# relative at most: exp2.approx ~2^-22, the fp32 argument (z - max)/T, the
# fp32 normaliser), so a drawn token may differ only where u*R lies within
# DRAW_TOL_LOGITS (normalised mass) of a boundary between the two answers.
ACCEPT_BAND_LOGITS = 1e-9
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
            assert margin <= ACCEPT_BAND_LOGITS * p, (
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
    TALLY["sequences"] += int(np.asarray(n_ref).shape[0])
    TALLY["draws"] += int(np.asarray(n_ref).shape[0])
    TALLY["logits_accept"] += sum(1 for _, k in explained if k == "accept")
    TALLY["logits_draw"] += sum(1 for _, k in explained if k == "draw")
    return explained
