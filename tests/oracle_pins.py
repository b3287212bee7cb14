"""Pins that tie the CPU oracle to facts fixed outside it.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError if
the oracle disagrees with something the pages or the mathematics fix:

* exact rational brute force of the speculative-sampling output law on tiny
  vocabularies (Leviathan et al. / Chen et al. theorem, cited by the
  "spec-verify" page, section "Method"), including distribution preservation
  of the first emitted token;
* plain greedy decoding of a deterministic toy target ("spec-verify",
  section "Method": the emitted stream is identical to plain greedy decoding;
  section "Correctness");
* the analytic accepted-length law E[n] = sum_m prod_{j<m} alpha_j with
  alpha_j = sum(min(p_j, q_j)) ("spec-verify", sections "Measured" and
  "Correctness");
* numpy's first-occurrence argmax and cumsum/searchsorted as independent
  library routines for the argmax and the inverse CDF;
* the exactly rounded sum (math.fsum) for the fp64 mass sums ("spec-verify",
  section "Correctness": masses summed exactly);
* closed-form special cases (q == p, one-hot targets, a single-token residual,
  power-of-two scaling, zero-mass fallback, invalid ids).

``tests/test_oracle_pins.py`` runs them on the real oracle and
``tests/test_oracle_mutants.py`` shows that planted mistakes fail them.
"""
from __future__ import annotations

import hashlib
import itertools
import math
from collections import defaultdict
from fractions import Fraction as Fr

import numpy as np

# ---------------------------------------------------------------------------
# helpers (input construction and closed forms only)


def _composition(rng, V, total):
    """V non-negative integers summing to ``total``."""
    cuts = np.sort(rng.integers(0, total + 1, size=V - 1))
    return np.diff(np.concatenate([[0], cuts, [total]])).astype(np.int64)


def _softmax(x):
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def _first_token_interval_us(r_int):
    """For integer masses r, the midpoint uniform of each token's inverse-CDF
    interval [C_{v-1}/R, C_v/R) and its exact probability r_v/R."""
    R = int(sum(int(x) for x in r_int))
    out = []
    c = 0
    for v, m in enumerate(r_int):
        m = int(m)
        if m > 0:
            out.append((v, float(Fr(2 * c + m, 2 * R)), Fr(m, R)))
        c += m
    return out


def _exact_law_from_oracle(orc, p_int, q_int, denom):
    """Output law of the oracle's sampling rule, integrating draft tokens
    t_i ~ q_i and the two uniforms exactly: returns {(n, next): Fraction}."""
    K, V = q_int.shape
    p = (p_int / denom).astype(np.float32)
    q = (q_int / denom).astype(np.float32)
    cases = []      # (t tuple, u_acc list, u_res, weight)
    for tup in itertools.product(range(V), repeat=K):
        w_t = Fr(1)
        for i, x in enumerate(tup):
            w_t *= Fr(int(q_int[i, x]), denom)
        if w_t == 0:
            continue
        # stop position m (first rejection, or K when all are accepted)
        prefix_w = Fr(1)
        u_acc_prefix = []
        for m in range(K + 1):
            if m < K:
                pm, qm = int(p_int[m, tup[m]]), int(q_int[m, tup[m]])
                a = Fr(min(pm, qm), qm)
                rej_w = 1 - a
                if rej_w > 0:
                    ratio = pm / qm
                    u_rej = (1.0 + ratio) / 2.0
                    r_int = np.maximum(p_int[m] - q_int[m], 0)
                    if r_int.sum() == 0:
                        r_int = p_int[m]
                    for v, u_res, pv in _first_token_interval_us(r_int):
                        u_acc = u_acc_prefix + [u_rej] + [0.5] * (K - m - 1)
                        cases.append((tup, u_acc, u_res, w_t * prefix_w * rej_w * pv))
                if a == 0:
                    break
                u_acc_prefix = u_acc_prefix + [(pm / qm) / 2.0 if a < 1 else 0.5]
                prefix_w *= a
            else:
                for v, u_res, pv in _first_token_interval_us(p_int[K]):
                    cases.append((tup, list(u_acc_prefix), u_res, w_t * prefix_w * pv))
    B = len(cases)
    P = np.broadcast_to(p, (B, K + 1, V)).copy()
    Q = np.broadcast_to(q, (B, K, V)).copy()
    T = np.array([c[0] for c in cases], dtype=np.int32).reshape(B, K)
    UA = np.array([c[1] for c in cases], dtype=np.float32).reshape(B, K)
    UR = np.array([c[2] for c in cases], dtype=np.float64)
    n, nxt, st = orc.verify_sample(P, Q, T, UA, UR)
    assert st == 0, f"unexpected status {st}"
    law = defaultdict(Fr)
    first = defaultdict(Fr)
    for c, ni, vi in zip(cases, n, nxt):
        law[(int(ni), int(vi))] += c[3]
        y0 = c[0][0] if ni >= 1 else int(vi)
        first[y0] += c[3]
    return law, first


def _closed_form_law(p_int, q_int, denom):
    """P(n=m, next=v) = prod_{j<m} alpha_j (1 - alpha_m) r_m(v)/R_m for m < K and
    prod_{j<K} alpha_j p_K(v) for m = K (rejection-sampling theorem)."""
    K, V = q_int.shape
    alpha = [Fr(int(np.minimum(p_int[j], q_int[j]).sum()), denom) for j in range(K)]
    law = {}
    pre = Fr(1)
    for m in range(K + 1):
        if m < K:
            r = np.maximum(p_int[m] - q_int[m], 0)
            R = int(r.sum())
            for v in range(V):
                if r[v] > 0:
                    law[(m, v)] = pre * (1 - alpha[m]) * Fr(int(r[v]), R)
            pre *= alpha[m]
        else:
            for v in range(V):
                if p_int[K, v] > 0:
                    law[(K, v)] = pre * Fr(int(p_int[K, v]), denom)
    return {k: v for k, v in law.items() if v != 0}


# ---------------------------------------------------------------------------
# pins


def pin_output_law_bruteforce(orc):
    """Exact output law on V in {3,4,5}, K in {1,2,3} (rational arithmetic)."""
    rng = np.random.default_rng(11)
    denom = 32
    for V, K in [(3, 1), (3, 2), (4, 2), (5, 1), (3, 3), (4, 3)]:
        for trial in range(3):
            p_int = np.stack([_composition(rng, V, denom) for _ in range(K + 1)])
            q_int = np.stack([_composition(rng, V, denom) for _ in range(K)])
            law, first = _exact_law_from_oracle(orc, p_int, q_int, denom)
            law = {k: v for k, v in law.items() if v != 0}
            expect = _closed_form_law(p_int, q_int, denom)
            assert law == expect, f"V={V} K={K} trial={trial}: law {law} != {expect}"
            # distribution preservation of the first emitted token
            for v in range(V):
                assert first.get(v, Fr(0)) == Fr(int(p_int[0, v]), denom), \
                    f"first emitted token not distributed as p_0 (V={V} K={K})"


def _toy_target(prefix, V):
    h = hashlib.blake2b(np.asarray(prefix, dtype=np.int64).tobytes(), digest_size=8)
    rng = np.random.default_rng(int.from_bytes(h.digest(), "little"))
    # coarse probabilities so that ties between maxima are common
    p = np.floor(_softmax(rng.normal(0.0, 1.5, V)) * 48.0) / 48.0
    return p.astype(np.float32)


def _toy_draft(prefix, V):
    h = hashlib.blake2b(b"draft" + np.asarray(prefix, dtype=np.int64).tobytes(),
                        digest_size=8)
    rng = np.random.default_rng(int.from_bytes(h.digest(), "little"))
    if rng.random() < 0.65:
        return int(np.argmax(_toy_target(prefix, V)))
    return int(rng.integers(0, V))


def pin_greedy_identity(orc):
    """Greedy speculative rounds reproduce plain greedy decoding of a toy target."""
    V, N = 50, 160
    for K in (1, 3, 4, 7):
        plain = [7, 3]
        while len(plain) < N:
            plain.append(int(np.argmax(_toy_target(plain, V))))
        spec = [7, 3]
        rounds = 0
        accepted_any = False
        while len(spec) < N:
            drafts = []
            for _ in range(K):
                drafts.append(_toy_draft(spec + drafts, V))
            P = np.stack([_toy_target(spec + drafts[:i], V) for i in range(K + 1)])
            n, nxt, st = orc.verify_greedy(P[None], np.array([drafts], dtype=np.int32))
            assert st == 0
            n, nxt = int(n[0]), int(nxt[0])
            accepted_any |= n > 0
            spec += drafts[:n] + [nxt]
            rounds += 1
        assert spec[:N] == plain, f"K={K}: speculative stream differs from greedy decoding"
        assert rounds < N - 2 and accepted_any


def pin_argmax_first_occurrence(orc):
    """The argmax is numpy's first-occurrence argmax, including planted ties and zeros."""
    rng = np.random.default_rng(5)
    for V in (1, 2, 3, 7, 64, 1000, 4099):
        for _ in range(20):
            row = rng.integers(0, 6, size=V).astype(np.float32) / 4
            if rng.random() < 0.3:
                row[:] = 0.0
                row[rng.integers(0, V, size=max(1, V // 3))] = -0.0
            assert orc.argmax_lowest(row) == int(np.argmax(row))


def pin_greedy_rule(orc):
    """Greedy decisions against numpy's argmax on random batches with ties."""
    rng = np.random.default_rng(6)
    for V, K in ((5, 1), (9, 4), (300, 6)):
        B = 64
        P = (rng.integers(0, 4, size=(B, K + 1, V)) / 8).astype(np.float32)
        A = P.argmax(axis=-1)
        T = np.where(rng.random((B, K)) < 0.8, A[:, :K],
                     rng.integers(0, V, size=(B, K))).astype(np.int32)
        n, nxt, st = orc.verify_greedy(P, T)
        assert st == 0
        for b in range(B):
            miss = [i for i in range(K) if T[b, i] != A[b, i]]
            m = miss[0] if miss else K
            assert (n[b], nxt[b]) == (m, A[b, m]), f"seq {b}: {(n[b], nxt[b])} vs {(m, A[b, m])}"


def pin_accept_threshold(orc):
    """Accept iff u < p(t)/q(t): exact threshold at u* = p/q, both sides."""
    V, K = 4, 1
    cases = [(0.25, 0.5), (0.375, 0.75), (3.0, 4.0), (1e-3, 0.75), (0.5, 0.5), (0.0, 0.5),
             (0.5, 0.0)]
    for pt, qt in cases:
        p = np.zeros((1, K + 1, V), np.float32)
        q = np.zeros((1, K, V), np.float32)
        p[0, 0, :] = [pt, 1.0, 0.0, 0.0]
        q[0, 0, :] = [qt, 0.0, 1.0, 0.0]
        p[0, 1, 3] = 1.0
        t = np.array([[0]], np.int32)
        for u in (0.0, 0.25, 0.5, 0.75, 0.9999999):
            u32 = np.float32(u)
            want_accept = float(u32) * float(np.float32(qt)) < float(np.float32(pt))
            n, nxt, st = orc.verify_sample(p, q, t, np.array([[u32]]), np.array([0.3]))
            assert n[0] == (1 if want_accept else 0), (pt, qt, u)
            assert nxt[0] == (3 if want_accept else 1), (pt, qt, u, nxt[0])
        if qt > 0 and pt < qt and pt > 0:
            ustar = np.float32(pt / qt)
            if float(ustar) * qt == pt:   # representable threshold: u* itself rejects
                n, _, _ = orc.verify_sample(p, q, t, np.array([[ustar]]), np.array([0.3]))
                assert n[0] == 0
                below = np.nextafter(ustar, np.float32(0))
                n, _, _ = orc.verify_sample(p, q, t, np.array([[below]]), np.array([0.3]))
                assert n[0] == 1
    # p(t) = the fp32-rounded product u*q: the exact product decides (rationals)
    rng = np.random.default_rng(13)
    B = 400
    u = rng.random(B).astype(np.float32)
    qt = (rng.random(B) * 0.9 + 0.05).astype(np.float32)
    pt = (u * qt).astype(np.float32)                      # rounded to nearest in fp32
    P = np.zeros((B, 2, V), np.float32)
    Q = np.zeros((B, 1, V), np.float32)
    P[:, 0, 0], P[:, 0, 1], P[:, 1, 3] = pt, 1.0, 1.0
    Q[:, 0, 0], Q[:, 0, 2] = qt, 1.0
    n, nxt, st = orc.verify_sample(P, Q, np.zeros((B, 1), np.int32), u[:, None],
                                   np.full(B, 0.3))
    want = np.array([Fr(float(a)) * Fr(float(b)) < Fr(float(c)) for a, b, c in zip(u, qt, pt)])
    assert want.any() and not want.all()
    assert np.array_equal(n == 1, want)


def pin_icdf_library(orc):
    """Inverse CDF equals numpy cumsum + searchsorted(side='right'); step law on a grid."""
    rng = np.random.default_rng(7)
    for V in (1, 2, 5, 33, 1000):
        for _ in range(10):
            r = rng.random(V) * (rng.random(V) < 0.6)
            if r.sum() == 0:
                r[rng.integers(0, V)] = 0.5
            C = np.cumsum(r)
            for u in rng.random(25):
                j = int(np.searchsorted(C, u * C[-1], side="right"))
                if j == V:
                    j = int(np.nonzero(r)[0][-1])
                assert orc.icdf(r, u) == j
    # step-function law: frequencies on a uniform grid equal r_v / R
    r = np.array([0.0, 3.0, 0.0, 1.0, 0.5, 0.0, 2.5, 1.0])
    N = 20000
    counts = np.zeros(r.size)
    for k in range(N):
        counts[orc.icdf(r, (k + 0.5) / N)] += 1
    assert np.all(counts[r == 0] == 0)
    assert np.max(np.abs(counts / N - r / r.sum())) <= 1.0 / N + 1e-12
    assert orc.icdf(np.zeros(6), 0.3) == -1


def pin_fp64_mass_sum(orc):
    """Mass sums are fp64: matches math.fsum within V * 2^-53, and a mass lost in
    fp32 accumulation still moves the draw."""
    rng = np.random.default_rng(8)
    for V in (10, 1000, 100000):
        p = rng.random(V).astype(np.float32)
        q = (rng.random(V) * 0.9).astype(np.float32)
        C, R = orc.residual_cumsum(p, q)
        terms = np.maximum(p.astype(np.float64) - q.astype(np.float64), 0.0)
        exact = math.fsum(terms.tolist())
        assert abs(R - exact) <= V * 2.0 ** -53 * exact
        assert C[-1] == R and np.all(np.diff(C) >= 0)
    # one large mass followed by 2^20 masses each below half an fp32 ulp of it
    r = np.full(1 + (1 << 20), 1e-9)
    r[0] = 1.0
    j = orc.icdf(r, 0.9995)
    assert j > 400000, j
    # the same through the full sampling path (bonus row, unnormalised)
    V = r.size
    p = np.zeros((1, 2, V), np.float32)
    p[0, 1] = r.astype(np.float32)
    p[0, 0, 0] = 1.0
    q = np.zeros((1, 1, V), np.float32)
    q[0, 0, 0] = 1.0
    n, nxt, st = orc.verify_sample(p, q, np.array([[0]], np.int32),
                                   np.array([[0.5]], np.float32), np.array([0.9995]))
    assert n[0] == 1 and nxt[0] > 400000


def pin_analytic_length_law(orc, rounds=1200, V=2048):
    """Mean and histogram of n over many rounds match the exact per-round law."""
    from speculative_decoding_verification_08_gb300.inputs import make_inputs
    from scipy import stats

    K = 4
    bt = make_inputs(1, "cpu", seed=424242, B=rounds, V=V, K=K)
    p, q, t, ua, ur, _ = bt.numpy()
    n, nxt, st = orc.verify_sample(p, q, t, ua, ur, nthreads=4)
    assert st == 0
    alpha = np.empty((rounds, K))                         # sum(min(p_hat, q_hat))
    for r0 in range(0, rounds, 64):
        ph = p[r0:r0 + 64, :K].astype(np.float64)
        qh = q[r0:r0 + 64].astype(np.float64)
        ph /= ph.sum(-1, keepdims=True)
        qh /= qh.sum(-1, keepdims=True)
        alpha[r0:r0 + 64] = np.minimum(ph, qh).sum(-1)
    probs = np.zeros((rounds, K + 1))
    pre = np.ones(rounds)
    for m in range(K):
        probs[:, m] = pre * (1 - alpha[:, m])
        pre = pre * alpha[:, m]
    probs[:, K] = pre
    mean = (probs * np.arange(K + 1)).sum(1)
    var = (probs * np.arange(K + 1) ** 2).sum(1) - mean ** 2
    z = (n.mean() - mean.mean()) / math.sqrt(var.sum() / rounds ** 2)
    assert abs(z) < 4.0, f"mean n {n.mean():.4f} vs law {mean.mean():.4f} (z={z:.2f})"
    obs = np.bincount(n, minlength=K + 1)
    exp = probs.sum(0)
    keep = exp >= 5
    chi = ((obs[keep] - exp[keep]) ** 2 / exp[keep]).sum()
    assert stats.chi2.sf(chi, keep.sum() - 1) > 1e-3, f"histogram {obs} vs {exp}"
    return float(n.mean()), float(mean.mean()), float(alpha.mean())


def pin_alpha(orc):
    """Per-position acceptance rate alpha = sum min(p_hat, q_hat) and the
    expected accepted length sum_m prod_{j<m} alpha_j, pinned to:
    the identity alpha = 1 - TV(p_hat, q_hat) (a different formula, with
    |.| instead of min); exact rationals on small integer rows; closed forms
    (identical rows, disjoint supports, one-hot p, zero rows, power-of-two
    scaling); and the mean accepted length of the oracle's own sampler over
    many rounds (the law, not the formula)."""
    rng = np.random.default_rng(8080)
    # identity with total variation, unnormalised rows of assorted scales
    B, K, V = 6, 3, 700
    p = (rng.random((B, K + 1, V)) ** 3 * rng.uniform(0.2, 5, (B, K + 1, 1))).astype(np.float32)
    q = (rng.random((B, K, V)) ** 3 * rng.uniform(0.2, 5, (B, K, 1))).astype(np.float32)
    a, e = orc.alpha(p, q)
    ph = p[:, :K].astype(np.float64) / p[:, :K].astype(np.float64).sum(-1, keepdims=True)
    qh = q.astype(np.float64) / q.astype(np.float64).sum(-1, keepdims=True)
    tv = 0.5 * np.abs(ph - qh).sum(-1)
    assert np.allclose(a, 1.0 - tv, atol=1e-12, rtol=0), (a, 1 - tv)
    assert ((0 <= a) & (a <= 1 + 1e-12)).all()
    # exact rationals
    pi = rng.integers(0, 9, (2, 3, 5))
    qi = rng.integers(0, 9, (2, 2, 5))
    pi[:, :, 0] += 1
    qi[:, :, 0] += 1
    a, e = orc.alpha(pi.astype(np.float32), qi.astype(np.float32))
    for b in range(2):
        exp_len, reach = Fr(0), Fr(1)
        for i in range(2):
            P, Q = int(pi[b, i].sum()), int(qi[b, i].sum())
            ex = sum(min(Fr(int(x), P), Fr(int(y), Q)) for x, y in zip(pi[b, i], qi[b, i]))
            assert abs(a[b, i] - float(ex)) < 1e-15, (a[b, i], ex)
            reach *= ex
            exp_len += reach
        assert abs(e[b] - float(exp_len)) < 1e-14, (e[b], exp_len)
    # closed forms: position 0 identical after scaling, 1 disjoint supports,
    # 2 one-hot p, 3 an all-zero p row; row 4 is the (unused) bonus row
    V = 64
    base = rng.random(V).astype(np.float32) + 0.01
    low = (np.arange(V) < 32).astype(np.float32)
    p = np.stack([base * 4, base * (1 - low), np.eye(V, dtype=np.float32)[7] * 3,
                  np.zeros(V, np.float32), base])
    q = np.stack([base * 0.25, base * low, base, base])
    a, e = orc.alpha(p[None], q[None])
    assert abs(a[0, 0] - 1.0) < V * 2.0 ** -52, a
    assert a[0, 1] == 0.0 and a[0, 3] == 0.0, a
    assert abs(a[0, 2] - float(base[7]) / float(base.astype(np.float64).sum())) < 1e-15, a
    assert e[0] == a[0, 0], e                                    # 1 + 0 + 0 + 0 terms after a_0
    s1, e1 = orc.alpha(p[None] * np.float32(2.0 ** 5), q[None] * np.float32(2.0 ** -7))
    assert np.array_equal(s1, a) and np.array_equal(e1, e)       # scaling invariance, exact
    # the law, through the sampler: rows fixed, drafts and uniforms fresh each round
    R, K, V = 4000, 3, 40
    prow = _softmax(rng.normal(0, 1.5, (K + 1, V))).astype(np.float32)
    qrow = _softmax(rng.normal(0, 1.5, (K, V)) + 0.4 * rng.normal(0, 1, (K, V))).astype(np.float32)
    a, e = orc.alpha(prow[None], qrow[None])
    pp = np.broadcast_to(prow, (R, K + 1, V)).copy()
    qq = np.broadcast_to(qrow, (R, K, V)).copy()
    qn = qrow.astype(np.float64) / qrow.astype(np.float64).sum(-1, keepdims=True)
    t = np.stack([rng.choice(V, size=R, p=qn[i]) for i in range(K)], 1).astype(np.int32)
    ua = rng.random((R, K)).astype(np.float32)
    ur = rng.random(R)
    n, _, st = orc.verify_sample(pp, qq, t, ua, ur, nthreads=4)
    assert st == 0
    probs, pre = [], 1.0
    for m in range(K):
        probs.append(pre * (1 - a[0, m]))
        pre *= a[0, m]
    probs.append(pre)
    probs = np.array(probs)
    var = (probs * np.arange(K + 1) ** 2).sum() - e[0] ** 2
    z = (n.mean() - e[0]) / math.sqrt(var / R)
    assert abs(z) < 4.0, f"sampler mean {n.mean():.4f} vs expected length {e[0]:.4f} (z={z:.2f})"


def pin_logits(orc):
    """Sampling from logits (temperature softmax in fp64, then the rule),
    pinned to: scipy's softmax (a library routine); exact shift and
    temperature identities; huge logits (no overflow: the max is
    subtracted); agreement with the probability oracle on the same
    distributions, away from its decision boundaries; and distribution
    preservation of the first emitted token (the rejection-sampling theorem),
    by a chi-square test over many rounds."""
    from scipy import special, stats

    rng = np.random.default_rng(9191)
    z = (rng.normal(0, 3, 1000)).astype(np.float32)
    for tau in (0.5, 1.0, 1.7):
        ref = special.softmax(z.astype(np.float64) / tau)
        got = orc.softmax(z, tau)
        assert np.allclose(got, ref, rtol=1e-13, atol=0), tau
        assert abs(got.sum() - 1.0) < 1e-13
    # exact identities: a shift by a representable constant, and tau = 2 on z
    # equals tau = 1 on z / 2 (both exact in fp32 here)
    zq16 = (np.round(z * 1024) / 1024).astype(np.float32)
    assert np.array_equal(orc.softmax(zq16, 1.3), orc.softmax(zq16 + np.float32(8.0), 1.3))
    assert np.array_equal(orc.softmax(zq16, 2.0), orc.softmax(zq16 / np.float32(2.0), 1.0))
    big = np.array([3.0e38, 2.9e38, -3.0e38, 3.0e38], dtype=np.float32)
    sb = orc.softmax(big, 1e36)
    assert np.isfinite(sb).all() and abs(sb.sum() - 1) < 1e-12 and sb[0] == sb[3] > sb[1]
    # the same draws as the probability oracle, except near its boundaries
    B, K, V = 300, 3, 200
    zp = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    zqq = (zp[:, :K] + rng.normal(0, 0.8, (B, K, V))).astype(np.float32)
    tau = 0.9
    P = np.stack([[orc.softmax(zp[b, i], tau) for i in range(K + 1)] for b in range(B)])
    Q = np.stack([[orc.softmax(zqq[b, i], tau) for i in range(K)] for b in range(B)])
    t = np.stack([[rng.choice(V, p=Q[b, i] / Q[b, i].sum()) for i in range(K)] for b in range(B)])
    t = t.astype(np.int32)
    ua = rng.random((B, K)).astype(np.float32)
    ur = rng.random(B)
    n1, x1, s1 = orc.verify_sample_logits(zp, zqq, t, ua, ur, tau)
    n0, x0, s0 = orc.verify_sample(P.astype(np.float32), Q.astype(np.float32), t, ua, ur)
    assert s1 == 0 and s0 == 0
    agree = (n1 == n0) & (x1 == x0)
    assert agree.mean() > 0.97, agree.mean()
    for b in np.nonzero(~agree)[0]:   # a disagreement needs a near-tie somewhere
        i = min(int(n0[b]), int(n1[b]))
        if n0[b] != n1[b]:
            pt, qt = P[b, i, t[b, i]], Q[b, i, t[b, i]]
            assert abs(ua[b, i] * qt - pt) <= 1e-6 * max(pt, 1e-30), (b, i, ua[b, i] * qt, pt)
        else:
            r = np.maximum(P[b, i] - Q[b, i], 0) if i < K else P[b, K]
            C = np.cumsum(r)
            T = ur[b] * C[-1]
            lo, hi = sorted((int(x0[b]), int(x1[b])))
            assert np.abs(C[lo:hi + 1] - T).min() <= 1e-6 * C[-1], (b, lo, hi)
    # distribution preservation: the first emitted token ~ p_0
    R, K, V = 20000, 2, 12
    zp1 = rng.normal(0, 1.2, (K + 1, V)).astype(np.float32)
    zq1 = (zp1[:K] + rng.normal(0, 0.7, (K, V))).astype(np.float32)
    tau = 1.3
    q0 = np.stack([orc.softmax(zq1[i], tau) for i in range(K)])
    zpb = np.broadcast_to(zp1, (R, K + 1, V)).copy()
    zqb = np.broadcast_to(zq1, (R, K, V)).copy()
    t = np.stack([rng.choice(V, size=R, p=q0[i] / q0[i].sum()) for i in range(K)], 1).astype(np.int32)
    n, x, st = orc.verify_sample_logits(zpb, zqb, t, rng.random((R, K)).astype(np.float32),
                                        rng.random(R), tau)
    first = np.where(n > 0, t[:, 0], x)
    p0 = orc.softmax(zp1[0], tau)
    obs = np.bincount(first, minlength=V)
    chi = ((obs - R * p0) ** 2 / (R * p0)).sum()
    assert stats.chi2.sf(chi, V - 1) > 1e-3, (obs, R * p0)


def pin_special_cases(orc):
    """q == p accepts everything; one-hot targets and single-token residuals are
    deterministic; power-of-two scaling changes nothing."""
    rng = np.random.default_rng(9)
    V, K, B = 257, 5, 16
    p = rng.random((B, K + 1, V)).astype(np.float32)
    q = rng.random((B, K, V)).astype(np.float32)
    t = rng.integers(0, V, size=(B, K)).astype(np.int32)
    ua = rng.random((B, K)).astype(np.float32)
    ur = rng.random(B)
    # q == p: every position accepted, bonus drawn from p_K
    n, nxt, st = orc.verify_sample(p, p[:, :K].copy(), t, ua, ur)
    assert st == 0 and np.all(n == K)
    for b in range(B):
        C = np.cumsum(p[b, K].astype(np.float64))
        assert nxt[b] == int(np.searchsorted(C, ur[b] * C[-1], side="right"))
    # one-hot targets: a draft off the hot token is always rejected in favour of it
    ph = np.zeros_like(p)
    hot = rng.integers(0, V, size=(B, K + 1))
    for b in range(B):
        ph[b, np.arange(K + 1), hot[b]] = 1.5
    td = np.where(t == hot[:, :K], (t + 1) % V, t).astype(np.int32)
    n, nxt, st = orc.verify_sample(ph, q, td, ua, ur)
    assert st == 0 and np.all(n == 0) and np.all(nxt == hot[:, 0])
    # greedy on one-hot targets with drafts on the hot tokens: bonus is the hot token
    n, nxt, st = orc.verify_greedy(ph, hot[:, :K].astype(np.int32))
    assert np.all(n == K) and np.all(nxt == hot[:, K])
    # single-token residual: the resample is that token for every uniform
    x = rng.integers(0, V, size=B)
    qs = np.repeat(p[:, :1], K, axis=1).copy()
    for b in range(B):
        qs[b, 0, x[b]] = p[b, 0, x[b]] * 0.25
        y = (x[b] + 1) % V
        qs[b, 0, y] = p[b, 0, y] + 2.0
    ts = np.tile(((x + 1) % V)[:, None], (1, K)).astype(np.int32)
    for u in (0.0, 0.37, 0.999999):
        n, nxt, st = orc.verify_sample(p, qs, ts, np.full((B, K), 0.9999, np.float32),
                                       np.full(B, u))
        assert np.all(n == 0) and np.all(nxt == x), (n, nxt, x)
    # scaling every row of a sequence by 2^k leaves (n, next) bit-identical
    base = orc.verify_sample(p, q, t, ua, ur)
    for k in (-3, -1, 2, 5):
        s = np.float32(2.0 ** k)
        got = orc.verify_sample(p * s, q * s, t, ua, ur)
        assert np.array_equal(got[0], base[0]) and np.array_equal(got[1], base[1])
    g0 = orc.verify_greedy(p, t)
    g1 = orc.verify_greedy(p * np.float32(8.0), t)
    assert np.array_equal(g0[0], g1[0]) and np.array_equal(g0[1], g1[1])


def pin_zero_mass_and_invalid(orc):
    """Zero-residual fallback to p_i, zero total mass, out-of-range ids, bad modes."""
    V, K = 3, 1
    # unnormalised rows with p <= q everywhere: a rejection draws from p_0
    p = np.array([[[1.0, 0.5, 0.5], [0.0, 0.0, 1.0]]], np.float32)
    q = np.array([[[1.0, 2.0, 1.0]]], np.float32)
    t = np.array([[1]], np.int32)
    n, nxt, st = orc.verify_sample(p, q, t, np.array([[0.3]], np.float32), np.array([0.6]))
    assert (n[0], nxt[0], st) == (0, 1, 0)        # T = 1.2 falls in (1.0, 1.5]
    n, nxt, st = orc.verify_sample(p, q, t, np.array([[0.2]], np.float32), np.array([0.6]))
    assert (n[0], nxt[0], st) == (1, 2, 0)        # 0.2*2 < 0.5: accepted, bonus token 2
    # zero mass everywhere: next = -1 and the ZERO_MASS bit
    pz = np.zeros((1, 2, V), np.float32)
    qz = np.array([[[1.0, 0.0, 0.0]]], np.float32)
    n, nxt, st = orc.verify_sample(pz, qz, np.array([[0]], np.int32),
                                   np.array([[0.5]], np.float32), np.array([0.5]))
    assert (n[0], nxt[0], st) == (0, -1, 2)
    # bonus row with zero mass
    pb = np.array([[[1.0, 0.0, 0.0], [0.0, 0.0, 0.0]]], np.float32)
    n, nxt, st = orc.verify_sample(pb, qz, np.array([[0]], np.int32),
                                   np.array([[0.5]], np.float32), np.array([0.5]))
    assert (n[0], nxt[0], st) == (1, -1, 2)
    # draft ids outside [0, V): the sequence is invalid, others unaffected
    P = np.tile(p, (3, 1, 1))
    Q = np.tile(q, (3, 1, 1))
    T = np.array([[1], [V], [-1]], np.int32)
    n, nxt, st = orc.verify_sample(P, Q, T, np.full((3, 1), 0.2, np.float32), np.full(3, 0.6))
    assert list(n) == [1, 0, 0] and list(nxt) == [2, -1, -1] and st == 1
    n, nxt, st = orc.verify_greedy(P, T)
    assert list(nxt[1:]) == [-1, -1] and list(n[1:]) == [0, 0] and st == 1
    # mode values other than 0 and 1
    n, nxt, st = orc.verify_round(np.array([0, 1, 7], np.uint8), P, Q,
                                  np.array([[1], [1], [1]], np.int32),
                                  np.full((3, 1), 0.2, np.float32), np.full(3, 0.6))
    assert list(n) == [0, 1, 0] and list(nxt) == [0, 2, -1] and st == 8


def pin_round_and_commit(orc):
    """Mixed rounds apply each sequence's rule; commit appends t[:n] + next."""
    rng = np.random.default_rng(10)
    V, K, B = 97, 6, 40
    p = rng.random((B, K + 1, V)).astype(np.float32)
    q = rng.random((B, K, V)).astype(np.float32)
    A = p.argmax(-1)
    t = np.where(rng.random((B, K)) < 0.7, A[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    ua = rng.random((B, K)).astype(np.float32)
    ur = rng.random(B)
    mode = (np.arange(B) % 2).astype(np.uint8)
    n, nxt, st = orc.verify_round(mode, p, q, t, ua, ur)
    g = orc.verify_greedy(p, t)
    s = orc.verify_sample(p, q, t, ua, ur)
    for b in range(B):
        ref = g if mode[b] == 0 else s
        assert (n[b], nxt[b]) == (ref[0][b], ref[1][b])
    max_len = 12
    tokens = np.full((B, max_len), -7, np.int32)
    lengths = rng.integers(0, 6, size=B).astype(np.int32)
    before = lengths.copy()
    stc = orc.commit(t, n, nxt, tokens, lengths)
    for b in range(B):
        if before[b] + n[b] + 1 > max_len:
            assert lengths[b] == before[b]
            assert stc & 4
            continue
        L = before[b]
        assert lengths[b] == L + n[b] + 1
        assert list(tokens[b, L:L + n[b]]) == list(t[b, :n[b]])
        assert tokens[b, L + n[b]] == nxt[b]
        assert np.all(tokens[b, :L] == -7) and np.all(tokens[b, L + n[b] + 1:] == -7)


def pin_threads_agree(orc):
    """The multi-threaded oracle returns exactly the single-threaded results."""
    rng = np.random.default_rng(12)
    V, K, B = 500, 3, 37
    p = rng.random((B, K + 1, V)).astype(np.float32)
    q = rng.random((B, K, V)).astype(np.float32)
    t = rng.integers(0, V, (B, K)).astype(np.int32)
    ua = rng.random((B, K)).astype(np.float32)
    ur = rng.random(B)
    a = orc.verify_sample(p, q, t, ua, ur, nthreads=1)
    b = orc.verify_sample(p, q, t, ua, ur, nthreads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2]


PINS = [
    pin_output_law_bruteforce,
    pin_greedy_identity,
    pin_argmax_first_occurrence,
    pin_greedy_rule,
    pin_accept_threshold,
    pin_icdf_library,
    pin_fp64_mass_sum,
    pin_special_cases,
    pin_zero_mass_and_invalid,
    pin_round_and_commit,
    pin_threads_agree,
    pin_analytic_length_law,
    pin_alpha,
    pin_logits,
]
