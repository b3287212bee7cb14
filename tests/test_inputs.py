"""The seeded input generator (inputs.py) produces the workloads it documents,
at reduced sizes on the CPU: normalised rows where they should be, planted
exact ties and higher-duplicate drafts, alternating modes, identical draft and
target rows, one-hot targets, single-token residuals, unnormalised scales,
uniforms in [0, 1), and the same tensors for the same seed."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_08_gb300.inputs import make_inputs


def _np(bt):
    return bt.numpy()


def test_same_seed_same_inputs_other_seed_other_inputs():
    a = make_inputs(3, "cpu", seed=11, B=6, V=700, K=3)
    b = make_inputs(3, "cpu", seed=11, B=6, V=700, K=3)
    c = make_inputs(3, "cpu", seed=12, B=6, V=700, K=3)
    for x, y in zip(_np(a), _np(b)):
        assert np.array_equal(x, y)
    assert not np.array_equal(a.p.numpy(), c.p.numpy())


@pytest.mark.parametrize("cfg", [1, 3])
def test_sampling_workloads_are_normalised_with_valid_drafts_and_uniforms(cfg):
    bt = make_inputs(cfg, "cpu", seed=5, B=16, V=1500, K=4)
    p, q, t, ua, ur, md = _np(bt)
    assert p.shape == (16, 5, 1500) and q.shape == (16, 4, 1500) and t.shape == (16, 4)
    assert np.all(np.isfinite(p)) and np.all(p >= 0) and np.all(q >= 0)
    assert np.allclose(p.sum(-1), 1.0, atol=1e-5) and np.allclose(q.sum(-1), 1.0, atol=1e-5)
    assert t.dtype == np.int32 and np.all((t >= 0) & (t < 1500))
    assert ua.dtype == np.float32 and np.all((ua >= 0) & (ua < 1))
    assert ur.dtype == np.float64 and np.all((ur >= 0) & (ur < 1))
    assert np.all(md == 1)
    # drafts are drawn from q: a drafted token has draft mass
    assert np.all(np.take_along_axis(q, t[..., None].astype(np.int64), 2) > 0)


def test_greedy_workload_plants_exact_ties_and_higher_duplicate_drafts():
    B, V, K = 400, 2000, 4
    bt = make_inputs(2, "cpu", seed=9, B=B, V=V, K=K)
    p, _, t, _, _, md = _np(bt)
    assert np.all(md == 0)
    top = p.max(-1, keepdims=True)
    ties = (p == top).sum(-1)                       # [B][K+1]
    planted = int((ties >= 2).sum())
    assert planted == bt.meta["planted_rows"]
    rows = B * (K + 1)
    assert 0.03 * rows < planted < 0.07 * rows     # about 5% of rows
    first = p.argmax(-1)[:, :K]
    last = (V - 1 - p[..., ::-1].argmax(-1))[:, :K]
    tie_rows = ties[:, :K] >= 2
    # drafts on the higher of two equal maxima: the ones the recipe flips there,
    # plus plain hits on rows whose original maximum is the higher duplicate
    higher = tie_rows & (t == last) & (last != first)
    assert higher.sum() >= bt.meta["higher_dup_drafts"] > 0
    hit = (t == first)[~tie_rows].mean()
    assert 0.6 < hit < 0.8                          # the draft is the argmax w.p. 0.7


def test_mixed_workload_alternates_modes_and_greedy_sequences_draft_the_argmax():
    bt = make_inputs(4, "cpu", seed=3, B=64, V=1000, K=8)
    p, q, t, ua, ur, md = _np(bt)
    assert np.array_equal(md, np.arange(64) % 2)
    assert 0.3 <= bt.meta["sig_d_min"] <= bt.meta["sig_d_max"] <= 2.5
    greedy = md == 0
    assert np.array_equal(t[greedy], q[greedy].argmax(-1))


def test_edge_workload_special_sequences():
    B, V, K = 200, 3000, 6
    bt = make_inputs(5, "cpu", seed=7, B=B, V=V, K=K)
    p, q, t, _, _, _ = _np(bt)
    same, onehot, single = bt.meta["same"], bt.meta["onehot"], bt.meta["single"]
    assert len(same) == len(onehot) == B // 10 and len(single) == B // 20
    assert not (set(same) & set(onehot)) and not (set(single) & (set(same) | set(onehot)))
    assert np.all(np.isfinite(p)) and np.all(p >= 0) and np.all(q >= 0)
    for b in same:
        assert np.array_equal(q[b], p[b, :K])       # identical rows, scale included
    for b in onehot:
        assert np.all((p[b] > 0).sum(-1) == 1)
    for b in single:
        residual = np.maximum(p[b, :K].astype(np.float64) - q[b], 0.0)
        assert np.all((residual > 0).sum(-1) == 1)
    plain = [b for b in range(B) if b not in set(same) | set(onehot) | set(single)]
    sums = p[plain].sum(-1)
    assert sums.min() >= 0.5 - 1e-4 and sums.max() <= 2.0 + 1e-4   # rows left unnormalised
    assert sums.std() > 0.1
    assert np.all(np.take_along_axis(q, t[..., None].astype(np.int64), 2) > 0)
