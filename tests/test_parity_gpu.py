"""CUDA path against the CPU oracle, element by element, on the same seeded
inputs: greedy outputs and accept decisions bit-exact, drawn tokens exact up
to counted boundary cases (oracle/compare.py).  Needs a GPU (-m gpu)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_08_gb300 as sv
from speculative_decoding_verification_08_gb300.inputs import make_inputs
from oracle.compare import compare

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.build()
    sv.load()
    yield


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def gpu_greedy(bt):
    n, nx = sv.verify_greedy(bt.p, bt.t)
    ws = sv._workspace(None, bt.B, bt.K, bt.V, bt.p.device)
    st = ws.status()
    return n.cpu().numpy(), nx.cpu().numpy(), st


def gpu_sample(bt):
    n, nx = sv.verify_sample(bt.p, bt.q, bt.t, bt.u_acc, bt.u_res)
    ws = sv._workspace(None, bt.B, bt.K, bt.V, bt.p.device)
    st = ws.status()
    return n.cpu().numpy(), nx.cpu().numpy(), st


def gpu_round(bt, mode=None, tokens=None, lengths=None):
    mode = bt.mode if mode is None else mode
    n, nx = sv.verify_round(mode, bt.p, bt.q, bt.t, bt.u_acc, bt.u_res, tokens=tokens,
                            lengths=lengths)
    ws = sv._workspace(None, bt.B, bt.K, bt.V, bt.p.device)
    st = ws.status()
    return n.cpu().numpy(), nx.cpu().numpy(), st


def check_greedy(bt, host=None):
    p, q, t, ua, ur, md = host if host is not None else bt.numpy()
    n0, x0, s0 = oracle.verify_greedy(p, t, nthreads=8)
    n1, x1, s1 = gpu_greedy(bt)
    compare(p, q, ur, 0, bt.K, n0, x0, n1, x1, s0, s1)
    return n0


def check_sample(bt, host=None, label=""):
    p, q, t, ua, ur, md = host if host is not None else bt.numpy()
    n0, x0, s0 = oracle.verify_sample(p, q, t, ua, ur, nthreads=8)
    n1, x1, s1 = gpu_sample(bt)
    compare(p, q, ur, 1, bt.K, n0, x0, n1, x1, s0, s1,
            label=label or bt.meta.get("name"))
    return n0


# ---------------------------------------------------------------------------
# scaled-down workloads: several segments and CTAs, ragged tails

@pytest.mark.parametrize("V", [1, 3, 31, 1000, 1024, 1025, 4099, 20000 + 37])
def test_greedy_scaled_ragged(V):
    bt = make_inputs(2, "cuda", seed=100 + V, B=24, V=V, K=4)
    check_greedy(bt)


@pytest.mark.parametrize("V", [1, 2, 5, 1023, 1024, 1025, 3 * 1024 + 7, 50000 + 3])
def test_sample_scaled_ragged(V):
    bt = make_inputs(3, "cuda", seed=200 + V, B=33, V=V, K=5)
    check_sample(bt, label=f"scaled V={V}")


@pytest.mark.parametrize("K", [0, 1, 2, 7, 16, 33, 64])
def test_draft_lengths(K):
    bt = make_inputs(4, "cuda", seed=300 + K, B=20, V=2500, K=K)
    check_greedy(bt)
    check_sample(bt, label=f"K={K}")
    p, q, t, ua, ur, md = bt.numpy()
    n0, x0, s0 = oracle.verify_round(md, p, q, t, ua, ur)
    n1, x1, s1 = gpu_round(bt)
    compare(p, q, ur, md, K, n0, x0, n1, x1, s0, s1)


def test_edge_distributions_scaled():
    """Unnormalised rows, q == p, one-hot targets, single-token residuals."""
    bt = make_inputs(5, "cuda", seed=5000, B=60, V=9000, K=16)
    n = check_sample(bt, label="edge scaled")
    check_greedy(bt)
    same = bt.meta["same"]
    assert np.all(n[same] == 16)


@pytest.mark.parametrize("ctas", [1, 2, 3, 5, 0])
def test_launch_shapes_agree(ctas):
    """Grids from one CTA per SM (many items per warp) to full residency."""
    bt = make_inputs(3, "cuda", seed=777, B=40, V=40000, K=5)
    host = bt.numpy()
    try:
        sv.set_ctas_per_sm(ctas)
        check_sample(bt, host, label=f"ctas={ctas}")
        check_greedy(bt, host)
        p, q, t, ua, ur, md = host
        n0, x0, s0 = oracle.verify_round(md, p, q, t, ua, ur)
        n1, x1, s1 = gpu_round(bt)
        compare(p, q, ur, md, bt.K, n0, x0, n1, x1, s0, s1)
    finally:
        sv.set_ctas_per_sm(0)


def test_unaligned_rows_and_strides():
    """Rows that do not start on 16 bytes take the scalar path; results agree."""
    B, K, V = 9, 3, 5003
    bt = make_inputs(3, "cuda", seed=31, B=B, V=V, K=K)
    p, q, t, ua, ur, md = bt.numpy()
    n0, x0, s0 = oracle.verify_sample(p, q, t, ua, ur)
    g0 = oracle.verify_greedy(p, t)
    for pad in (1, 2, 3, 4):
        Pbig = torch.zeros(B, K + 1, V + pad, device="cuda")
        Qbig = torch.zeros(B, K, V + pad, device="cuda")
        Pbig[:, :, :V] = bt.p
        Qbig[:, :, :V] = bt.q
        pv, qv = Pbig[:, :, :V], Qbig[:, :, :V]
        n1, x1 = sv.verify_sample(pv, qv, bt.t, bt.u_acc, bt.u_res)
        compare(p, q, ur, 1, K, n0, x0, n1.cpu().numpy(), x1.cpu().numpy())
        n2, x2 = sv.verify_greedy(pv, bt.t)
        compare(p, q, ur, 0, K, g0[0], g0[1], n2.cpu().numpy(), x2.cpu().numpy())
    # base pointer offset by one element
    flat = torch.zeros(B * (K + 1) * V + 1, device="cuda")
    flat[1:] = bt.p.reshape(-1)
    pv = flat[1:].view(B, K + 1, V)
    n3, x3 = sv.verify_greedy(pv, bt.t)
    compare(p, q, ur, 0, K, g0[0], g0[1], n3.cpu().numpy(), x3.cpu().numpy())


def test_repeated_calls_are_identical_and_clean():
    bt = make_inputs(3, "cuda", seed=41, B=50, V=30000, K=5)
    a = gpu_sample(bt)
    for _ in range(3):
        b = gpu_sample(bt)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and b[2] == 0
    g = gpu_greedy(bt)
    for _ in range(3):
        h = gpu_greedy(bt)
        assert np.array_equal(g[0], h[0]) and np.array_equal(g[1], h[1]) and h[2] == 0


def test_error_statuses():
    B, K, V = 6, 3, 700
    bt = make_inputs(3, "cuda", seed=51, B=B, V=V, K=K)
    t = bt.t.clone()
    t[1, 2] = V
    t[3, 0] = -5
    bt.t = t
    p, q, tt, ua, ur, md = bt.numpy()
    n0, x0, s0 = oracle.verify_sample(p, q, tt, ua, ur)
    n1, x1, s1 = gpu_sample(bt)
    assert s0 == s1 == sv.STATUS_BAD_TOKEN
    compare(p, q, ur, 1, K, n0, x0, n1, x1)
    g0 = oracle.verify_greedy(p, tt)
    n2, x2, s2 = gpu_greedy(bt)
    assert s2 == sv.STATUS_BAD_TOKEN
    compare(p, q, ur, 0, K, g0[0], g0[1], n2, x2)
    # invalid modes
    mode = torch.tensor([0, 1, 2, 255, 1, 0], dtype=torch.uint8, device="cuda")
    bt.t = bt.t.clamp(0, V - 1)
    p, q, tt, ua, ur, md = bt.numpy()
    n0, x0, s0 = oracle.verify_round(mode.cpu().numpy(), p, q, tt, ua, ur)
    n1, x1, s1 = gpu_round(bt, mode=mode)
    assert s0 == s1 == sv.STATUS_BAD_MODE
    compare(p, q, ur, mode.cpu().numpy(), K, n0, x0, n1, x1)


def test_zero_mass_paths():
    """Rejection with zero residual falls back to p_i; all-zero rows give -1."""
    B, K, V = 4, 2, 3000
    p = torch.rand(B, K + 1, V, device="cuda")
    q = p[:, :K] * 2.0                     # p <= q everywhere: residual mass is zero
    p[2, 0] = 0.0                           # sequence 2: zero residual and zero p_0
    p[3, K] = 0.0                           # sequence 3: q == p below, bonus row empty
    q[3] = p[3, :K]
    t = torch.randint(0, V, (B, K), device="cuda", dtype=torch.int32)
    ua = torch.full((B, K), 0.999, device="cuda")
    ur = torch.rand(B, dtype=torch.float64, device="cuda")
    n1, x1 = sv.verify_sample(p, q, t, ua, ur)
    st = sv._workspace(None, B, K, V, p.device).status()
    n0, x0, s0 = oracle.verify_sample(p.cpu().numpy(), q.cpu().numpy(), t.cpu().numpy(),
                                      ua.cpu().numpy(), ur.cpu().numpy())
    assert s0 == st == sv.STATUS_ZERO_MASS
    compare(p.cpu().numpy(), q.cpu().numpy(), ur.cpu().numpy(), 1, K, n0, x0,
            n1.cpu().numpy(), x1.cpu().numpy())
    assert x1[2].item() == -1 and x1[3].item() == -1 and n1[3].item() == K


def test_commit_matches_oracle():
    B, K, V, L = 64, 6, 5000, 20
    bt = make_inputs(4, "cuda", seed=61, B=B, V=V, K=K)
    p, q, t, ua, ur, md = bt.numpy()
    rng = np.random.default_rng(3)
    lengths0 = rng.integers(0, 15, size=B).astype(np.int32)
    tokens0 = np.full((B, L), -9, np.int32)
    n0, x0, s0 = oracle.verify_round(md, p, q, t, ua, ur)
    tok_ref, len_ref = tokens0.copy(), lengths0.copy()
    sc = oracle.commit(t, n0, x0, tok_ref, len_ref)
    tok = torch.from_numpy(tokens0).cuda()
    lens = torch.from_numpy(lengths0).cuda()
    n1, x1, s1 = gpu_round(bt, tokens=tok, lengths=lens)
    bnd = compare(p, q, ur, md, K, n0, x0, n1, x1, label="commit")
    assert s1 == (s0 | sc)
    if not bnd:
        assert np.array_equal(tok.cpu().numpy(), tok_ref)
        assert np.array_equal(lens.cpu().numpy(), len_ref)


def test_accept_test_edges_are_exact():
    """u*q against p at the edges of fp32: exact equality of the product, one
    ulp either side, and magnitudes whose difference underflows.  n must match
    the oracle's exact fp64 test bit for bit."""
    rng = np.random.default_rng(17)
    cases = []
    for _ in range(200):   # p exactly equal to the fp32 product u*q, and one ulp either side
        u = np.float32(rng.integers(1, 1 << 24) / (1 << 24))
        q = np.float32(rng.uniform(1e-6, 1e-2))
        prod = np.float32(u * q)
        for p in (prod, np.nextafter(prod, np.float32(1)), np.nextafter(prod, np.float32(0))):
            cases.append((u, q, p))
    for e in (-100, -120, -126, -130, -140, -149):   # tiny magnitudes, products far below p's ulp
        tiny = np.float32(2.0 ** e)
        for u in (np.float32(0.5), np.float32(0.75), np.float32(1 - 2 ** -24)):
            for q in (tiny, np.float32(2 * tiny), np.float32(2.0 ** -60)):
                for p in (tiny, np.float32(0.0), np.nextafter(np.float32(u * q), np.float32(1))):
                    cases.append((u, q, p))
    B, K, V = len(cases), 1, 8
    p = np.full((B, K + 1, V), 1e-3, dtype=np.float32)
    q = np.full((B, K, V), 1e-3, dtype=np.float32)
    t = np.zeros((B, K), dtype=np.int32)
    ua = np.zeros((B, K), dtype=np.float32)
    for b, (u, qt, pt) in enumerate(cases):
        p[b, 0, 0], q[b, 0, 0], ua[b, 0] = pt, qt, u
    ur = np.full(B, 0.5)
    n0, x0, s0 = oracle.verify_sample(p, q, t, ua, ur)
    dev = lambda a: torch.from_numpy(a).cuda()
    n1, x1 = sv.verify_sample(dev(p), dev(q), dev(t), dev(ua), dev(torch.from_numpy(ur).numpy()))
    assert np.array_equal(n0, n1.cpu().numpy())
    assert (n0 == 0).any() and (n0 == 1).any()


def test_boundary_thresholds_are_counted_not_wrong():
    """Uniforms placed exactly on the oracle's CDF boundaries: the GPU may pick
    either neighbour, and every difference must be boundary-explained."""
    B, K, V = 64, 1, 4096
    g = torch.Generator(device="cuda").manual_seed(9)
    p = torch.rand(B, K + 1, V, device="cuda", generator=g)
    q = torch.rand(B, K, V, device="cuda", generator=g)
    t = torch.zeros(B, K, dtype=torch.int32, device="cuda")
    q[:, 0, 0] = 10.0                       # draft token 0 is always rejected
    ua = torch.full((B, K), 0.5, device="cuda")
    ph, qh = p.cpu().numpy(), q.cpu().numpy()
    ur = np.empty(B)
    rng = np.random.default_rng(2)
    for b in range(B):
        C, R = oracle.residual_cumsum(ph[b, 0], qh[b, 0])
        k = int(rng.integers(1, V - 1))
        ur[b] = C[k] / R
    u = torch.from_numpy(ur).cuda()
    n1, x1 = sv.verify_sample(p, q, t, ua, u)
    n0, x0, s0 = oracle.verify_sample(ph, qh, t.cpu().numpy(), ua.cpu().numpy(), ur)
    compare(ph, qh, ur, 1, K, n0, x0, n1.cpu().numpy(), x1.cpu().numpy(),
            label="uniforms on oracle CDF boundaries")


# ---------------------------------------------------------------------------
# full-size workloads (the bench's launch configuration), every output checked

def test_single_sequence_600_rounds():
    """The single-sequence workload: 600 independent B=1 rounds, greedy and sampling."""
    bt = make_inputs(1, "cuda", seed=20261201, B=600)
    check_sample(bt, label="single-seq batch")
    check_greedy(bt)
    p, q, t, ua, ur, md = bt.numpy()
    n0, x0, _ = oracle.verify_sample(p, q, t, ua, ur, nthreads=8)
    for r in range(0, 600, 37):      # the B=1 launch itself
        n1, x1 = sv.verify_sample(bt.p[r:r + 1], bt.q[r:r + 1], bt.t[r:r + 1],
                                  bt.u_acc[r:r + 1], bt.u_res[r:r + 1])
        compare(p[r:r + 1], q[r:r + 1], ur[r:r + 1], 1, 4, n0[r:r + 1], x0[r:r + 1],
                n1.cpu().numpy(), x1.cpu().numpy())


def test_greedy_batched_full():
    bt = make_inputs(2, "cuda")
    n = check_greedy(bt)
    assert bt.meta["planted_rows"] > 0 and bt.meta["higher_dup_drafts"] > 0
    assert len(set(n.tolist())) > 2
    del bt
    _free()


def test_sampling_batched_full():
    """Headline workload B=256, V=128256, K=5: every output against the oracle."""
    bt = make_inputs(3, "cuda")
    host = bt.numpy()
    check_sample(bt, host, label="sampling B=256 V=128256 K=5")
    check_greedy(bt, host)
    del bt
    _free()


def test_sampling_full_fresh_and_reused_workspace():
    """Headline workload on three more seeds, each on a freshly zeroed workspace
    and again on one still holding the previous batch's sums: every stage must
    be reduced before the draw reads its sums, so neither zeros nor another
    batch's sums may reach an output."""
    reused = None
    for seed in (11, 12, 13):
        bt = make_inputs(3, "cuda", seed=seed)
        p, q, t, ua, ur, md = bt.numpy()
        n0, x0, s0 = oracle.verify_sample(p, q, t, ua, ur, nthreads=8)
        fresh = sv.Workspace(bt.B, bt.K, bt.V)
        if reused is None:
            reused = sv.Workspace(bt.B, bt.K, bt.V)
        for ws in (fresh, reused):
            n1, x1 = sv.verify_sample(bt.p, bt.q, bt.t, bt.u_acc, bt.u_res, ws=ws)
            compare(p, q, ur, 1, bt.K, n0, x0, n1.cpu().numpy(), x1.cpu().numpy(), s0,
                    ws.status(), label=f"sampling seed {seed}")
        del bt, fresh
        _free()


def test_workspace_reused_across_sizes():
    """One workspace serves calls of several sizes and both launch paths in turn
    (per-sequence state is laid out by size, so a change of sizes must clear it)."""
    shapes = [(160, 20000, 5), (170, 30000, 3), (40, 50000, 5), (160, 20000, 5), (200, 9000, 8)]
    big = max(sv.workspace_size(B, K, V) for B, V, K in shapes)
    ws = sv.Workspace(1, 1, 1)
    ws.buf = torch.empty(big, dtype=torch.uint8, device="cuda")
    ws.nbytes = big
    assert sv.load().sv_workspace_init(ws.ptr, big, None) == 0
    for i, (B, V, K) in enumerate(shapes):
        bt = make_inputs(4, "cuda", seed=900 + i, B=B, V=V, K=K)
        p, q, t, ua, ur, md = bt.numpy()
        if i % 2 == 0:
            n0, x0, s0 = oracle.verify_greedy(p, t, nthreads=8)
            n1, x1 = sv.verify_greedy(bt.p, bt.t, ws=ws)
            compare(p, q, ur, 0, K, n0, x0, n1.cpu().numpy(), x1.cpu().numpy(), s0, ws.status())
        else:
            n0, x0, s0 = oracle.verify_sample(p, q, t, ua, ur, nthreads=8)
            n1, x1 = sv.verify_sample(bt.p, bt.q, bt.t, bt.u_acc, bt.u_res, ws=ws)
            compare(p, q, ur, 1, K, n0, x0, n1.cpu().numpy(), x1.cpu().numpy(), s0,
                    ws.status(), label=f"reused workspace {B}x{V}")


def test_implicit_workspaces_are_per_stream():
    """Calls that share a workspace must be ordered on one stream, so the
    binding keeps one implicit workspace per (sizes, stream)."""
    dev = torch.device("cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    w1 = sv._workspace(None, 4, 3, 1000, dev, s1)
    w2 = sv._workspace(None, 4, 3, 1000, dev, s2)
    assert w1 is not w2
    assert sv._workspace(None, 4, 3, 1000, dev, s1) is w1
    assert sv._workspace(None, 4, 3, 1000, dev) is not w1   # the current stream
    torch.cuda.synchronize()


@pytest.mark.parametrize("mapped", [True, False])
def test_host_resident_inputs(mapped):
    """Inputs in pinned host memory, read in place (mapped) or copied first:
    the same outputs as the oracle, through the public HostVerifier."""
    B, V, K = 160, 20000, 5
    bt = make_inputs(3, "cuda", seed=1700, B=B, V=V, K=K)
    p, q, t, ua, ur, md = bt.numpy()
    hp, hq = bt.p.cpu().pin_memory(), bt.q.cpu().pin_memory()
    ht, hua, hur = bt.t.cpu().pin_memory(), bt.u_acc.cpu().pin_memory(), bt.u_res.cpu().pin_memory()
    hv = sv.HostVerifier(B, K, V, sampling=True, mapped=mapped)
    n1, x1 = hv.sample(hp, hq, ht, hua, hur)
    n0, x0, s0 = oracle.verify_sample(p, q, t, ua, ur, nthreads=8)
    compare(p, q, ur, 1, K, n0, x0, n1.numpy().copy(), x1.numpy().copy(), s0,
            hv.ws.status(), label=f"host inputs mapped={mapped}")
    assert hv.h2d_bytes() > 0
    hg = sv.HostVerifier(B, K, V, sampling=False, mapped=mapped)
    n1, x1 = hg.greedy(hp, ht)
    n0, x0, s0 = oracle.verify_greedy(p, t, nthreads=8)
    compare(p, q, ur, 0, K, n0, x0, n1.numpy().copy(), x1.numpy().copy(), s0, hg.ws.status())
    if mapped:
        assert sv.last_kernel_count() == 3  # host rows take the plain-load chain


def test_pageable_host_memory_rejected():
    """A pageable CPU array is refused on the host, before anything runs."""
    B, V, K = 4, 1000, 2
    lib = sv.load()
    p = torch.rand(B, K + 1, V)            # pageable
    t = torch.zeros(B, K, dtype=torch.int32, device="cuda")
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    nx = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = sv.Workspace(B, K, V)
    rc = lib.sv_verify_greedy(ctypes.c_void_p(p.data_ptr()), V, ctypes.c_void_p(t.data_ptr()),
                              B, K, V, ctypes.c_void_p(n.data_ptr()),
                              ctypes.c_void_p(nx.data_ptr()), ws.ptr, ws.nbytes, None)
    assert rc == sv.SV_EINVAL
    with pytest.raises(sv.SpecVerifyError):
        sv.verify_greedy(p, t)


def test_mixed_round_full():
    bt = make_inputs(4, "cuda")
    p, q, t, ua, ur, md = bt.numpy()
    n0, x0, s0 = oracle.verify_round(md, p, q, t, ua, ur, nthreads=16)
    n1, x1, s1 = gpu_round(bt)
    compare(p, q, ur, md, bt.K, n0, x0, n1, x1, s0, s1,
            label="mixed B=1024")
    counts = np.bincount(n0, minlength=bt.K + 1)
    assert counts[0] > 0 and counts[bt.K] > 0
    del bt
    _free()


@pytest.mark.parametrize("V", [131072 + 9 * 1024 + 4, 300000])  # rows 16-byte aligned
def test_item_path_rows_in_several_items(V):
    """Rows longer than one sampling item (128 segments of 1024) on the
    single-launch item kernel (160 sequences, more than the SMs): a residual row's
    sums then come from several CTAs, and the last item to retire draws."""
    B, K = 160, 2
    bt = make_inputs(3, "cuda", seed=V % 1000, B=B, V=V, K=K)
    host = bt.numpy()
    check_sample(bt, host, label=f"rows in several items V={V}")
    assert sv.last_kernel_count() == 1
    check_greedy(bt, host)
    p, q, t, ua, ur, _ = host
    md = (np.arange(B) % 2).astype(np.uint8)
    n0, x0, s0 = oracle.verify_round(md, p, q, t, ua, ur, nthreads=8)
    n1, x1, s1 = gpu_round(bt, mode=torch.from_numpy(md).cuda())
    compare(p, q, ur, md, K, n0, x0, n1, x1, s0, s1,
            label=f"rows in several items V={V}")
    del bt
    _free()


def _mode_pattern(pattern, B, seed):
    rng = np.random.default_rng(seed)
    if pattern == "all_greedy":
        m = np.zeros(B, np.uint8)
    elif pattern == "all_sample":
        m = np.ones(B, np.uint8)
    elif pattern == "alternate":
        m = (np.arange(B) % 2).astype(np.uint8)
    elif pattern == "sample_block_first":
        m = (np.arange(B) < B // 3).astype(np.uint8)
    else:  # random, with a few invalid modes
        m = rng.integers(0, 2, size=B).astype(np.uint8)
        m[rng.choice(B, size=5, replace=False)] = [2, 255, 7, 2, 128]
    return m


@pytest.mark.parametrize("B,V,pattern", [
    (777, 6000, "all_greedy"), (777, 6000, "all_sample"), (777, 6000, "alternate"),
    (777, 6000, "sample_block_first"), (777, 6000, "invalid"), (5003, 700, "alternate"),
    (5003, 700, "invalid")])
def test_mixed_round_item_path_mode_patterns(B, V, pattern):
    """On aligned device rows a mixed round is the ordering kernel and one item
    launch that takes the greedy sequences first; every mode pattern (including invalid
    modes, and B not a multiple of the ordering kernel's threads) gives the
    oracle's outputs and commit, sequence by sequence."""
    K, L = 5, 12
    bt = make_inputs(4, "cuda", seed=4100 + B + len(pattern), B=B, V=V, K=K)
    md = _mode_pattern(pattern, B, seed=B)
    mode = torch.from_numpy(md).cuda()
    p, q, t, ua, ur, _ = bt.numpy()
    rng = np.random.default_rng(11)
    lengths0 = rng.integers(0, 6, size=B).astype(np.int32)
    tokens0 = np.full((B, L), -9, np.int32)
    n0, x0, s0 = oracle.verify_round(md, p, q, t, ua, ur, nthreads=8)
    tok_ref, len_ref = tokens0.copy(), lengths0.copy()
    oracle.commit(t, n0, x0, tok_ref, len_ref)
    tok = torch.from_numpy(tokens0).cuda()
    lens = torch.from_numpy(lengths0).cuda()
    for _ in range(2):  # the second call reuses the workspace the first left
        tok.copy_(torch.from_numpy(tokens0))
        lens.copy_(torch.from_numpy(lengths0))
        n1, x1, s1 = gpu_round(bt, mode=mode, tokens=tok, lengths=lens)
        assert sv.last_kernel_count() == 2, "expected the ordering kernel and the item kernel"
        compare(p, q, ur, md, K, n0, x0, n1, x1, s0, s1,
                label=f"mixed {pattern} B={B}")
        same = x1 == x0  # a boundary-explained draw commits the GPU's own token
        np.testing.assert_array_equal(lens.cpu().numpy(), len_ref)
        np.testing.assert_array_equal(tok.cpu().numpy()[same], tok_ref[same])
    if pattern == "invalid":
        assert s1 == sv.STATUS_BAD_MODE


def test_edge_full():
    bt = make_inputs(5, "cuda")
    host = bt.numpy()
    n = check_sample(bt, host, label="edge B=128 V=262144 K=16")
    check_greedy(bt, host)
    assert np.all(n[bt.meta["same"]] == 16)
    del bt
    _free()


def test_empty_batch_every_entry_point():
    """B = 0 is a valid call: nothing is launched and nothing is written."""
    bt = make_inputs(3, "cuda", seed=9, B=3, V=2000, K=4)
    p, q, t, ua, ur = bt.p[:0], bt.q[:0], bt.t[:0], bt.u_acc[:0], bt.u_res[:0]
    for n, nx in (sv.verify_greedy(p, t), sv.verify_sample(p, q, t, ua, ur),
                  sv.verify_round(bt.mode[:0], p, q, t, ua, ur)):
        assert n.numel() == 0 and nx.numel() == 0
    a, e = sv.alpha(p, q)
    assert a.numel() == 0 and e.numel() == 0
