"""Sampling verification from logits on the GPU against the oracle's fp64
softmax: every accept decision (n) equals the oracle's but where the two fp64
computations may round to different sides (|u*q - p| <= 1e-9 p), and drawn
tokens differ only within the draw tolerance of the fp32 warp
(oracle/compare.py); such cases are counted.  Greedy from logits is
bit-exact."""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.compare import compare_logits
import speculative_decoding_verification_08_gb300 as sv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.build()
    sv.load()


def make_logits(B, V, K, tau, seed, target_std=2.0, noise=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    zp = torch.randn(B, K + 1, V, device="cuda", generator=g) * target_std
    zq = zp[:, :K] + noise * torch.randn(B, K, V, device="cuda", generator=g)
    if K > 0:
        q = torch.softmax(zq.double() / tau, -1)
        t = torch.multinomial(q.reshape(B * K, V).float(), 1, generator=g).reshape(B, K)
    else:
        t = torch.zeros(B, 0, dtype=torch.int64, device="cuda")
    ua = torch.rand(B, K, device="cuda", generator=g)
    ur = torch.rand(B, device="cuda", generator=g, dtype=torch.float64)
    return zp.contiguous(), zq.contiguous(), t.to(torch.int32).contiguous(), ua, ur


def tau32(tau):
    """The temperature as the C ABI takes it (a float): the oracle is given
    the same value."""
    return float(np.float32(tau))


def run(zp, zq, t, ua, ur, tau):
    """GPU against the oracle: returns (the oracle's n, the explained
    differences); accept decisions may differ only inside the fp64 band."""
    n1, x1 = sv.verify_sample_logits(zp, zq, t, ua, ur, tau)
    h = [x.cpu().numpy() for x in (zp, zq, t, ua, ur)]
    n0, x0, s0 = oracle.verify_sample_logits(*h, tau32(tau))
    assert s0 == 0
    expl = compare_logits(h[0], h[1], tau32(tau), h[2], h[3], h[4], n0, x0, n1.cpu().numpy(),
                          x1.cpu().numpy())
    return n0, expl


def draws(expl):
    return [e for e in expl if e[1] == "draw"]


# (64, 32000, 4): mass groups deferred and two-position groups at once; (8, 2000, 48): chains of up
# to 49 steps, draft ids past the first 32
@pytest.mark.parametrize("B,V,K,tau", [(64, 4096, 4, 1.0), (33, 20011, 5, 0.7), (8, 1, 3, 1.0),
                                       (16, 50000, 8, 1.6), (5, 3000, 0, 1.0), (9, 777, 16, 0.5),
                                       (64, 32000, 4, 1.0), (8, 2000, 48, 1.0)])
def test_logits_match_oracle(B, V, K, tau):
    zp, zq, t, ua, ur = make_logits(B, V, K, tau, seed=7000 + V + K)
    n0, expl = run(zp, zq, t, ua, ur, tau)
    assert len(draws(expl)) <= max(1, B // 20), expl
    if K > 0 and V > 1:
        assert len(set(n0.tolist())) > 1


def test_logits_headline_shape():
    """B=256, V=128256, K=5 logits, the warp at T=1."""
    zp, zq, t, ua, ur = make_logits(256, 128256, 5, 1.0, seed=20261203)
    n0, expl = run(zp, zq, t, ua, ur, 1.0)
    assert len(draws(expl)) <= 6, expl
    counts = np.bincount(n0, minlength=6)
    assert counts[0] > 0 and counts[5] > 0


def test_logits_unaligned_rows_and_equal_rows():
    B, V, K, tau = 12, 3001, 3, 1.0
    zp, zq, t, ua, ur = make_logits(B, V + 1, K, tau, seed=99)
    zp = zp[..., 1:]          # rows start off a 16-byte boundary
    zq = zq[..., 1:]
    t = torch.clamp(t, max=V - 1)
    zq[0] = zp[0, :K]         # identical rows: every draft accepted
    n0, expl = run(zp, zq, t, ua, ur, tau)
    assert n0[0] == K and len(draws(expl)) <= 1


def test_greedy_from_logits_is_exact():
    """argmax softmax(z/T) = argmax z: the greedy entry point on raw logits
    (negative values, planted ties) equals the oracle's greedy on the same."""
    B, V, K = 40, 5000, 4
    g = torch.Generator(device="cuda").manual_seed(3)
    zp = torch.randn(B, K + 1, V, device="cuda", generator=g) * 3 - 5
    am = zp.argmax(-1)
    t = am[:, :K].clone()
    t[::3, 1] = (t[::3, 1] + 1) % V          # some misses
    dup = torch.arange(0, B, 4, device="cuda")
    zp[dup, 0, 17] = zp[dup, 0].max(-1).values   # exact ties, lowest index wins
    n1, x1 = sv.verify_greedy(zp, t.to(torch.int32).contiguous())
    n0, x0, s0 = oracle.verify_greedy(zp.cpu().numpy(), t.to(torch.int32).cpu().numpy())
    assert np.array_equal(n1.cpu().numpy(), n0) and np.array_equal(x1.cpu().numpy(), x0)


@pytest.mark.parametrize("tau", [0.0, -1.0, float("inf"), float("nan")])
def test_bad_temperature_rejected(tau):
    zp, zq, t, ua, ur = make_logits(2, 100, 2, 1.0, seed=1)
    with pytest.raises(sv.SpecVerifyError):
        sv.verify_sample_logits(zp, zq, t, ua, ur, tau)


def test_repeated_calls_reuse_the_workspace_cleanly():
    """The queue counters, group records and arrival counts return to zero at
    the end of every call: repeated calls on one workspace, alternating inputs
    and sizes, give the same outputs and no status bits."""
    B, V, K, tau = 160, 6000, 4, 1.0
    a = make_logits(B, V, K, tau, seed=41)
    b = make_logits(B, V, K, tau, seed=42)
    small = make_logits(9, 2500, 2, tau, seed=43)
    ws = sv.Workspace(B, K, V)
    first = {}
    for r in range(3):
        for name, x in (("a", a), ("b", b)):
            n, nx = sv.verify_sample_logits(*x, tau, ws=ws)
            got = (n.cpu().numpy(), nx.cpu().numpy())
            if r == 0:
                first[name] = got
                run(*x, tau)      # the oracle agrees with the first call
            else:
                assert np.array_equal(got[0], first[name][0])
                assert np.array_equal(got[1], first[name][1])
        sv.verify_sample_logits(*small, tau)   # another size on its own workspace in between
    assert ws.status() == 0


def test_plain_load_workers_at_a_large_batch():
    """Rows off a 16-byte boundary take the plain-load workers; here with more
    sequences than SMs, so the queue runs many groups at once."""
    B, V, K, tau = 200, 4001, 4, 0.9
    zp, zq, t, ua, ur = make_logits(B, V + 1, K, tau, seed=77)
    zp = zp[..., 1:]
    zq = zq[..., 1:]
    t = torch.clamp(t, max=V - 1)
    n0, expl = run(zp, zq, t, ua, ur, tau)
    assert len(draws(expl)) <= 2, expl
    assert len(set(n0.tolist())) > 2


@pytest.mark.parametrize("aligned", [True, False])
def test_deferred_mass_groups_on_both_worker_kernels(aligned):
    """At batches whose first groups alone give every worker a claim, each
    sequence's mass group (its chain's last step) waits in a pending list
    until a worker finds no other work.  On both worker kernels the outputs
    equal the oracle's, and a second call on the same workspace gives the same
    outputs (the pending list and its counters are back at zero after a call)."""
    K, tau = 4, 1.0
    B, V = (400, 40000) if aligned else (240, 40001)
    zp, zq, t, ua, ur = make_logits(B, V + (0 if aligned else 1), K, tau, seed=8100 + B)
    if not aligned:
        zp = zp[..., 1:]   # rows off a 16-byte boundary: the plain-load workers
        zq = zq[..., 1:]
        t = torch.clamp(t, max=V - 1)
    ws = sv.Workspace(B, K, V)
    n1, x1 = sv.verify_sample_logits(zp, zq, t, ua, ur, tau, ws=ws)
    grid = sv.last_grid_size()
    nseg = -(-V // 1024)
    claims, workers = (-(-nseg // 16), grid) if aligned else (nseg, grid * 8)
    assert B * claims >= workers, "this size must take the deferring schedule"
    h = [x.cpu().numpy() for x in (zp, zq, t, ua, ur)]
    n0, x0, s0 = oracle.verify_sample_logits(*h, tau32(tau))
    assert s0 == 0
    expl = compare_logits(h[0], h[1], tau32(tau), h[2], h[3], h[4], n0, x0, n1.cpu().numpy(),
                          x1.cpu().numpy())
    assert len(draws(expl)) <= 2, expl
    n2, x2 = sv.verify_sample_logits(zp, zq, t, ua, ur, tau, ws=ws)
    assert torch.equal(n1, n2) and torch.equal(x1, x2)
    assert ws.status() == 0


@pytest.mark.parametrize("B,V", [(6000, 20011), (1400, 40011)])
def test_large_batch_takes_whole_chunks(B, V):
    """A batch whose first groups give every bulk-copy worker at least 4
    claims of 32 segments moves 32-segment chunks (smaller batches take 8 or
    4, which the other tests cover).  V=20011: each row is one ragged chunk of
    20 segments, the last of them partial; V=40011: a whole chunk and a ragged
    one.  The outputs equal the oracle's."""
    K, tau = 2, 1.0
    zp, zq, t, ua, ur = make_logits(B, V + 1, K, tau, seed=8300 + B)
    zp, zq = zp[..., :V], zq[..., :V]   # row stride V + 1: 16-byte aligned rows
    t = torch.clamp(t, max=V - 1)
    n0, expl = run(zp, zq, t, ua, ur, tau)
    nseg = -(-V // 1024)
    assert B * -(-nseg // 32) >= 4 * sv.last_grid_size(), "this size must take 32-segment chunks"
    assert len(draws(expl)) <= max(1, B // 2000), expl
    assert len(set(n0.tolist())) == K + 1


def test_empty_batch():
    zp, zq, t, ua, ur = make_logits(1, 100, 3, 1.0, seed=5)
    n, nx = sv.verify_sample_logits(zp[:0], zq[:0], t[:0], ua[:0], ur[:0], 1.0)
    assert n.numel() == 0 and nx.numel() == 0


def test_pinned_host_rows():
    """Logits in page-locked host memory are read in place by the plain-load
    workers (no copy).  With 16-byte-aligned rows the same rows on the device
    take the bulk-copy workers, so equal outputs also check that the two
    kernels compute bit for bit the same."""
    B, V, K, tau = 24, 5004, 3, 1.1
    zp, zq, t, ua, ur = make_logits(B, V, K, tau, seed=61)
    n1, x1 = sv.verify_sample_logits(zp, zq, t, ua, ur, tau)
    hp, hq = zp.cpu().pin_memory(), zq.cpu().pin_memory()
    ht, hua, hur = t.cpu().pin_memory(), ua.cpu().pin_memory(), ur.cpu().pin_memory()
    n2, x2 = sv.verify_sample_logits(hp, hq, ht, hua, hur, tau)
    assert np.array_equal(n1.cpu().numpy(), n2.cpu().numpy())
    assert np.array_equal(x1.cpu().numpy(), x2.cpu().numpy())
    run(zp, zq, t, ua, ur, tau)


def test_timeout_is_reported_and_the_context_stays_usable():
    """A bounded wait that runs out ends the launch with SV_STATUS_TIMEOUT --
    no hang, no fault -- and once the workspace is initialised again the same
    context verifies correctly.  The wait is made to run out by presetting the
    workspace's count of appended groups (the u64 at byte 24 of its header)
    past the group list: every append then falls outside the list and is
    dropped (SV_STATUS_OVERFLOW), so the workers wait for groups that never
    come, each for the 250 ms limit."""
    SV_STATUS_OVERFLOW, SV_STATUS_TIMEOUT = 4, 16
    B, V, K, tau = 32, 4096, 3, 1.0
    x = make_logits(B, V, K, tau, seed=5150)
    ws = sv.Workspace(B, K, V)
    ws.buf.view(torch.int64)[3] = 1 << 40
    sv.verify_sample_logits(*x, tau, ws=ws)
    st = ws.status()
    assert st & SV_STATUS_TIMEOUT and st & SV_STATUS_OVERFLOW, st
    # the context is fine: initialise the workspace again and verify
    assert sv.load().sv_workspace_init(ws.ptr, ctypes.c_size_t(ws.nbytes), None) == 0
    n1, x1 = sv.verify_sample_logits(*x, tau, ws=ws)
    assert ws.status() == 0
    n2, x2 = sv.verify_sample_logits(*x, tau)     # a fresh workspace: the same bits
    assert np.array_equal(n1.cpu().numpy(), n2.cpu().numpy())
    assert np.array_equal(x1.cpu().numpy(), x2.cpu().numpy())
    n0, expl = run(*x, tau)
    assert len(draws(expl)) <= 1


@pytest.mark.parametrize("shift,pos", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_near_threshold_accept_tests_are_decided_exactly(shift, pos):
    """Uniforms placed within an ulp of the accept threshold p/q of position
    pos (p, q the oracle's fp64 softmax at the draft token): far inside the
    fast fp32 test's error bound, so every such test is made again in fp64,
    and n must equal the oracle's for every sequence but inside the 1e-9
    band.  shift=1 starts the rows off a 16-byte boundary (plain-load
    workers).  pos=1 accepts position 0 (u = 0) and tests position 1, whose
    group may also cover position 2 at this small batch: a recheck there
    leaves the second position's normalisers unused."""
    B, V, K, tau = 96, 7001, 3, 0.9
    zp, zq, t, ua, ur = make_logits(B, V + shift, K, tau, seed=4242 + shift + 10 * pos)
    if shift:
        zp, zq = zp[..., shift:], zq[..., shift:]
        t = torch.clamp(t, max=V - 1)
    hp, hq, ht = zp.cpu().numpy(), zq.cpu().numpy(), t.cpu().numpy()
    u = ua.cpu().numpy().copy()
    placed = 0
    for b in range(B):
        if pos == 1:
            u[b, 0] = 0.0
        x = int(ht[b, pos])
        r = oracle.softmax(hp[b, pos], tau32(tau))[x] / oracle.softmax(hq[b, pos], tau32(tau))[x]
        if r < 0.999:
            u0 = np.float32(r)
            u[b, pos] = [np.nextafter(u0, np.float32(0)), u0, np.nextafter(u0, np.float32(1))][b % 3]
            placed += 1
    assert placed >= B // 5
    n0, expl = run(zp, zq, t, torch.from_numpy(u).cuda(), ur, tau)
    assert not [e for e in expl if e[1] == "accept"], expl
    assert 0 < (n0 == pos).sum() < B and (n0 >= pos).all()


def test_ex2_approx_error_is_within_the_assumed_bound(tmp_path):
    """The logits kernels decide an accept test in fp32 only when its margin
    exceeds an error bound that assumes ex2.approx.f32 is within 2^-20 of
    2^a (relative).  Measured here against fp64 exp2 over 2^27 arguments in
    [-100, 0]: the worst case must be at most half of that."""
    import subprocess
    from speculative_decoding_verification_08_gb300 import _build
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "probes", "ex2_probe.cu")
    so = str(tmp_path / "ex2_probe.so")
    subprocess.run([_build.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                    "-Xcompiler", "-fPIC", "-shared", "-o", so, src], check=True)
    lib = ctypes.CDLL(so)
    worst = ctypes.c_double(-1.0)
    assert lib.ex2_worst_relative_error(ctypes.byref(worst)) == 0
    assert 0.0 < worst.value <= 2.0 ** -21, worst.value
