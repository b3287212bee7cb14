"""Acceptance-rate diagnostic on the GPU against the oracle: alpha within the
bound the arithmetic gives (two fp32 roundings per term, 2 * 2^-24 * alpha
~ 1.2e-7; tested at 1e-6), the expected length within K times that."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_08_gb300 as sv
from speculative_decoding_verification_08_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

ALPHA_TOL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.build()
    sv.load()


def check(p, q):
    a1, e1 = sv.alpha(p, q)
    a0, e0 = oracle.alpha(p.cpu().numpy(), q.cpu().numpy())
    a1, e1 = a1.cpu().numpy(), e1.cpu().numpy()
    K = a0.shape[1]
    assert np.abs(a1 - a0).max() <= ALPHA_TOL, np.abs(a1 - a0).max()
    assert np.abs(e1 - e0).max() <= K * ALPHA_TOL, np.abs(e1 - e0).max()
    return a0


@pytest.mark.parametrize("cfg,B,V,K", [(3, 40, 20000, 5), (1, 3, 32000, 4), (4, 24, 9000, 8),
                                       (5, 16, 50003, 16), (3, 7, 1, 2), (3, 5, 1021, 64)])
def test_alpha_matches_oracle(cfg, B, V, K):
    bt = make_inputs(cfg, "cuda", seed=4100 + cfg, B=B, V=V, K=K)
    a = check(bt.p, bt.q)
    assert ((a >= 0) & (a <= 1 + 1e-12)).all()


def test_alpha_headline_shape():
    """The sampling workload's full shape (B=256, V=128256, K=5)."""
    bt = make_inputs(3, "cuda")
    check(bt.p, bt.q)


def test_alpha_edge_rows_and_strides():
    B, K, V = 6, 3, 3001
    g = torch.Generator(device="cuda").manual_seed(5)
    p = torch.rand(B, K + 1, V + 5, device="cuda", generator=g)[..., 1:V + 1]   # unaligned rows
    q = torch.rand(B, K, V + 3, device="cuda", generator=g)[..., :V]
    p[0, 0] = q[0, 0] * 4.0          # identical after (exact) scaling: alpha = 1
    p[1, 1] = 0.0                    # zero row: alpha = 0
    q[2, 0, : V // 2] = 0.0          # disjoint supports: alpha = 0
    p[2, 0, V // 2:] = 0.0
    a = check(p, q)
    assert abs(a[0, 0] - 1) < 1e-12 and a[1, 1] == 0 and a[2, 0] == 0


def test_alpha_matches_the_sampler_mean():
    """The GPU's expected length against the mean accepted length of the GPU
    sampler over many rounds of the same rows (the law, end to end)."""
    R, K, V = 3000, 4, 512
    g = torch.Generator(device="cuda").manual_seed(11)
    zp = torch.randn(K + 1, V, device="cuda", generator=g) * 1.5
    p = torch.softmax(zp, -1)
    q = torch.softmax(zp[:K] + 0.6 * torch.randn(K, V, device="cuda", generator=g), -1)
    a, e = sv.alpha(p[None].contiguous(), q[None].contiguous())
    pp = p.expand(R, K + 1, V).contiguous()
    qq = q.expand(R, K, V).contiguous()
    t = torch.stack([torch.multinomial(q[i], R, replacement=True, generator=g) for i in range(K)], 1)
    ua = torch.rand(R, K, device="cuda", generator=g)
    ur = torch.rand(R, device="cuda", generator=g, dtype=torch.float64)
    n, _ = sv.verify_sample(pp, qq, t.to(torch.int32).contiguous(), ua, ur)
    a = a[0].cpu().numpy()
    probs, pre = [], 1.0
    for m in range(K):
        probs.append(pre * (1 - a[m]))
        pre *= a[m]
    probs.append(pre)
    probs = np.array(probs)
    mean = float(e[0])
    var = float((probs * np.arange(K + 1) ** 2).sum() - mean ** 2)
    z = (n.double().mean().item() - mean) / np.sqrt(var / R)
    assert abs(z) < 4.0, (n.double().mean().item(), mean, z)


def test_alpha_host_arguments_checked():
    lib = sv.load()
    ws = sv.Workspace(2, 2, 10)
    x = torch.empty(2, dtype=torch.float64, device="cuda")
    rc = lib.sv_alpha(None, 10, None, 10, 2, 2, 10, ctypes.c_void_p(x.data_ptr()), None, ws.ptr,
                      ws.nbytes, None)
    assert rc == sv.SV_EINVAL
