"""Seeded synthetic inputs for batched speculative-decoding verification.

This module builds target probabilities p [B][K+1][V], draft probabilities
q [B][K][V], draft tokens t [B][K], uniforms u_accept [B][K] (f32) and
u_resample [B] (f64), and a per-sequence mode [B] (0 greedy, 1 sampling).
It holds none of the verification arithmetic: it only draws random numbers and
shapes them into the five workloads below, so both the CUDA path and the CPU
oracle can be fed the same tensors.

The pages measure on a Raspberry Pi with "a deliberately imperfect draft" and
no public dataset ("spec-verify" page, section "Measured"); these seeded
distributions stand in for model outputs.

Workloads (sizes can be overridden to build scaled-down cases with the same
value distributions):

1. single sequence: B=1, V=32000, K=4, one fresh round per call; target logits
   N(0, 2^2), draft logits = target logits + N(0, 0.82^2); both softmaxed;
   t ~ q, uniforms U[0, 1).  The workload is specified by its acceptance rate
   alpha = sum(min(p, q)) ~ 0.68 (the page's 0.678); a draft noise of 0.82
   gives that (the 1.2 quoted beside it gives alpha ~ 0.55).
2. greedy batched: B=64, V=32000, K=4; p = softmax(N(0, 3^2)); t_i is the
   target argmax with probability 0.7, else a uniform other id; 5% of rows get
   an exact duplicate of their maximum at a random other index, and for half of
   those (with a draft position) the draft token is the higher duplicate.
3. sampling batched: B=256, V=128256, K=5; p = softmax(N(0, 2^2));
   q = softmax(target logits + N(0, 1^2)); t ~ q.
4. large mixed batch: B=1024, V=128256, K=8; as 3 but the draft noise std is
   U[0.3, 2.5] per sequence; mode = b mod 2; greedy sequences draft with
   t_i = argmax(q_i) (a temperature-0 drafter), sampling sequences t_i ~ q_i.
5. long draft and edge cases: B=128, V=262144, K=16; as 3, then every p and q
   row is multiplied by U[0.5, 2]; 10% of sequences have q == p (rows and
   scale identical); 10% have a one-hot target (times its row factor); 5% have
   a residual max(0, p - q) that is non-zero at one token only.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

SEED_BASE = 20261200

CONFIGS = {
    1: dict(B=1, V=32000, K=4, name="single-seq B=1 V=32000 K=4"),
    2: dict(B=64, V=32000, K=4, name="greedy-batched B=64 V=32000 K=4"),
    3: dict(B=256, V=128256, K=5, name="sampling-batched B=256 V=128256 K=5"),
    4: dict(B=1024, V=128256, K=8, name="mixed B=1024 V=128256 K=8"),
    5: dict(B=128, V=262144, K=16, name="edge B=128 V=262144 K=16"),
}


@dataclass
class Batch:
    cfg: int
    B: int
    K: int
    V: int
    p: torch.Tensor                 # [B][K+1][V] f32
    t: torch.Tensor                 # [B][K] i32
    q: Optional[torch.Tensor]       # [B][K][V] f32 (None for greedy-only inputs)
    u_acc: torch.Tensor             # [B][K] f32 in [0,1)
    u_res: torch.Tensor             # [B] f64 in [0,1)
    mode: torch.Tensor              # [B] u8: 0 greedy, 1 sampling
    meta: dict = field(default_factory=dict)

    def to(self, device, non_blocking=False):
        mv = lambda x: None if x is None else x.to(device, non_blocking=non_blocking)
        return Batch(self.cfg, self.B, self.K, self.V, mv(self.p), mv(self.t), mv(self.q),
                     mv(self.u_acc), mv(self.u_res), mv(self.mode), dict(self.meta))

    def numpy(self):
        """Host numpy copies (p, q, t, u_acc, u_res, mode); q may be None."""
        cv = lambda x: None if x is None else x.detach().cpu().numpy()
        return (cv(self.p), cv(self.q), cv(self.t), cv(self.u_acc), cv(self.u_res),
                cv(self.mode))


def _block(B, V, K):
    """Sequences generated per block: bounds the temporaries to ~1 GiB."""
    per_seq = (2 * K + 1) * V * 4 * 3
    return max(1, min(B, (1 << 30) // max(per_seq, 1)))


def _sample_rows(q, gen):
    """One draw per row of q [N][V] (unnormalised rows allowed)."""
    return torch.multinomial(q, 1, generator=gen).squeeze(1)


def _logit_pair(nb, K, V, sig_t, sig_d, gen, device):
    """Target logits [nb][K+1][V] and draft logits [nb][K][V]; sig_d is a float or [nb]."""
    lt = torch.randn(nb, K + 1, V, generator=gen, device=device) * sig_t
    nz = torch.randn(nb, K, V, generator=gen, device=device)
    if isinstance(sig_d, torch.Tensor):
        nz.mul_(sig_d.view(nb, 1, 1))
    else:
        nz.mul_(sig_d)
    ld = lt[:, :K] + nz
    del nz
    return lt, ld


def _uniforms(B, K, gen, device):
    u_acc = torch.rand(B, K, generator=gen, device=device, dtype=torch.float32)
    u_res = torch.rand(B, generator=gen, device=device, dtype=torch.float64)
    return u_acc, u_res


def _gen_sampling(B, V, K, sig_t, sig_d, gen, device, greedy_draft_mask=None):
    p = torch.empty(B, K + 1, V, device=device, dtype=torch.float32)
    q = torch.empty(B, K, V, device=device, dtype=torch.float32)
    t = torch.empty(B, K, device=device, dtype=torch.int32)
    blk = _block(B, V, K)
    for b0 in range(0, B, blk):
        b1 = min(B, b0 + blk)
        sd = sig_d[b0:b1] if isinstance(sig_d, torch.Tensor) else sig_d
        lt, ld = _logit_pair(b1 - b0, K, V, sig_t, sd, gen, device)
        p[b0:b1] = torch.softmax(lt, dim=-1)
        del lt
        qb = torch.softmax(ld, dim=-1)
        del ld
        q[b0:b1] = qb
        tb = _sample_rows(qb.reshape(-1, V), gen).view(b1 - b0, K)
        if greedy_draft_mask is not None:
            gm = greedy_draft_mask[b0:b1]
            if bool(gm.any()):
                tg = qb.argmax(dim=-1)
                tb = torch.where(gm.view(-1, 1), tg, tb)
        t[b0:b1] = tb.to(torch.int32)
        del qb
    return p, q, t


def _cfg1_or_3(B, V, K, sig_t, sig_d, gen, device):
    p, q, t = _gen_sampling(B, V, K, sig_t, sig_d, gen, device)
    u_acc, u_res = _uniforms(B, K, gen, device)
    mode = torch.ones(B, dtype=torch.uint8, device=device)
    return p, q, t, u_acc, u_res, mode, {}


def _cfg2(B, V, K, gen, device):
    p = torch.softmax(torch.randn(B, K + 1, V, generator=gen, device=device) * 3.0, dim=-1)
    a = p.argmax(dim=-1)                                     # [B][K+1]
    hit = torch.rand(B, K, generator=gen, device=device) < 0.7
    other = (a[:, :K] + torch.randint(1, max(V, 2), (B, K), generator=gen, device=device)) % V
    t = torch.where(hit, a[:, :K], other)
    # exact duplicate of the row maximum at a random other index in 5% of rows
    rows = B * (K + 1)
    planted = torch.rand(rows, generator=gen, device=device) < 0.05
    d = (a.reshape(-1) + torch.randint(1, max(V, 2), (rows,), generator=gen, device=device)) % V
    flip = torch.rand(rows, generator=gen, device=device) < 0.5
    pf = p.view(rows, V)
    idx = planted.nonzero().squeeze(1)
    if idx.numel():
        pf[idx, d[idx]] = pf[idx, a.reshape(-1)[idx]]
    # for half of the planted rows with a draft position, draft the higher duplicate
    hi_dup = torch.maximum(a.reshape(-1), d).view(B, K + 1)[:, :K]
    use_hi = (planted & flip).view(B, K + 1)[:, :K]
    t = torch.where(use_hi, hi_dup, t).to(torch.int32)
    u_acc, u_res = _uniforms(B, K, gen, device)
    mode = torch.zeros(B, dtype=torch.uint8, device=device)
    meta = dict(planted_rows=int(planted.sum()), higher_dup_drafts=int(use_hi.sum()))
    return p, None, t, u_acc, u_res, mode, meta


def _cfg4(B, V, K, gen, device):
    sig_d = torch.empty(B, device=device).uniform_(0.3, 2.5, generator=gen)
    mode = (torch.arange(B, device=device) % 2).to(torch.uint8)
    p, q, t = _gen_sampling(B, V, K, 2.0, sig_d, gen, device,
                            greedy_draft_mask=(mode == 0))
    u_acc, u_res = _uniforms(B, K, gen, device)
    return p, q, t, u_acc, u_res, mode, dict(sig_d_min=float(sig_d.min()),
                                             sig_d_max=float(sig_d.max()))


def _cfg5(B, V, K, gen, device):
    p, q, t = _gen_sampling(B, V, K, 2.0, 1.0, gen, device)
    p.mul_(torch.empty(B, K + 1, 1, device=device).uniform_(0.5, 2.0, generator=gen))
    q.mul_(torch.empty(B, K, 1, device=device).uniform_(0.5, 2.0, generator=gen))
    perm = torch.randperm(B, generator=gen, device=device)
    n10, n5 = max(1, B // 10), max(1, B // 20)
    same = perm[:n10]
    onehot = perm[n10:2 * n10]
    single = perm[2 * n10:2 * n10 + n5]
    if same.numel():
        q[same] = p[same, :K]
    if onehot.numel():
        hot = torch.randint(0, V, (onehot.numel(), K + 1), generator=gen, device=device)
        scale = p[onehot].amax(dim=-1)                       # keeps the row factor's size
        p[onehot] = 0.0
        rows = p[onehot]
        rows.scatter_(2, hot.unsqueeze(2), scale.unsqueeze(2))
        p[onehot] = rows
    if single.numel():
        # q = p except at x (q < p there: the only residual mass) and at y
        # (q > p there, so that drafting y can be rejected)
        ns = single.numel()
        x = torch.randint(0, V, (ns, K), generator=gen, device=device)
        y = (x + torch.randint(1, max(V, 2), (ns, K), generator=gen, device=device)) % V
        rows = p[single, :K].clone()
        px = rows.gather(2, x.unsqueeze(2))
        py = rows.gather(2, y.unsqueeze(2))
        rows.scatter_(2, x.unsqueeze(2), 0.5 * px)
        rows.scatter_(2, y.unsqueeze(2), py + 0.5 * px + 0.3)
        q[single] = rows
    # draft tokens are drawn from the final draft rows
    t = _sample_rows(q.view(-1, V), gen).view(B, K).to(torch.int32)
    u_acc, u_res = _uniforms(B, K, gen, device)
    mode = torch.ones(B, dtype=torch.uint8, device=device)
    meta = dict(same=same.tolist(), onehot=onehot.tolist(), single=single.tolist())
    return p, q, t, u_acc, u_res, mode, meta


def make_inputs(cfg: int, device="cpu", seed: Optional[int] = None, *, B=None, V=None,
                K=None) -> Batch:
    """Seeded inputs for workload ``cfg`` (1..5) on ``device``; B/V/K override sizes."""
    if cfg not in CONFIGS:
        raise ValueError(f"unknown workload {cfg}")
    c = CONFIGS[cfg]
    B = c["B"] if B is None else int(B)
    V = c["V"] if V is None else int(V)
    K = c["K"] if K is None else int(K)
    seed = SEED_BASE + cfg if seed is None else int(seed)
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    with torch.no_grad():
        if cfg == 1:
            out = _cfg1_or_3(B, V, K, 2.0, 0.82, gen, device)
        elif cfg == 2:
            out = _cfg2(B, V, K, gen, device)
        elif cfg == 3:
            out = _cfg1_or_3(B, V, K, 2.0, 1.0, gen, device)
        elif cfg == 4:
            out = _cfg4(B, V, K, gen, device)
        else:
            out = _cfg5(B, V, K, gen, device)
    p, q, t, u_acc, u_res, mode, meta = out
    meta.update(seed=seed, name=c["name"].split(" ")[0] + f" B={B} V={V} K={K}")
    return Batch(cfg, B, K, V, p.contiguous(), t.contiguous(),
                 None if q is None else q.contiguous(), u_acc.contiguous(),
                 u_res.contiguous(), mode.contiguous(), meta)
