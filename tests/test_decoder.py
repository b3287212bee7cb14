"""The round drivers and the speculation governor.

The governor is host logic (CPU tests).  The drivers run their verification
on the GPU: greedy decoding through them must give exactly the stream plain
greedy decoding of the target gives ("spec-verify", section "Method"), with
or without the governor switching to one-token rounds; sampled rounds must
agree with the oracle on the same rows and uniforms.  The drivers' own
bookkeeping (drafts, the pending token, rollbacks, the commit, target passes)
is also checked on the CPU, with the oracle standing in for the verification
step through the drivers' ``verify`` hook."""
import hashlib

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_08_gb300 as sv
from speculative_decoding_verification_08_gb300.decoder import (BatchedSpeculativeDecoder,
                                                                 PendingTokenDecoder,
                                                                 SpeculationGovernor,
                                                                 SpeculativeDecoder)

V = 48


def _logits(prefix, salt):
    h = hashlib.sha256((salt + ",".join(map(str, prefix[-4:]))).encode()).digest()
    rng = np.random.default_rng(int.from_bytes(h[:8], "little"))
    z = rng.normal(0, 2.0, V)
    z[rng.integers(0, V)] = z.max()          # frequent exact ties: lowest index must win
    return z


def _softmax(z):
    e = np.exp(z - z.max())
    return (e / e.sum()).astype(np.float32)


def target_row(prefix):
    return _softmax(_logits(prefix, "target"))


def draft_row(prefix, noise):
    z = _logits(prefix, "target") + noise * _logits(prefix, "draft")
    return _softmax(z)


def make_callbacks(noise=0.6, greedy_draft=True, seed=0):
    rng = np.random.default_rng(seed)

    def draft_step(prefix, k):
        toks, probs = [], []
        p = list(prefix)
        for _ in range(k):
            q = draft_row(p, noise)
            x = int(np.argmax(q)) if greedy_draft else int(rng.choice(V, p=q / q.sum()))
            toks.append(x)
            probs.append(q)
            p.append(x)
        return toks, np.stack(probs)

    def target_step(prefix, proposed):
        p = list(prefix)
        rows = [target_row(p)]
        for x in proposed:
            p.append(int(x))
            rows.append(target_row(p))
        return np.stack(rows)

    return draft_step, target_step


def plain_greedy(prompt, max_new):
    p = list(prompt)
    for _ in range(max_new):
        p.append(int(oracle.argmax_lowest(target_row(p))))
    return p[len(prompt):]


# ---------------------------------------------------------------------------
# governor (CPU)

def test_governor_trips_on_zero_accept_and_never_resumes():
    g = SpeculationGovernor(window=4, alpha_threshold=0.0)
    assert g.record(3, 4) and g.record(1, 4)
    assert not g.record(0, 4) and g.reason == "zero-accept round"
    assert not g.record(4, 4) and not g.speculating


def test_governor_threshold_over_a_full_window():
    g = SpeculationGovernor(window=3, alpha_threshold=0.5, stop_on_zero_accept=False)
    assert g.record(1, 4) and g.record(1, 4)          # window not yet full
    assert not g.record(2, 4)                          # 4/12 < 0.5 once full
    assert g.reason == "acceptance below threshold"
    g2 = SpeculationGovernor(window=2, alpha_threshold=0.5)
    for _ in range(10):
        assert g2.record(3, 4)                         # rolling 0.75 stays above
    assert g2.rate == 0.75


def test_governor_rejects_bad_counts():
    g = SpeculationGovernor()
    with pytest.raises(ValueError):
        g.record(5, 4)
    with pytest.raises(ValueError):
        SpeculationGovernor(window=0)


# ---------------------------------------------------------------------------
# driver (GPU)

@pytest.mark.gpu
@pytest.mark.parametrize("k", [1, 3, 4, 7])
def test_greedy_driver_equals_plain_greedy(k):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    draft_step, target_step = make_callbacks(noise=0.6)
    dec = SpeculativeDecoder(draft_step, target_step, k=k, greedy=True)
    prompt = [1, 2, 3]
    out = dec.generate(prompt, max_new=60)
    assert out == plain_greedy(prompt, 60)
    assert any(n > 0 for _, n, _ in dec.trace) and any(n < k for _, n, _ in dec.trace)


@pytest.mark.gpu
def test_governor_switches_to_single_token_rounds():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    draft_step, target_step = make_callbacks(noise=8.0)     # a poor draft: zero-accept rounds
    gov = SpeculationGovernor(window=4, alpha_threshold=0.4)
    dec = SpeculativeDecoder(draft_step, target_step, k=4, greedy=True, governor=gov)
    out = dec.generate([5, 6], max_new=40)
    assert out == plain_greedy([5, 6], 40)
    assert not gov.speculating
    ks = [k for k, _, _ in dec.trace]
    first_ar = ks.index(0)
    assert all(k == 0 for k in ks[first_ar:]) and all(k == 4 for k in ks[:first_ar])


@pytest.mark.gpu
def test_sampling_rounds_match_the_oracle():
    """Each sampled round equals the oracle's verification of the same rows
    with the same uniforms (the decoder's generator is replayed here)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    k = 4
    draft_step, target_step = make_callbacks(noise=0.8, greedy_draft=False, seed=5)
    dec = SpeculativeDecoder(draft_step, target_step, k=k, greedy=False, seed=123)
    prompt = [9, 9]
    out = dec.generate(prompt, max_new=50)
    assert len(out) == 50
    # replay: same callbacks (fresh rng with the same seed), same generator
    draft_step, target_step = make_callbacks(noise=0.8, greedy_draft=False, seed=5)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(123)
    prefix = list(prompt)
    for kk, n, nxt in dec.trace:
        toks, q = draft_step(prefix, kk)
        p = target_step(prefix, toks)
        ua = torch.rand(1, kk, generator=gen, device="cuda").cpu().numpy()
        ur = torch.rand(1, generator=gen, device="cuda", dtype=torch.float64).cpu().numpy()
        n0, x0, _ = oracle.verify_sample(p[None], q[None], np.array([toks], dtype=np.int32), ua, ur)
        assert (int(n0[0]), int(x0[0])) == (n, nxt)
        prefix = prefix + list(toks[:n]) + [nxt]
    assert prefix[len(prompt):len(prompt) + 50] == out


# ---------------------------------------------------------------------------
# the pending-token driver, and the drivers' bookkeeping on the CPU

class CachedToyTarget:
    """The toy target with a cache of processed tokens: forward(tokens)
    appends them and returns one row per token (the distribution of the token
    after it); rollback(n) drops the last n."""

    def __init__(self):
        self.cache = []
        self.passes = 0

    def forward(self, tokens):
        self.passes += 1
        rows = []
        for x in tokens:
            self.cache.append(int(x))
            rows.append(target_row(self.cache))
        return np.stack(rows)

    def rollback(self, n):
        assert 0 < n <= len(self.cache)
        del self.cache[-n:]


def oracle_verify(mode, p, q, t, ua, ur, tokens, lengths):
    """The verification step with the commit, computed by the oracle on CPU
    tensors (test stand-in for the drivers' device verifier)."""
    n, x, _ = oracle.verify_round(mode.numpy(), p.numpy(), q.numpy(), t.numpy(), ua.numpy(),
                                  ur.numpy())
    assert oracle.commit(t.numpy(), n, x, tokens.numpy(), lengths.numpy()) == 0
    return torch.from_numpy(n), torch.from_numpy(x)


def committed_length(prompt, trace):
    return len(prompt) + sum(n + 1 for _, n, _ in trace)


@pytest.mark.parametrize("k", [1, 3, 4, 7])
def test_pending_driver_greedy_on_cpu(k):
    draft_step, _ = make_callbacks(noise=0.6)
    target = CachedToyTarget()
    dec = PendingTokenDecoder(draft_step, target, k=k, greedy=True, device="cpu",
                              verify=oracle_verify)
    prompt = [1, 2, 3]
    out = dec.generate(prompt, max_new=60)
    assert out == plain_greedy(prompt, 60)
    # one target pass per round, plus the prompt's prefill
    assert target.passes == dec.target_passes == len(dec.trace) + 1
    # the cache holds every committed token but the pending one
    total = committed_length(prompt, dec.trace)
    assert target.cache == (prompt + plain_greedy(prompt, total))[:total - 1]
    assert any(n > 0 for _, n, _ in dec.trace) and any(n < k for _, n, _ in dec.trace)


def test_uncached_driver_greedy_on_cpu():
    draft_step, target_step = make_callbacks(noise=0.6)
    dec = SpeculativeDecoder(draft_step, target_step, k=4, greedy=True, device="cpu",
                             verify=oracle_verify)
    assert dec.generate([4, 4], max_new=40) == plain_greedy([4, 4], 40)


def test_pending_and_uncached_drivers_sample_the_same_stream():
    """Same callbacks and seed: the cached target's rows equal the recomputed
    ones, so both drivers make the same draws."""
    k, prompt = 4, [7, 1, 8]
    draft_a, target_step = make_callbacks(noise=0.8, greedy_draft=False, seed=11)
    plain = SpeculativeDecoder(draft_a, target_step, k=k, greedy=False, seed=5, device="cpu",
                               verify=oracle_verify)
    out_a = plain.generate(prompt, max_new=50)
    draft_b, _ = make_callbacks(noise=0.8, greedy_draft=False, seed=11)
    target = CachedToyTarget()
    pend = PendingTokenDecoder(draft_b, target, k=k, greedy=False, seed=5, device="cpu",
                               verify=oracle_verify)
    out_b = pend.generate(prompt, max_new=50)
    assert out_a == out_b and plain.trace == pend.trace
    assert len(out_b) == 50 and target.passes == len(pend.trace) + 1
    assert any(n < k for _, n, _ in pend.trace)


def test_pending_driver_governor_and_one_token_prompt_on_cpu():
    draft_step, _ = make_callbacks(noise=8.0)           # a poor draft: zero-accept rounds
    gov = SpeculationGovernor(window=4, alpha_threshold=0.4)
    target = CachedToyTarget()
    dec = PendingTokenDecoder(draft_step, target, k=4, greedy=True, governor=gov, device="cpu",
                              verify=oracle_verify)
    out = dec.generate([5], max_new=30)
    assert out == plain_greedy([5], 30)
    assert not gov.speculating
    ks = [k for k, _, _ in dec.trace]
    assert 0 in ks and all(k == 0 for k in ks[ks.index(0):])
    assert target.passes == len(dec.trace)               # a one-token prompt needs no prefill
    total = committed_length([5], dec.trace)
    assert target.cache == ([5] + plain_greedy([5], total))[:total - 1]
    with pytest.raises(ValueError):
        dec.generate([], max_new=3)


@pytest.mark.gpu
def test_pending_driver_on_the_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    draft_step, _ = make_callbacks(noise=0.6)
    target = CachedToyTarget()
    dec = PendingTokenDecoder(draft_step, target, k=4, greedy=True)
    out = dec.generate([1, 2, 3], max_new=60)
    assert out == plain_greedy([1, 2, 3], 60)
    assert target.passes == len(dec.trace) + 1


# ---------------------------------------------------------------------------
# the batched driver (bookkeeping on the CPU, the oracle in the verify hook)

def batched_callbacks(noise=0.6, greedy_draft=True, seed=0):
    draft_one, target_one = make_callbacks(noise, greedy_draft, seed)

    def draft_step(prefixes, k):
        out = [draft_one(pr, k) for pr in prefixes]
        return [t for t, _ in out], np.stack([q for _, q in out])

    def target_step(prefixes, proposed):
        return np.stack([target_one(pr, pp) for pr, pp in zip(prefixes, proposed)])

    return draft_step, target_step


PROMPTS = [[1, 2, 3], [7], [4, 4, 4, 4, 4], [9, 8], [3, 1, 4, 1, 5, 9]]


def test_batched_driver_greedy_on_cpu():
    draft_step, target_step = batched_callbacks(noise=0.6)
    dec = BatchedSpeculativeDecoder(draft_step, target_step, k=4, greedy=True, device="cpu",
                                    verify=oracle_verify)
    outs = dec.generate(PROMPTS, max_new=40)
    assert outs == [plain_greedy(pr, 40) for pr in PROMPTS]
    ns = [n for _, rnd in dec.trace for _, n, _ in rnd]
    assert 0 < max(ns) and min(ns) < 4


def test_batched_driver_mixed_modes_and_eos_on_cpu():
    """Greedy sequences still decode exactly; an end token retires a sequence
    early, so later rounds verify a subset of the batch."""
    plains = [plain_greedy(pr, 40) for pr in PROMPTS]
    eos = plains[0][6]
    flags = [True, False, True, False, True]
    draft_step, target_step = batched_callbacks(noise=0.7, greedy_draft=False, seed=3)
    dec = BatchedSpeculativeDecoder(draft_step, target_step, k=3, greedy=flags, seed=9,
                                    device="cpu", verify=oracle_verify)
    outs = dec.generate(PROMPTS, max_new=40, eos_id=eos)
    for b, (out, plain) in enumerate(zip(outs, plains)):
        if eos in out:
            assert out.index(eos) == len(out) - 1
        else:
            assert len(out) == 40
        if flags[b]:
            want = plain[:plain.index(eos) + 1] if eos in plain else plain
            assert out == want, b
    sizes = [len(rnd) for _, rnd in dec.trace]
    assert sizes[0] == len(PROMPTS) and min(sizes) < len(PROMPTS)   # a subset ran


def test_batched_driver_governor_and_single_sequence_sampling_on_cpu():
    draft_step, target_step = batched_callbacks(noise=8.0)           # zero-accept rounds
    gov = SpeculationGovernor(window=2, alpha_threshold=0.4)
    dec = BatchedSpeculativeDecoder(draft_step, target_step, k=4, greedy=True, governor=gov,
                                    device="cpu", verify=oracle_verify)
    outs = dec.generate(PROMPTS[:3], max_new=25)
    assert outs == [plain_greedy(pr, 25) for pr in PROMPTS[:3]]
    ks = [k for k, _ in dec.trace]
    assert not gov.speculating and 0 in ks and all(k == 0 for k in ks[ks.index(0):])
    # one sequence: the same uniforms as the single-sequence driver, the same stream
    one_d, one_t = make_callbacks(noise=0.8, greedy_draft=False, seed=21)
    single = SpeculativeDecoder(one_d, one_t, k=4, greedy=False, seed=77, device="cpu",
                                verify=oracle_verify)
    want = single.generate([2, 7, 1], max_new=30)
    draft_step, target_step = batched_callbacks(noise=0.8, greedy_draft=False, seed=21)
    dec = BatchedSpeculativeDecoder(draft_step, target_step, k=4, greedy=False, seed=77,
                                    device="cpu", verify=oracle_verify)
    assert dec.generate([[2, 7, 1]], max_new=30) == [want]
    with pytest.raises(ValueError):
        BatchedSpeculativeDecoder(draft_step, target_step, greedy=[True], device="cpu",
                                  verify=oracle_verify).generate(PROMPTS[:2], max_new=3)


def test_device_verifier_reuses_a_workspace_per_k_and_v(monkeypatch):
    """One workspace per (K, V), replaced only when a larger batch comes (the
    library clears per-size state itself); the CUDA calls are stubbed here."""
    import speculative_decoding_verification_08_gb300.decoder as dm

    made, used = [], []

    class FakeWorkspace:
        def __init__(self, B, K, V, device=None):
            self.B, self.K, self.V = B, K, V
            made.append((B, K, V))

        def fits(self, B, K, V):
            return K == self.K and V == self.V and B <= self.B

    def fake_round(mode, p, q, t, ua, ur, tokens=None, lengths=None, ws=None):
        used.append(ws)
        return None, None

    monkeypatch.setattr(dm, "Workspace", FakeWorkspace)
    monkeypatch.setattr(dm, "verify_round", fake_round)
    ver = dm.DeviceVerifier("cpu")

    def call(B, K, V):
        p = torch.zeros(B, K + 1, V)
        ver(None, p, torch.zeros(B, K, V), torch.zeros(B, K, dtype=torch.int32), None, None,
            None, None)

    call(5, 4, 10)
    call(3, 4, 10)          # smaller batch: the same workspace
    call(5, 4, 10)
    call(6, 4, 10)          # larger: a new one
    call(2, 0, 10)          # another K: its own
    call(4, 4, 10)
    assert made == [(5, 4, 10), (6, 4, 10), (2, 0, 10)]
    assert used[0] is used[1] is used[2] and used[3] is used[5] and used[3] is not used[0]


def _batched_callbacks(noise, seed=0):
    """Batched draft/target callbacks over the toy target: every running
    sequence draws its drafts from its own draft row (any draft is valid
    for both rules; the rule is the verifier's)."""
    rng = np.random.default_rng(seed)

    def draft_step(prefixes, k):
        toks, probs = [], []
        for pre in prefixes:
            p = list(pre)
            tt, pp = [], []
            for _ in range(k):
                q = draft_row(p, noise)
                x = int(rng.choice(V, p=q / q.sum()))
                tt.append(x)
                pp.append(q)
                p.append(x)
            toks.append(tt)
            probs.append(np.stack(pp))
        return toks, np.stack(probs)

    def target_step(prefixes, proposed):
        out = []
        for pre, prop in zip(prefixes, proposed):
            p = list(pre)
            rows = [target_row(p)]
            for x in prop:
                p.append(int(x))
                rows.append(target_row(p))
            out.append(np.stack(rows))
        return np.stack(out)

    return draft_step, target_step


@pytest.mark.gpu
def test_batched_driver_on_the_gpu_matches_the_oracle_every_round():
    """64 sequences, half greedy and half sampling, through the device round
    (sv_verify_round with the commit) until each has 30 new tokens: every
    round's (n_accepted, next_token) equals the oracle's on the same rows and
    uniforms, and every greedy sequence is exactly plain greedy decoding."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from oracle.compare import compare
    from speculative_decoding_verification_08_gb300.decoder import DeviceVerifier
    B = 64
    flags = [b % 2 == 0 for b in range(B)]
    prompts = [[1 + b % 7, 2 + b % 5, b % 11] for b in range(B)]
    draft_step, target_step = _batched_callbacks(0.3)
    device_verify = DeviceVerifier()
    rounds = []

    def checked_verify(mode, p, q, t, ua, ur, tokens, lengths):
        host = [x.cpu().numpy() for x in (mode, p, q, t, ua, ur)]
        n, x = device_verify(mode, p, q, t, ua, ur, tokens, lengths)
        n0, x0, s0 = oracle.verify_round(*host)
        assert s0 == 0
        compare(host[1], host[2], host[5], host[0], host[3].shape[1], n0, x0, n.cpu().numpy(),
                x.cpu().numpy(), label="batched driver round")
        rounds.append(int(mode.shape[0]))
        return n, x

    dec = BatchedSpeculativeDecoder(draft_step, target_step, k=4, greedy=flags, seed=5,
                                    verify=checked_verify)
    outs = dec.generate(prompts, max_new=30)
    assert len(rounds) >= 8 and rounds[0] == B
    for b in range(B):
        assert len(outs[b]) == 30
        if flags[b]:
            assert outs[b] == plain_greedy(prompts[b], 30), b
    # sampled rounds accepted some drafts and rejected some
    ns = [n for _, per in dec.trace for _, n, _ in per]
    assert 0 in ns and 4 in ns
