"""Round driver for speculative decoding over user callbacks, and the
speculation governor.

The driver follows the "spec-verify" page, sections "Usage" and "API": the
caller supplies ``draft_step(prefix, k) -> (tokens [k], probs [k][V])`` and
``target_step(prefix, proposed) -> probs [len(proposed) + 1][V]``; each round
the draft proposes k tokens, the target scores the prefix extended by them,
and the verification keeps the accepted proposals and appends the emitted
token.  Verification and the commit into the token buffer run on the GPU
(``sv_verify_round``); only the callbacks and the loop are host code.

``PendingTokenDecoder`` drives a target that keeps a cache of the tokens it
has processed, with the deferred ("pending") correction token of the SPEL
page, section 1.2 (Speculative decoding), and the llms-explorer post's
backend: one target pass per round over [pending, d_0, ..., d_{k-1}], the
rejected drafts rolled back, the emitted token left pending for the next pass.

The governor follows the SPEL page, section 1.3 (Dynamic Speculation
Governor): it keeps the ratio of accepted to proposed tokens over a rolling
window of rounds and stops drafting for the rest of the call once that ratio
falls below a threshold or a round accepts nothing; it never resumes within
the call.  The remaining tokens are then decoded one at a time (K = 0 rounds
of the same verification call: the argmax, or a draw from the target row).
"""
from __future__ import annotations

from collections import deque
from typing import Callable, List, Optional, Sequence, Tuple

from . import SpecVerifyError, _torch, verify_round, Workspace


class SpeculationGovernor:
    """Rolling accepted/proposed ratio over the last ``window`` rounds.

    ``record(accepted, proposed)`` returns whether drafting continues.  It
    stops (for good) when a round with proposals accepts none (if
    ``stop_on_zero_accept``) or when the window is full and its ratio is below
    ``alpha_threshold``."""

    def __init__(self, window: int = 16, alpha_threshold: float = 0.0,
                 stop_on_zero_accept: bool = True):
        if window < 1:
            raise ValueError("window must be >= 1")
        if not 0.0 <= alpha_threshold <= 1.0:
            raise ValueError("alpha_threshold must be in [0, 1]")
        self.window = window
        self.alpha_threshold = alpha_threshold
        self.stop_on_zero_accept = stop_on_zero_accept
        self._rounds: deque = deque(maxlen=window)
        self.speculating = True
        self.reason: Optional[str] = None

    @property
    def rate(self) -> Optional[float]:
        """Accepted / proposed over the window, or None before any proposal."""
        prop = sum(p for _, p in self._rounds)
        return None if prop == 0 else sum(a for a, _ in self._rounds) / prop

    def record(self, accepted: int, proposed: int) -> bool:
        if not self.speculating:
            return False
        if accepted < 0 or proposed < 0 or accepted > proposed:
            raise ValueError("need 0 <= accepted <= proposed")
        self._rounds.append((accepted, proposed))
        if self.stop_on_zero_accept and proposed > 0 and accepted == 0:
            self.speculating, self.reason = False, "zero-accept round"
        elif len(self._rounds) == self.window and self.rate is not None \
                and self.rate < self.alpha_threshold:
            self.speculating, self.reason = False, "acceptance below threshold"
        return self.speculating


class DeviceVerifier:
    """One verification round on the GPU (``sv_verify_round``) with the commit
    into the caller's device token buffer: the step both drivers take each
    round.  Keeps one workspace per (K, V), replaced only by a larger batch:
    a smaller batch reuses it (the library clears per-size state itself when
    the sizes change between calls on one workspace).

    ``__call__(mode, p, q, t, u_acc, u_res, tokens, lengths)`` takes the
    tensors of ``verify_round`` (q is None when K = 0) and returns
    (n_accepted [B], next_token [B]) on the device."""

    def __init__(self, device=None):
        torch = _torch()
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self._ws = {}

    def __call__(self, mode, p, q, t, u_acc, u_res, tokens, lengths):
        B, K, V = p.shape[0], t.shape[1], p.shape[2]
        w = self._ws.get((K, V))
        if w is None or not w.fits(B, K, V):
            w = self._ws[(K, V)] = Workspace(B, K, V, self.device)
        return verify_round(mode, p, q if K > 0 else None, t, u_acc, u_res, tokens=tokens,
                            lengths=lengths, ws=w)


class _RoundDriver:
    """What the drivers share: the draft callback, the rule,
    the uniforms' generator, the governor, the device token buffer and one
    verification round over given rows.

    ``verify`` is the verification step, called as ``DeviceVerifier`` is.  It
    defaults to ``DeviceVerifier`` (the CUDA library); there is no CPU path.
    The tests pass the oracle here to check a driver's own bookkeeping on a
    machine without a GPU."""

    def __init__(self, draft_step: Callable, k: int, greedy: bool, seed: int,
                 governor: Optional[SpeculationGovernor], device, verify: Optional[Callable]):
        if k < 1:
            raise ValueError("k must be >= 1")
        torch = _torch()
        self.draft_step = draft_step
        self.k, self.greedy = k, greedy
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.gen = torch.Generator(device=self.device)
        self.gen.manual_seed(seed)
        self.governor = governor
        self.verify = DeviceVerifier(self.device) if verify is None else verify
        self.trace: List[Tuple[int, int, int]] = []

    def _probs(self, x, rows: int, V: Optional[int], what: str):
        torch = _torch()
        x = torch.as_tensor(x, dtype=torch.float32, device=self.device)
        if x.dim() == 1:
            x = x.unsqueeze(0)
        if x.shape[0] != rows or (V is not None and x.shape[1] != V):
            raise SpecVerifyError(f"{what}: expected [{rows}][V], got {tuple(x.shape)}")
        return x.contiguous()

    def _k(self) -> int:
        """Drafts this round: k while the governor lets the call speculate, else 0."""
        return self.k if self.governor is None or self.governor.speculating else 0

    def _draft(self, prefix: Sequence[int], k: int):
        """(draft tokens [k] as ints, draft probs [k][V] or None)."""
        if k == 0:
            return [], None
        toks, qprobs = self.draft_step(list(prefix), k)
        toks = [int(x) for x in toks]
        if len(toks) != k:
            raise SpecVerifyError(f"draft_step returned {len(toks)} tokens, expected {k}")
        return toks, qprobs

    def _buffers(self, prefix: Sequence[int], max_new: int):
        torch = _torch()
        start = len(prefix)
        cap = start + max_new + self.k + 1
        tokens_buf = torch.zeros(1, cap, dtype=torch.int32, device=self.device)
        tokens_buf[0, :start] = torch.tensor(list(prefix), dtype=torch.int32)
        lengths_buf = torch.tensor([start], dtype=torch.int32, device=self.device)
        return tokens_buf, lengths_buf

    def _verify(self, toks, qprobs, target_rows, tokens_buf, lengths_buf):
        """Verifies the drafts toks against target_rows [k+1][V] (draft probs
        qprobs [k][V]) and appends the kept drafts and the emitted token to
        the token buffer; returns (n_accepted, next_token)."""
        torch = _torch()
        k = len(toks)
        target = self._probs(target_rows, k + 1, None, "target")
        V = target.shape[1]
        if k > 0:
            t = torch.as_tensor(toks, dtype=torch.int32, device=self.device).reshape(1, k)
            q = self._probs(qprobs, k, V, "draft probs").unsqueeze(0)
        else:
            t = torch.zeros(1, 0, dtype=torch.int32, device=self.device)
            q = torch.zeros(1, 0, V, device=self.device)
        mode = torch.tensor([0 if self.greedy else 1], dtype=torch.uint8, device=self.device)
        ua = torch.rand(1, k, generator=self.gen, device=self.device)
        ur = torch.rand(1, generator=self.gen, device=self.device, dtype=torch.float64)
        n, nxt = self.verify(mode, target.unsqueeze(0), q, t, ua, ur, tokens_buf, lengths_buf)
        n, nxt = int(n[0].item()), int(nxt[0].item())
        if nxt < 0:
            raise SpecVerifyError("verification produced no token (invalid draft ids or "
                                  "zero-mass rows)")
        return n, nxt

    @staticmethod
    def _eos_cut(out: List[int], eos_id: Optional[int], max_new: int) -> Optional[List[int]]:
        if eos_id is not None and eos_id in out:
            return out[:out.index(eos_id) + 1][:max_new]
        return None


class SpeculativeDecoder(_RoundDriver):
    """Speculative decoding of one sequence with user callbacks (the page's
    ``SpeculativeDecoder(draft_step, target_step, k=4, greedy=True)``).

    ``generate(prompt_ids, max_new)`` returns the new token ids.  Greedy mode
    emits exactly the stream plain greedy decoding of the target would;
    sampling mode draws its uniforms from a seeded CUDA generator, so a fixed
    seed gives a fixed stream.  ``trace`` records (proposed, n_accepted,
    next_token) per round."""

    def __init__(self, draft_step: Callable, target_step: Callable, k: int = 4,
                 greedy: bool = True, seed: int = 0, governor: Optional[SpeculationGovernor] = None,
                 device=None, verify: Optional[Callable] = None):
        super().__init__(draft_step, k, greedy, seed, governor, device, verify)
        self.target_step = target_step

    def generate(self, prompt_ids: Sequence[int], max_new: int = 128,
                 eos_id: Optional[int] = None) -> List[int]:
        prefix = list(int(x) for x in prompt_ids)
        start = len(prefix)
        tokens_buf, lengths_buf = self._buffers(prefix, max_new)
        self.trace = []
        while len(prefix) - start < max_new:
            k = self._k()
            toks, qprobs = self._draft(prefix, k)
            rows = self.target_step(list(prefix), list(toks))
            n, nxt = self._verify(toks, qprobs, rows, tokens_buf, lengths_buf)
            self.trace.append((k, n, nxt))
            prefix = tokens_buf[0, :int(lengths_buf.item())].tolist()   # the committed history
            if self.governor is not None and k > 0:
                self.governor.record(n, k)
            cut = self._eos_cut(prefix[start:], eos_id, max_new)
            if cut is not None:
                return cut
        return prefix[start:start + max_new]


class PendingTokenDecoder(_RoundDriver):
    """Speculative decoding of one sequence against a target that keeps a
    cache of the tokens it has processed, with a deferred ("pending")
    correction token.

    The token a round emits is not run through the target at once.  The next
    round runs the target once over [pending, d_0, ..., d_{k-1}]: row j of
    that pass is the distribution that follows the prefix, the pending token
    and d_0..d_{j-1}, which are exactly the k + 1 rows verification needs.
    The accepted drafts stay in the cache, the rejected ones are rolled back,
    and the emitted token (correction or bonus) becomes the next pending
    token.  Every round therefore costs one target pass, and no round needs a
    separate pass for the token it emits.  The stream is the one
    ``SpeculativeDecoder`` produces with the same callbacks and seed.

    ``target`` provides
      ``forward(tokens) -> probs [len(tokens)][V]``: appends tokens to its
        cache; row j is the distribution of the token after tokens[j];
      ``rollback(n)``: drops the last n tokens from its cache.
    ``draft_step(prefix, k) -> (tokens [k], probs [k][V])`` as for
    ``SpeculativeDecoder``.  ``target_passes`` counts forward calls (the
    prompt's prefill included) and ``trace`` records (proposed, n_accepted,
    next_token) per round."""

    def __init__(self, draft_step: Callable, target, k: int = 4, greedy: bool = True,
                 seed: int = 0, governor: Optional[SpeculationGovernor] = None, device=None,
                 verify: Optional[Callable] = None):
        super().__init__(draft_step, k, greedy, seed, governor, device, verify)
        self.target = target
        self.target_passes = 0

    def _forward(self, tokens: List[int]):
        self.target_passes += 1
        return self.target.forward(list(tokens))

    def generate(self, prompt_ids: Sequence[int], max_new: int = 128,
                 eos_id: Optional[int] = None) -> List[int]:
        """New token ids after prompt_ids (at least one token).  The target's
        cache must be empty; on return it holds every committed token but
        the last (still pending)."""
        prefix = list(int(x) for x in prompt_ids)
        if not prefix:
            raise ValueError("the prompt needs at least one token")
        start = len(prefix)
        tokens_buf, lengths_buf = self._buffers(prefix, max_new)
        self.trace = []
        self.target_passes = 0
        if len(prefix) > 1:
            self._forward(prefix[:-1])          # prefill; its rows are not needed
        pending = prefix[-1]
        while len(prefix) - start < max_new:
            k = self._k()
            toks, qprobs = self._draft(prefix, k)
            rows = self._forward([pending] + toks)
            n, nxt = self._verify(toks, qprobs, rows, tokens_buf, lengths_buf)
            if k > n:
                self.target.rollback(k - n)     # the rejected drafts leave the cache
            pending = nxt
            self.trace.append((k, n, nxt))
            prefix = tokens_buf[0, :int(lengths_buf.item())].tolist()   # the committed history
            if self.governor is not None and k > 0:
                self.governor.record(n, k)
            cut = self._eos_cut(prefix[start:], eos_id, max_new)
            if cut is not None:
                return cut
        return prefix[start:start + max_new]


class BatchedSpeculativeDecoder(_RoundDriver):
    """Speculative decoding of several sequences at once: one mixed
    verification round per step over every sequence still running (a
    per-sequence rule, greedy or sampling, and the commit into a device token
    buffer of one row per sequence), as the batched kernels are built for.

    ``draft_step(prefixes, k) -> (tokens [B'][k], probs [B'][k][V])`` and
    ``target_step(prefixes, proposed) -> probs [B'][k + 1][V]`` take the
    prefixes of the B' running sequences, in the order ``generate`` was given
    them.  ``greedy`` is one flag for all sequences or one per sequence.  The
    governor, if any, sees the batch's accepted and proposed totals per round
    and, once it trips, every sequence continues with one-token rounds.
    ``verify`` as for ``SpeculativeDecoder`` (default: ``DeviceVerifier``).
    ``trace`` records (proposed, [(sequence, n_accepted, next_token), ...])
    per round."""

    def __init__(self, draft_step: Callable, target_step: Callable, k: int = 4, greedy=True,
                 seed: int = 0, governor: Optional[SpeculationGovernor] = None, device=None,
                 verify: Optional[Callable] = None):
        super().__init__(draft_step, k, greedy, seed, governor, device, verify)
        self.target_step = target_step
        self.trace: List[Tuple[int, List[Tuple[int, int, int]]]] = []

    def _modes(self, B: int) -> List[int]:
        flags = [self.greedy] * B if isinstance(self.greedy, bool) else list(self.greedy)
        if len(flags) != B:
            raise ValueError(f"greedy: expected {B} flags, got {len(flags)}")
        return [0 if g else 1 for g in flags]

    def _tensor(self, x, dtype):
        """Callback output (a tensor, an array or nested lists) on the device."""
        import numpy as np
        torch = _torch()
        if isinstance(x, torch.Tensor):
            return x.to(device=self.device, dtype=dtype)
        if isinstance(x, (list, tuple)):
            x = np.stack([np.asarray(r) for r in x]) if len(x) else np.zeros((0,))
        return torch.as_tensor(np.asarray(x), dtype=dtype, device=self.device)

    def _rows(self, x, shape: Tuple[int, ...], what: str):
        x = self._tensor(x, _torch().float32)
        if tuple(x.shape[:-1]) != shape:
            raise SpecVerifyError(f"{what}: expected {list(shape)} rows of V, got {tuple(x.shape)}")
        return x.contiguous()

    def generate(self, prompts: Sequence[Sequence[int]], max_new: int = 128,
                 eos_id: Optional[int] = None) -> List[List[int]]:
        torch = _torch()
        prefixes = [[int(x) for x in pr] for pr in prompts]
        B = len(prefixes)
        if B == 0:
            return []
        starts = [len(pr) for pr in prefixes]
        modes = self._modes(B)
        cap = max(starts) + max_new + self.k + 1
        tokens_buf = torch.zeros(B, cap, dtype=torch.int32, device=self.device)
        for b, pr in enumerate(prefixes):
            tokens_buf[b, :len(pr)] = torch.tensor(pr, dtype=torch.int32)
        lengths_buf = torch.tensor(starts, dtype=torch.int32, device=self.device)
        live = list(range(B))
        self.trace = []
        while live:
            k = self._k()
            L = len(live)
            pre = [list(prefixes[b]) for b in live]
            if k > 0:
                toks, qprobs = self.draft_step(pre, k)
                t = self._tensor(toks, torch.int32).reshape(L, k).contiguous()
                rows = self.target_step(pre, t.cpu().tolist())
            else:
                t = torch.zeros(L, 0, dtype=torch.int32, device=self.device)
                rows = self.target_step(pre, [[] for _ in live])
            p = self._rows(rows, (L, k + 1), "target")
            V = p.shape[-1]
            q = (self._rows(qprobs, (L, k), "draft probs") if k > 0
                 else torch.zeros(L, 0, V, device=self.device))
            if q.shape[-1] != V:
                raise SpecVerifyError("draft and target rows differ in V")
            mode = torch.tensor([modes[b] for b in live], dtype=torch.uint8, device=self.device)
            ua = torch.rand(L, k, generator=self.gen, device=self.device)
            ur = torch.rand(L, generator=self.gen, device=self.device, dtype=torch.float64)
            idx = torch.tensor(live, dtype=torch.int64, device=self.device)
            whole = L == B
            tok = tokens_buf if whole else tokens_buf.index_select(0, idx)
            lens = lengths_buf if whole else lengths_buf.index_select(0, idx)
            n, nxt = self.verify(mode, p, q, t, ua, ur, tok, lens)
            if not whole:                      # the running rows back into place
                tokens_buf.index_copy_(0, idx, tok)
                lengths_buf.index_copy_(0, idx, lens)
            n, nxt = n.cpu().tolist(), nxt.cpu().tolist()
            if min(nxt) < 0:
                raise SpecVerifyError("verification produced no token (invalid draft ids or "
                                      "zero-mass rows)")
            self.trace.append((k, [(b, int(n[i]), int(nxt[i])) for i, b in enumerate(live)]))
            lengths = lengths_buf.cpu().tolist()
            rows_host = tokens_buf.cpu()
            done = []
            for b in live:
                prefixes[b] = rows_host[b, :lengths[b]].tolist()
                out = prefixes[b][starts[b]:]
                if len(out) >= max_new or (eos_id is not None and eos_id in out):
                    done.append(b)
            if self.governor is not None and k > 0:
                self.governor.record(sum(int(x) for x in n), k * L)
            live = [b for b in live if b not in done]
        results = []
        for b in range(B):
            out = prefixes[b][starts[b]:]
            if eos_id is not None and eos_id in out:
                out = out[:out.index(eos_id) + 1]
            results.append(out[:max_new])
        return results

