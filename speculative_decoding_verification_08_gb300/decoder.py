"""Round driver for speculative decoding over user callbacks, and the
speculation governor.

The driver follows the "spec-verify" page, sections "Usage" and "API": the
caller supplies ``draft_step(prefix, k) -> (tokens [k], probs [k][V])`` and
``target_step(prefix, proposed) -> probs [len(proposed) + 1][V]``; each round
the draft proposes k tokens, the target scores the prefix extended by them,
and the verification keeps the accepted proposals and appends the emitted
token.  Verification and the commit into the token buffer run on the GPU
(``sv_verify_round``); only the callbacks and the loop are host code.

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


class SpeculativeDecoder:
    """Speculative decoding of one sequence with user callbacks (the page's
    ``SpeculativeDecoder(draft_step, target_step, k=4, greedy=True)``).

    ``generate(prompt_ids, max_new)`` returns the new token ids.  Greedy mode
    emits exactly the stream plain greedy decoding of the target would;
    sampling mode draws its uniforms from a seeded CUDA generator, so a fixed
    seed gives a fixed stream.  ``trace`` records (proposed, n_accepted,
    next_token) per round."""

    def __init__(self, draft_step: Callable, target_step: Callable, k: int = 4,
                 greedy: bool = True, seed: int = 0, governor: Optional[SpeculationGovernor] = None,
                 device=None):
        if k < 1:
            raise ValueError("k must be >= 1")
        torch = _torch()
        self.draft_step, self.target_step = draft_step, target_step
        self.k, self.greedy = k, greedy
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.gen = torch.Generator(device=self.device)
        self.gen.manual_seed(seed)
        self.governor = governor
        self.trace: List[Tuple[int, int, int]] = []

    def _probs(self, x, rows: int, V: Optional[int], what: str):
        torch = _torch()
        x = torch.as_tensor(x, dtype=torch.float32, device=self.device)
        if x.dim() == 1:
            x = x.unsqueeze(0)
        if x.shape[0] != rows or (V is not None and x.shape[1] != V):
            raise SpecVerifyError(f"{what}: expected [{rows}][V], got {tuple(x.shape)}")
        return x.contiguous()

    def _round(self, prefix: Sequence[int], tokens_buf, lengths_buf, ws_cache: dict):
        """One verification round appended to tokens_buf; returns (proposed, n, next)."""
        torch = _torch()
        spec = self.governor is None or self.governor.speculating
        k = self.k if spec else 0
        if k > 0:
            toks, qprobs = self.draft_step(list(prefix), k)
            t = torch.as_tensor(list(toks), dtype=torch.int32, device=self.device).reshape(1, k)
            target = self._probs(self.target_step(list(prefix), list(toks)), k + 1, None, "target")
            q = self._probs(qprobs, k, target.shape[1], "draft probs").unsqueeze(0)
        else:
            t = torch.zeros(1, 0, dtype=torch.int32, device=self.device)
            target = self._probs(self.target_step(list(prefix), []), 1, None, "target")
            q = None
        V = target.shape[1]
        mode = torch.tensor([0 if self.greedy else 1], dtype=torch.uint8, device=self.device)
        ua = torch.rand(1, k, generator=self.gen, device=self.device)
        ur = torch.rand(1, generator=self.gen, device=self.device, dtype=torch.float64)
        if q is None:
            q = torch.zeros(1, 0, V, device=self.device)
        key = (k, V)
        if key not in ws_cache:
            ws_cache[key] = Workspace(1, k, V, self.device)
        n, nxt = verify_round(mode, target.unsqueeze(0), q if k > 0 else None, t, ua, ur,
                              tokens=tokens_buf, lengths=lengths_buf, ws=ws_cache[key])
        n, nxt = int(n.item()), int(nxt.item())
        if nxt < 0:
            raise SpecVerifyError("verification produced no token (invalid draft ids or "
                                  "zero-mass rows)")
        return k, n, nxt

    def generate(self, prompt_ids: Sequence[int], max_new: int = 128,
                 eos_id: Optional[int] = None) -> List[int]:
        torch = _torch()
        prefix = list(int(x) for x in prompt_ids)
        start = len(prefix)
        cap = start + max_new + self.k + 1
        tokens_buf = torch.zeros(1, cap, dtype=torch.int32, device=self.device)
        tokens_buf[0, :start] = torch.tensor(prefix, dtype=torch.int32)
        lengths_buf = torch.tensor([start], dtype=torch.int32, device=self.device)
        ws_cache: dict = {}
        self.trace = []
        while len(prefix) - start < max_new:
            k, n, nxt = self._round(prefix, tokens_buf, lengths_buf, ws_cache)
            self.trace.append((k, n, nxt))
            length = int(lengths_buf.item())
            prefix = tokens_buf[0, :length].tolist()     # the committed history
            if self.governor is not None and k > 0:
                self.governor.record(n, k)
            if eos_id is not None and eos_id in prefix[start:]:
                out = prefix[start:]
                return out[:out.index(eos_id) + 1][:max_new]
        return prefix[start:start + max_new]
