"""Oracle of the adaptive draft-length controller.

TEST INFRASTRUCTURE ONLY (see the package docstring). Plain Python, one object
per sequence, restating the sliding-window controller of "Speculative
decoding principles and a vLLM production setup", sec. 4.3:

  * a step's acceptance rate is alpha = accepted / max(drafted, 1);
  * the rates of the last `window` steps are kept (the oldest falls out);
  * until `min_samples` rates are held nothing changes;
  * then the mean of the held rates moves K: one up (capped at k_max) when it
    is above the upper threshold, one down (floored at k_min) when it is below
    the lower one; the page's thresholds are target +- 0.1;
  * K starts at k_min on the page (k_init here, a parameter).

The same rule with a 10-step window and thresholds 0.8 / 0.5 is the tuning
advice of "LLM inference optimisation: speculative decoding and dynamic
batching" (engineering parameters); `engineering_params` states the reading
used for it (bounds 2..8, start at 4: the page gives 4-8 as the starting
range and no bounds).

Pinned by tests/test_oracle_adaptive_k.py against hand-derived step counts.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass


@dataclass(frozen=True)
class Params:
    k_min: int = 2
    k_max: int = 8
    k_init: int = 2
    window: int = 50
    min_samples: int = 10
    up_threshold: float = 0.6 + 0.1
    down_threshold: float = 0.6 - 0.1


def vllm_params(k_min=2, k_max=8, window=50, target_alpha=0.6) -> Params:
    """The sec. 4.3 controller's defaults: start at k_min, at least 10 samples."""
    return Params(k_min=k_min, k_max=k_max, k_init=k_min, window=window, min_samples=10,
                  up_threshold=target_alpha + 0.1, down_threshold=target_alpha - 0.1)


def engineering_params() -> Params:
    return Params(k_min=2, k_max=8, k_init=4, window=10, min_samples=10, up_threshold=0.8, down_threshold=0.5)


class SequenceController:
    """K of one sequence."""

    def __init__(self, p: Params):
        self.p = p
        self.k = p.k_init
        self.rates = deque(maxlen=p.window)

    def observe(self, accepted: int, drafted: int) -> int:
        if not (0 <= accepted <= drafted):
            raise ValueError("need 0 <= accepted <= drafted")
        self.rates.append(accepted / max(drafted, 1))
        if len(self.rates) >= self.p.min_samples:
            mean = 0.0
            for r in self.rates:  # oldest first
                mean += r
            mean /= len(self.rates)
            if mean > self.p.up_threshold:
                self.k = min(self.k + 1, self.p.k_max)
            elif mean < self.p.down_threshold:
                self.k = max(self.k - 1, self.p.k_min)
        return self.k


class BatchController:
    """One SequenceController per sequence slot."""

    def __init__(self, batch: int, p: Params):
        self.p = p
        self.seqs = [SequenceController(p) for _ in range(batch)]

    def update(self, accepted, drafted) -> list[int]:
        if any(not (0 <= int(a) <= int(d)) for a, d in zip(accepted, drafted)):
            raise ValueError("need 0 <= accepted <= drafted")
        return [s.observe(int(a), int(d)) for s, a, d in zip(self.seqs, accepted, drafted)]

    def reset(self, b: int) -> None:
        self.seqs[b] = SequenceController(self.p)

    @property
    def k(self) -> list[int]:
        return [s.k for s in self.seqs]
