"""Acceptance statistics and the adaptive draft length (host side).

spec_verify_stats has the verdict of every sequence add the call's
acceptance counters on the device: sequences, drafts proposed, drafts
accepted, tokens emitted, and how many sequences accepted exactly n drafts
(the per-round figures "推测解码：草稿、验证与实际加速" asks a deployment to
record, section 在相同负载和质量下比较).  RoundStats reads them back.

AcceptanceMonitor keeps the acceptance rate over a window of recent calls,
and AdaptiveK turns it into the next call's draft length with the rule of
the engine in "推测解码采样验证优化策略 —— 深度调研报告" (part 1 §2, the
monitor step and _adjust_K): one draft more when the rate is above 0.85 (at
most max_K), one fewer when it is below 0.60 (at least 1), otherwise
unchanged.  The pages leave the window open; here it is the last `window`
calls, and the rate is their accepted drafts over their proposed drafts.

expected_tokens_per_round is the closed form those pages give for the
tokens one round yields under i.i.d. acceptance with probability a:
E[N] = (1 - a^(K+1)) / (1 - a) ("推测解码：草稿、验证与实际加速", section
好草稿也要算得便宜; "投机采样", section 收益账).
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass

from ._native import stats_words


@dataclass(frozen=True)
class RoundStats:
    """The counters of spec_verify_stats (one call, or a sum of calls)."""
    sequences: int
    proposed: int
    accepted: int
    emitted: int
    accepted_hist: tuple  # sequences that accepted exactly n drafts, n = 0..K

    @staticmethod
    def from_counters(counters) -> "RoundStats":
        """From the SV_STATS_WORDS(K) counters (a tensor or a sequence of ints)."""
        c = [int(v) for v in (counters.tolist() if hasattr(counters, "tolist") else counters)]
        if len(c) < 5:
            raise ValueError("expected SV_STATS_WORDS(K) >= 5 counters")
        return RoundStats(c[0], c[1], c[2], c[3], tuple(c[4:]))

    @property
    def K(self) -> int:
        return len(self.accepted_hist) - 1

    @property
    def acceptance_rate(self) -> float:
        """Accepted drafts over proposed drafts (0 when none was proposed)."""
        return self.accepted / self.proposed if self.proposed else 0.0

    @property
    def tokens_per_round(self) -> float:
        """Tokens emitted per verified sequence (accepted drafts + 1)."""
        return self.emitted / self.sequences if self.sequences else 0.0


def stats_buffer(K: int, device="cuda"):
    """A zeroed int64 device tensor of SV_STATS_WORDS(K) counters."""
    import torch
    return torch.zeros(stats_words(K), dtype=torch.int64, device=device)


class AcceptanceMonitor:
    """The acceptance rate over the last `window` calls."""

    def __init__(self, window: int):
        if window < 1:
            raise ValueError("window must be >= 1")
        self._calls = deque(maxlen=window)

    def update(self, accepted: int, proposed: int) -> float:
        self._calls.append((int(accepted), int(proposed)))
        return self.rate

    @property
    def rate(self) -> float:
        acc = sum(a for a, _ in self._calls)
        prop = sum(p for _, p in self._calls)
        return acc / prop if prop else 0.0


class AdaptiveK:
    """The draft length for the next call, from the windowed acceptance rate."""

    def __init__(self, initial_K: int, max_K: int, window: int = 16,
                 raise_above: float = 0.85, lower_below: float = 0.60):
        if not 1 <= initial_K <= max_K:
            raise ValueError("need 1 <= initial_K <= max_K")
        self.max_K = max_K
        self.current_K = initial_K
        self.raise_above = raise_above
        self.lower_below = lower_below
        self.monitor = AcceptanceMonitor(window)

    def update(self, stats: RoundStats) -> int:
        """Record one call's counters and return the next call's K."""
        rate = self.monitor.update(stats.accepted, stats.proposed)
        if rate > self.raise_above:
            self.current_K = min(self.max_K, self.current_K + 1)
        elif rate < self.lower_below:
            self.current_K = max(1, self.current_K - 1)
        return self.current_K


def expected_tokens_per_round(alpha: float, K: int) -> float:
    """E[N] = (1 - alpha^(K+1)) / (1 - alpha), i.e. K + 1 at alpha = 1."""
    if K < 0 or not 0.0 <= alpha <= 1.0:
        raise ValueError("need K >= 0 and 0 <= alpha <= 1")
    if alpha == 1.0:
        return float(K + 1)
    return (1.0 - alpha ** (K + 1)) / (1.0 - alpha)
