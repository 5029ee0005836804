"""Acceptance statistics and the adaptive draft length (host logic, no GPU)."""
import pytest

from speculative_decoding_sampling_gb300.adaptive import (AcceptanceMonitor, AdaptiveK, RoundStats,
                                                          expected_tokens_per_round)


def _stats(accepted, proposed, sequences=1, K=4):
    hist = [0] * (K + 1)
    return RoundStats(sequences, proposed, accepted, accepted + sequences, tuple(hist))


def test_expected_tokens_per_round_printed_values():
    """[NOTE] 好草稿也要算得便宜 prints 3.3616 (alpha .8) and 4.0951 (alpha .9)
    for four drafts; [KB] 参考答案 gives about 2.95 for alpha .8 and three."""
    assert round(expected_tokens_per_round(0.8, 4), 4) == 3.3616
    assert round(expected_tokens_per_round(0.9, 4), 4) == 4.0951
    assert round(expected_tokens_per_round(0.8, 3), 2) == 2.95
    assert expected_tokens_per_round(1.0, 5) == 6.0       # every draft accepted
    assert expected_tokens_per_round(0.0, 5) == 1.0       # only the final token
    assert expected_tokens_per_round(0.3, 0) == 1.0       # no drafts


def test_adjust_rule_thresholds_and_bounds():
    """[REPORT] part 1 §2 _adjust_K: strictly above 0.85 one more draft (at
    most max_K), strictly below 0.60 one fewer (at least 1)."""
    ak = AdaptiveK(initial_K=4, max_K=5, window=1)
    assert ak.update(_stats(85, 100)) == 4      # exactly 0.85: unchanged
    assert ak.update(_stats(86, 100)) == 5      # above: +1
    assert ak.update(_stats(99, 100)) == 5      # capped at max_K
    assert ak.update(_stats(60, 100)) == 5      # exactly 0.60: unchanged
    assert ak.update(_stats(59, 100)) == 4      # below: -1
    for _ in range(10):
        ak.update(_stats(0, 100))
    assert ak.current_K == 1                    # floor at 1


def test_monitor_window_is_accepted_over_proposed_of_recent_calls():
    m = AcceptanceMonitor(window=3)
    assert m.update(10, 10) == 1.0
    assert m.update(0, 30) == pytest.approx(10 / 40)
    assert m.update(5, 10) == pytest.approx(15 / 50)
    assert m.update(5, 10) == pytest.approx(10 / 50)   # the first call left the window
    assert AcceptanceMonitor(2).rate == 0.0


def test_round_stats_from_counters():
    # 3 sequences, K = 2: accepted 0, 2 and 1 drafts
    s = RoundStats.from_counters([3, 6, 3, 6, 1, 1, 1])
    assert (s.sequences, s.proposed, s.accepted, s.emitted) == (3, 6, 3, 6)
    assert s.K == 2 and s.accepted_hist == (1, 1, 1)
    assert s.acceptance_rate == 0.5 and s.tokens_per_round == 2.0
    with pytest.raises(ValueError):
        RoundStats.from_counters([1, 2, 3])


def test_bad_arguments():
    with pytest.raises(ValueError):
        AdaptiveK(initial_K=0, max_K=4)
    with pytest.raises(ValueError):
        AcceptanceMonitor(0)
    with pytest.raises(ValueError):
        expected_tokens_per_round(1.5, 3)
