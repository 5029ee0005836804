"""The filter comparison rule (CPU): the oracle's own rows pass, a row with
one id too many or too few outside the window fails."""
import numpy as np

from oracle import parity

import filter_rows


def test_rule_accepts_oracle_and_rejects_mistakes(orc):
    z = filter_rows.rows(3, 8, 500, "fp32")
    ref = orc.filter_logits(z, 1.0, 0, 0.9)
    assert parity.compare_filter(orc, z, 1.0, 0, 0.9, ref.logits, ref.kept).ok()
    for r in (0, 1):
        order = orc.filter_order(z, r, 1.0, 0, 0.9)
        n = int(ref.kept[r])
        bad = ref.logits.copy()
        bad_kept = ref.kept.copy()
        if n > 1:                          # drop the crossing id
            bad[r, order.ids[n - 1]] = -np.inf
            bad_kept[r] = n - 1
        else:                              # keep one id more
            bad[r, order.ids[n]] = z[r, order.ids[n]]
            bad_kept[r] = n + 1
        rep = parity.compare_filter(orc, z, 1.0, 0, 0.9, bad, bad_kept)
        assert not rep.ok() and rep.failures[0][0] == r
