"""The pipeline cost model (TileLang tutorial ch.22, section 1.1): its
closed forms, and the worked 6144^3 example the design notes fit to it."""
import math

import pytest

from pipelined_warp_specialized_gb300 import cost_model as cm


def test_closed_forms():
    c, L = 2.0, 6.0
    assert cm.block_time(c, L, 1) == L + c                    # one slot: load, then multiply
    assert cm.block_time(c, L, 2) == (L + c) / 2
    assert cm.saturation_stages(c, L) == 4.0
    for s in (4, 5, 9):                                        # from (L + c)/c slots on, c bounds it
        assert cm.block_time(c, L, s) == c
    assert cm.block_time(c, L, 8, issue=3.0) == 3.0             # an issue bound above both
    assert math.isclose(cm.loop_time(10, c, L, 3), 10 * (L + c) / 3)
    with pytest.raises(ValueError):
        cm.block_time(c, L, 0)


def test_fit_recovers_the_parameters():
    c, L, B = 0.53, 1.09, 384
    t1, tsat = cm.loop_time(B, c, L, 1), cm.loop_time(B, c, L, 6)
    c2, L2 = cm.fit(B, t1, tsat)
    assert math.isclose(c2, c) and math.isclose(L2, L)
    pred = cm.predict_sweep(B, t1, tsat, range(1, 7))
    assert all(math.isclose(pred[s], cm.loop_time(B, c, L, s)) for s in range(1, 7))
    # the time never rises with S, and is flat from saturation on ((L + c)/c
    # = 3.06 slots here: S = 3 is still latency-bound, S = 4 is not)
    assert all(pred[s + 1] <= pred[s] for s in range(1, 6))
    assert pred[3] > pred[4] and math.isclose(pred[4], pred[5]) and math.isclose(pred[5], pred[6])


def test_worked_6144_example():
    # busiest CTA pair: 4 wide units of 96 K blocks; a wide block is 1024
    # cycles of MMA, 0.53 us at the S = 1 run's clock; S = 1 took 622 us
    B, c = 4 * 96, 0.53
    L = 622.0 / B - c
    assert math.isclose(L, 1.09, abs_tol=0.01)
    assert math.isclose(cm.loop_time(B, c, L, 2), 311.0, abs_tol=1.0)
    assert cm.saturation_stages(c, L) == pytest.approx(3.06, abs=0.02)
