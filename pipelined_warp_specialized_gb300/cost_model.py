"""The pipeline cost model the TileLang tutorial ch.22 restates in section 1.1
(from its ch.11): the steady-state cost of one iteration of a multi-buffered
K loop.  Here it predicts the S sweep.

With S slots, each K block costs the largest of
- c, the time its multiplies take;
- i, the time to issue them;
- (L + c) / S, one slot's round trip (load-to-use latency L, then the
  multiply) shared by the S slots in flight.

A CTA running B blocks back to back therefore takes B * max(c, i, (L + c)/S).
S = 1 serialises load and multiply; from S = (L + c)/c on, the multiplies
bound the loop.

Host-only arithmetic: no GPU and no measurement here.  bench.py fits L and
c from two points of a measured sweep and prints the model's prediction
beside every other point.
"""
from __future__ import annotations


def block_time(c: float, latency: float, stages: int, issue: float = 0.0) -> float:
    """Steady-state time per K block with `stages` slots."""
    if stages < 1:
        raise ValueError("stages must be at least 1")
    return max(c, issue, (latency + c) / stages)


def loop_time(blocks: float, c: float, latency: float, stages: int, issue: float = 0.0) -> float:
    """Time of `blocks` K blocks through the ring."""
    return blocks * block_time(c, latency, stages, issue)


def saturation_stages(c: float, latency: float) -> float:
    """The ring depth from which the multiplies, not the latency, bound the loop."""
    return (latency + c) / c


def fit(blocks: float, t_serial: float, t_saturated: float) -> tuple[float, float]:
    """(c, L) from the time with one slot (blocks * (L + c)) and the time
    with enough slots that the multiplies bound the loop (blocks * c)."""
    if blocks <= 0 or t_saturated <= 0 or t_serial < t_saturated:
        raise ValueError("need blocks > 0 and 0 < t_saturated <= t_serial")
    c = t_saturated / blocks
    return c, t_serial / blocks - c


def predict_sweep(blocks: float, t_serial: float, t_saturated: float, stages) -> dict:
    """Model times for each S in `stages`, fitted on the two given points."""
    c, latency = fit(blocks, t_serial, t_saturated)
    return {s: loop_time(blocks, c, latency, s) for s in stages}
