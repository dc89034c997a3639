"""The bandwidth-adaptive level choice of the streaming path (host logic):
the finest level whose estimated piece size fits the link's rate times the
time budget, unmeasured levels tried, the coarsest when nothing fits, and the
estimates following the observed sizes."""
import pytest

from kv_cache_compression_cg_gb300.stream import AdaptiveLevels


def test_finest_fitting_level():
    # 3 levels at 100, 50, 20 bytes per token; pieces of 512 tokens; 1 ms per piece
    pol = AdaptiveLevels(3, 1e-3, bytes_per_second=60e6, prior_bytes_per_token=[100, 50, 20])
    assert pol.level_for(512) == 0           # 51.2 KB fits 60 KB
    pol.set_rate(30e6)
    assert pol.level_for(512) == 1           # 51.2 KB > 30 KB >= 25.6 KB
    pol.set_rate(12e6)
    assert pol.level_for(512) == 2           # 10.24 KB fits 12 KB
    pol.set_rate(1e6)
    assert pol.level_for(512) == 2           # nothing fits: the coarsest


def test_unmeasured_levels_are_tried_and_estimates_follow():
    pol = AdaptiveLevels(2, 1e-3, bytes_per_second=10e6, smoothing=0.5)
    assert pol.level_for(100) == 0           # nothing known: the finest
    pol.observe(0, 100, 50_000)              # 500 B/token: 50 KB > 10 KB
    assert pol.level_for(100) == 1           # level 1 not seen yet: try it
    pol.observe(1, 100, 20_000)              # 200 B/token: 20 KB > 10 KB
    assert pol.level_for(100) == 1           # nothing fits: the coarsest
    pol.observe(0, 100, 5_000)               # 0.5 * 500 + 0.5 * 50 = 275 B/token
    assert pol.est[0] == pytest.approx(275.0)
    pol.set_rate(30e6)                       # 27.5 KB fits 30 KB
    assert pol.level_for(100) == 0


def test_arguments_checked():
    with pytest.raises(ValueError):
        AdaptiveLevels(0, 1e-3, 1e6)
    with pytest.raises(ValueError):
        AdaptiveLevels(2, 1e-3, 1e6, prior_bytes_per_token=[1.0])
    with pytest.raises(ValueError):
        AdaptiveLevels(2, -1.0, 1e6)
    with pytest.raises(ValueError):
        AdaptiveLevels(2, 1e-3, 1e6).set_rate(0)
