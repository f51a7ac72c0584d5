"""Placement with measured costs (DMuon technical summary, §2.3: profile each
shape's update time, then place by makespan)."""
import pytest
import torch


@pytest.mark.gpu
def test_measured_costs_agree_with_the_model_and_are_cached():
    import newton_schulz_04_gb300 as m
    m.load(build_if_missing=True)
    shapes = [(1024, 1024)] * 4 + [(512, 2048)] * 3 + [(2048, 512)] + [(256, 1024)] * 6
    cache = {}
    meas = m.measure_costs(shapes, steps=5, cache=cache)
    model = m.cost_estimate(shapes, steps=5)
    assert all(x > 0 for x in meas)
    # one entry per (short, long) group; the transposed member shares its group's cost
    assert len(cache) == 3 and meas[7] == meas[4]
    for a, b in zip(meas, model):
        assert 0.2 < a / b < 20, (a, b)   # small batches pay fixed launch costs the model leaves out
    again = m.measure_costs(shapes, steps=5, cache=cache)
    assert again == meas                  # served from the cache
    owner, load = m.partition(meas, 3)
    assert sorted(set(owner)) == [0, 1, 2]
    assert max(load) <= sum(meas) / 3 + max(meas) + 1e-12
