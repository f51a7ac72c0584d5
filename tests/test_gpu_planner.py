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


@pytest.mark.gpu
def test_schedules_are_chosen_per_shape_by_measurement_and_cached():
    """DMuon technical summary, §2.3-2.4: profile each shape and pick its
    kernel configuration by measurement, cached.  Candidates per group are the
    accurate schedules (bf16: original space, Gram restarted every two steps)
    with shared or separate launches; the choice is the measured fastest, and
    a square group (where Gram space saves nothing) and a 1:8 group (where
    the restarted Gram recurrence saves ~40 % of the work) are timed at their
    real batch widths."""
    import newton_schulz_04_gb300 as m
    m.load(build_if_missing=True)
    shapes = [(1024, 1024)] * 16 + [(512, 4096)] * 6 + [(4096, 512)] * 2
    cache = {}
    chosen = m.tune_schedules(shapes, steps=5, cache=cache)
    print("\n| group (width) | chosen | " + " | ".join(m.schedule_candidates()) + " |")
    for key, entry in sorted(cache.items()):
        assert set(entry["ms"]) == set(m.schedule_candidates())
        assert entry["best"] == min(entry["ms"], key=entry["ms"].get)
        print(f"| {key} | {entry['best']} | " + " | ".join(f"{entry['ms'][c]:.3f}" for c in m.schedule_candidates())
              + " |")
    assert set(chosen) == {(1024, 1024), (512, 4096)} and len(cache) == 2
    assert chosen[(512, 4096)].startswith("gram_r2")
    assert m.tune_schedules(shapes, steps=5, cache=cache) == chosen  # served from the cache
    # the updater runs every group with its own measured schedule: the same
    # results, bit for bit, as calling each group with that schedule directly
    g = torch.Generator().manual_seed(3)
    G = [torch.randn(a, b, generator=g).to(torch.bfloat16).cuda() for (a, b) in shapes]
    W0 = [torch.randn(a, b, generator=g).mul_(0.02).to(torch.bfloat16).cuda() for (a, b) in shapes]
    Wt = [w.clone() for w in W0]
    upd = m.MuonUpdater(Wt, 0.95, 0.02, 5, schedule="tuned", tune_cache=cache, use_graph=True)
    assert upd.chosen == chosen
    upd.step(G)
    upd.step(G)  # graph replay
    Wd = [w.clone() for w in W0]
    Md = [torch.zeros(w.shape, dtype=torch.float32, device="cuda") for w in W0]
    for _ in range(2):
        for key in ((1024, 1024), (512, 4096)):
            idx = [i for i, sh in enumerate(shapes) if (min(sh), max(sh)) == key]
            m.muon_step([Wd[i] for i in idx], [G[i] for i in idx], [Md[i] for i in idx], 0.95, 0.02, 5,
                        schedule=chosen[key])
    torch.cuda.synchronize()
    for a, b in zip(Wt, Wd):
        assert torch.equal(a, b)
    for a, b in zip(upd.moms, Md):
        assert torch.equal(a, b)


@pytest.mark.gpu
def test_launch_mode_flags_do_not_change_the_numbers():
    import newton_schulz_04_gb300 as m
    m.load(build_if_missing=True)
    g = torch.Generator().manual_seed(4)
    X = torch.randn(3, 512, 2048, generator=g).to(torch.bfloat16).cuda()
    outs = [m.ns_batched(X, steps=5, schedule=s) for s in ("gram_r2", "gram_r2+shared", "gram_r2+separate")]
    outs += [m.ns_batched(X, steps=5, schedule=s) for s in ("orig", "orig+shared", "orig+separate")]
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert torch.equal(outs[3], outs[4]) and torch.equal(outs[3], outs[5])
