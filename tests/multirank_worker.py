"""One rank of the CPU multi-rank check, launched by tests/test_multirank.py
through torch.distributed.run (gloo backend, 127.0.0.1).

Each rank:
  1. sets up the process group the way bench.py does (env://, gloo on a host
     without CUDA);
  2. places a mixed list of matrices on owners with the library's LPT (host
     code) and checks that every rank computed the same placement;
  3. runs the fp64 oracle update for the matrices it owns, then all-gathers
     the results; rank 0 checks they equal a single-process update of every
     matrix bit for bit, each matrix updated exactly once;
  4. checks bench.shard (owner-placed and per-rank-batch configs) and the
     bench's cross-rank reductions.
Writes a one-line JSON summary to argv[1] + ".rank<r>".
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402
import newton_schulz_04_gb300 as m  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402


def main():
    out_path = sys.argv[1]
    world, rank, _ = bench.dist_setup(int(os.environ["WORLD_SIZE"]))
    assert world == 2 and dist.get_backend() == "gloo"

    # 2. placement, identical on every rank
    shapes = [(24, 40), (40, 24), (32, 32), (16, 64), (24, 40), (48, 16), (32, 32), (8, 56), (56, 8)]
    costs = m.cost_estimate(shapes, steps=5, dtype=torch.float32)
    owner, load = m.partition(costs, world, exact_limit=12)
    seen = [None] * world
    dist.all_gather_object(seen, owner)
    assert all(o == owner for o in seen), seen
    mine = [i for i, r in enumerate(owner) if r == rank]

    # 3. the owners' updates, gathered, equal the single-process update
    def inputs(i):
        mm, nn = shapes[i]
        g = synth.normal((mm, nn), 1.0, 50 + i).double().numpy()
        w = synth.normal((mm, nn), 0.02, 150 + i).double().numpy()
        return w, g, np.zeros((mm, nn))

    res = {}
    for i in mine:
        w, g, mo = inputs(i)
        w1, mo1, _ = oracle.muon_update(w, g, mo, beta=0.95, lr=0.02, steps=5)
        res[i] = (w1.tolist(), mo1.tolist())
    gathered = [None] * world
    dist.all_gather_object(gathered, res)
    merged = {}
    for part in gathered:
        assert not set(part) & set(merged), "a matrix was updated on two owners"
        merged.update(part)
    assert sorted(merged) == list(range(len(shapes)))
    if rank == 0:
        for i in range(len(shapes)):
            w, g, mo = inputs(i)
            w1, mo1, _ = oracle.muon_update(w, g, mo, beta=0.95, lr=0.02, steps=5)
            assert np.array_equal(np.array(merged[i][0]), w1) and np.array_equal(np.array(merged[i][1]), mo1)

    # 4. bench's sharding and reductions
    tiny = [torch.zeros(a, b) for a, b in shapes]
    owned_work, scaling = bench.shard(synth.Workload("c4", list(shapes), tiny, tiny), rank, world)
    assert scaling == "strong"
    parts = [None] * world
    dist.all_gather_object(parts, owned_work.shapes)
    assert sorted(parts[0] + parts[1]) == sorted(shapes)
    mine_bf16 = m.owned(shapes, rank, world, steps=5, dtype=torch.bfloat16)  # the workload's dtype
    assert owned_work.shapes == [shapes[i] for i in mine_bf16]
    batch_work, scaling_b = bench.shard(synth.Workload("c2", list(shapes), tiny, tiny), rank, world)
    assert scaling_b == "weak" and batch_work.shapes == shapes
    assert bench.max_over_ranks(float(rank + 1), world) == 2.0
    assert bench.sum_over_ranks(float(rank + 1), world) == 3.0
    bench.barrier(world)
    with open(f"{out_path}.rank{rank}", "w") as f:
        json.dump({"rank": rank, "owned": mine, "load": load, "ok": True}, f)
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
