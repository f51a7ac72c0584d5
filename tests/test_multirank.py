"""The N > 1 path on CPU: two gloo ranks launched by torch.distributed.run,
as bench.py is launched for several GPUs.  See tests/multirank_worker.py for
what each rank checks (same placement on every rank, owner-sharded oracle
updates equal to the single-process update, bench's sharding and reductions)."""
import json
import os
import socket
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_place_and_update_every_matrix_once(tmp_path):
    from newton_schulz_04_gb300 import build as b
    b.build()
    out = str(tmp_path / "mr")
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}",
           os.path.join(HERE, "multirank_worker.py"), out]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    ranks = [json.load(open(f"{out}.rank{q}")) for q in range(2)]
    assert all(x["ok"] for x in ranks)
    owned = sorted(ranks[0]["owned"] + ranks[1]["owned"])
    assert owned == list(range(9))
    assert ranks[0]["load"] == ranks[1]["load"]
