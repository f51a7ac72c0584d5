"""Benchmark of the owner-side Muon update on GB300.

One step = one pass of the whole update over a batch of synthetic matrices:
momentum accumulate + pack + norm, Newton-Schulz (5 steps, quintic), and the
apply W <- W - lr O, through the C ABI (muon_step).

Default workload: every 2-D matrix of a Llama-style 32-layer model with
d = 4096 and ffn = 14336 (q, k, v, o 4096x4096; gate, up 4096x14336; down
14336x4096; 7.78e9 parameters), bf16 gradients N(0, 1e-6) and weights, fp32
momentum.  Other workloads (--config): c2 (16 square 1024x1024 bf16 matrices,
the square case where Gram space gives no reduction), c4 (512 mixed small
matrices), c5_n<N>[_t<T>] and c5f32_n<N>[_t<T>] (1024 x N, batch 8, T NS
steps, 5 by default), c3_l<L> (the first L layers of the model).

Prints one JSON line (rank 0).  `value` is algorithmic TFLOP/s over all ranks
(symmetric Gram count 3 s^2 l + (4T - 3) s^3 per matrix), with inputs resident
in HBM; `e2e` is the same metric with the gradients copied from pinned host
memory and the updated weights copied back inside the timed region.
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload instead.

`--record-traffic CSV` reads an ncu log (`--csv --log-file` of the metrics
dram__bytes_read.sum, dram__bytes_write.sum, gpu__time_duration.sum) taken on
`--config`, and stores the mean DRAM bytes per launch of each kernel family
in profiles/dram_traffic.json, from which `roofline.traffic` is taken.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# fp32 FFMA peak from unit counts: 152 SMs x 128 FP32 lanes x 2 flops per FMA x SM clock
FP32_LANES = 152 * 128


def fp32_alu_peak_tflops(sm_mhz):
    return FP32_LANES * 2 * sm_mhz * 1e6 / 1e12


def peaks():
    """Roofline denominators: MEASURED_PEAKS.json if present, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            flat = {}

            def walk(x, pre=""):
                if isinstance(x, dict):
                    for k, v in x.items():
                        walk(v, f"{pre}{k}.")
                elif isinstance(x, (int, float)):
                    flat[pre[:-1]] = float(x)
            walk(d)
            hbm = next((v for k, v in flat.items() if "hbm" in k.lower() and "gb" in k.lower()), None)
            bf = next((v for k, v in flat.items() if "bf16" in k.lower() and "sustain" not in k.lower()
                       and "tflop" in k.lower()), None)
            bfs = next((v for k, v in flat.items() if "bf16" in k.lower() and "sustain" in k.lower()), None)
            if hbm and bf:
                return {"hbm_gbs": hbm, "bf16_tflops": bf, "bf16_tflops_sustained": bfs or bf,
                        "source": "measured"}
        except Exception:
            pass
    return dict(FALLBACK, source="fallback")


# source file of each kernel family (a recorded traffic row is valid only while
# its family's source is unchanged)
FAMILY_SOURCES = {"tc_gemm": "tc_gemm.cu", "simt_gemm": "simt_gemm.cu", "pack": "elementwise.cu",
                  "norm_finalize": "elementwise.cu", "final": "elementwise.cu", "adamw_tail": "adamw.cu"}
TRAFFIC_JSON = os.path.join("profiles", "dram_traffic.json")


def family_of(name: str) -> str:
    """Kernel family of a launch label of the library's profiler ("tc_rect",
    "tc_program", ...) or of an ncu kernel name ("void muon::tc_gemm_kernel<16>(...)")."""
    n = name.lower()
    for key, fam in (("tc_", "tc_gemm"), ("simt", "simt_gemm"), ("pack", "pack"), ("norm", "norm_finalize"),
                     ("final", "final"), ("adamw", "adamw_tail"), ("fill_diag", "norm_finalize")):
        if key in n:
            return fam
    return n


def source_sha(family: str, root=None) -> str | None:
    import hashlib
    src = FAMILY_SOURCES.get(family)
    if src is None:
        return None
    try:
        data = open(os.path.join(root or ROOT, "newton_schulz_04_gb300", "csrc", src), "rb").read()
    except OSError:
        return None
    return hashlib.sha256(data).hexdigest()[:16]


def recorded_traffic(workload: str, family: str):
    """Mean DRAM bytes (read + write) per launch of a kernel family on a
    workload, from profiles/dram_traffic.json, or None when there is no row, or
    when the family's source has changed since the row was recorded."""
    try:
        rows = json.load(open(os.path.join(ROOT, TRAFFIC_JSON)))["rows"]
    except (OSError, ValueError, KeyError):
        return None
    for r in rows:
        if r.get("workload") == workload and r.get("family") == family:
            if r.get("source_sha16") != source_sha(family):
                return None
            return float(r["bytes_per_launch"])
    return None


_UNITS = {"byte": 1.0, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12, "b": 1.0, "kb": 1e3, "mb": 1e6,
          "gb": 1e9, "nsecond": 1e-9, "usecond": 1e-6, "msecond": 1e-3, "second": 1.0, "ns": 1e-9, "us": 1e-6,
          "ms": 1e-3, "s": 1.0}


def parse_ncu_csv(path):
    """{launch id: {"kernel": name, metric: value in bytes or seconds}} from an
    ncu `--csv --log-file` metrics log (one row per launch and metric)."""
    import csv
    launches = {}
    with open(path, newline="") as f:
        lines = [ln for ln in f if ln.startswith('"')]  # ncu's own ==PROF== lines are not CSV
    for row in csv.DictReader(lines):
        try:
            lid = int(row["ID"])
            val = float(row["Metric Value"].replace(",", ""))
        except (KeyError, ValueError):
            continue
        d = launches.setdefault(lid, {"kernel": row.get("Kernel Name", "")})
        d[row["Metric Name"]] = val * _UNITS.get(row.get("Metric Unit", "").strip().lower(), 1.0)
    return launches


def record_traffic(csv_path, workload, command, scale=1.0, note=""):
    """Average the captured launches per kernel family and store them (the
    traffic per launch of `workload`, scaled by `scale` when the capture ran a
    smaller case with the same launch structure) in profiles/dram_traffic.json."""
    launches = parse_ncu_csv(csv_path)
    fams = {}
    for d in launches.values():
        if "dram__bytes_read.sum" not in d or "dram__bytes_write.sum" not in d:
            continue
        f = fams.setdefault(family_of(d["kernel"]), [0, 0.0, 0.0, 0.0])
        f[0] += 1
        f[1] += d["dram__bytes_read.sum"]
        f[2] += d["dram__bytes_write.sum"]
        f[3] += d.get("gpu__time_duration.sum", 0.0)
    path = os.path.join(ROOT, TRAFFIC_JSON)
    try:
        doc = json.load(open(path))
    except (OSError, ValueError):
        doc = {"rows": []}
    doc["about"] = ("DRAM bytes per launch by kernel family, averaged over the captured launches "
                    "(ncu dram__bytes_read.sum + dram__bytes_write.sum), written by bench.py --record-traffic")
    rows = [r for r in doc.get("rows", []) if not (r.get("workload") == workload and r.get("family") in fams)]
    for fam, (n, rd, wr, t) in sorted(fams.items()):
        rows.append({"workload": workload, "family": fam, "source_sha16": source_sha(fam), "launches": n,
                     "read_bytes_per_launch": scale * rd / n, "write_bytes_per_launch": scale * wr / n,
                     "bytes_per_launch": scale * (rd + wr) / n, "ncu_us_per_launch": 1e6 * t / n,
                     "scale": scale, "note": note, "command": command})
    doc["rows"] = sorted(rows, key=lambda r: (r["workload"], r["family"]))
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")
    return doc


def c5_params(name: str):
    """(n, NS steps) of a c5 config name: c5[f32][_n<N>][_t<T>]."""
    n, steps = 4096, 5
    for part in name.split("_")[1:]:
        if part.startswith("n"):
            n = int(part[1:])
        elif part.startswith("t"):
            steps = int(part[1:])
    return n, steps


def workload_desc(name: str) -> str:
    if name.startswith("c3_l") and name[4:].isdigit():
        return (f"the first {name[4:]} layers of the d=4096 ffn=14336 model (per layer 4 x 4096^2, 2 x 4096x14336, "
                f"14336x4096), bf16 grads N(0,1e-6), fp32 momentum, 5 NS steps")
    if name.startswith("c5"):
        n, steps = c5_params(name)
        dt = "fp32" if name.startswith("c5f32") else "bf16"
        return f"8 x 1024x{n} {dt} grads N(0,1) with row 0 x100, fp32 momentum, {steps} NS steps quintic"
    return WORKLOAD_DESC.get(name, name)


def operands_desc(dtype, schedule):
    if schedule.startswith("orig_f16x3"):
        return ("fp16-pair tensor-core operands (about 22 bits), three products per product, fp32 accumulation; "
                f"{'fp32' if dtype == torch.float32 else 'bf16'} in and out")
    if dtype == torch.float32:
        return "fp32 FFMA on the CUDA cores"
    return ("bf16 in and out; NS products on bf16 (step 0) and fp16 (later steps) tensor-core operands, "
            "fp32 accumulation")


def make_workload(name: str, device):
    if name == "c2":
        return synth.c2(device)
    if name == "c3":
        return synth.c3(device)
    if name == "c3_layer":  # one layer of c3 (same shapes), for profiling
        return synth.c3(device, layers=1)
    if name.startswith("c3_l") and name[4:].isdigit():  # the first L layers of c3
        return synth.c3(device, layers=int(name[4:]))
    if name == "c4":
        return synth.c4(device)
    if name == "c1":
        return synth.c1()
    if name.startswith("c5"):
        n, steps = c5_params(name)
        return synth.c5(device, n=n, dtype=torch.float32 if name.startswith("c5f32") else torch.bfloat16,
                        steps=steps)
    raise SystemExit(f"unknown config {name}")


WORKLOAD_DESC = {
    "c2": "16x square 1024x1024 bf16 grads N(0,0.02^2), fp32 momentum, bf16 W, 5 NS steps quintic",
    "c3": "Llama-style 32 layers d=4096 ffn=14336 (q,k,v,o 4096^2; gate/up 4096x14336; down 14336x4096), "
          "bf16 grads N(0,1e-6), fp32 momentum, 5 NS steps",
    "c4": "512 matrices from {256x1024,512x2048,768x3072}, rank-8 + 1e-4 noise, bf16, 5 NS steps",
    "c1": "single 128x256 fp32 matrix N(0,1) seed 0, 5 NS steps, beta 0.95, lr 0.02",
    "c3_layer": "one layer of the d=4096 ffn=14336 model (4 x 4096^2, 2 x 4096x14336, 14336x4096), bf16, 5 NS steps",
}


def smi_id(local: int) -> str:
    """nvidia-smi's name for CUDA device `local` of this process: its UUID (the
    CUDA ordinal can name another GPU when CUDA_VISIBLE_DEVICES remaps)."""
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        if u:
            return u if u.startswith("GPU-") else f"GPU-{u}"
    except Exception:
        pass
    return str(local)


class Clocks:
    """Samples nvidia-smi every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={smi_id(self.index)}", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p is not None:
            self.p.terminate()
            try:
                self.out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (getattr(self, "out", "") or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            try:
                pw.append(float(f[3]))
            except ValueError:
                pass
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        out = {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}
        if pw:
            out["power_w"] = float(np.median(pw))
        return out


REJECTED_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(clocks) -> bool:
    """A timed region whose clock record shows a hardware or thermal slowdown,
    or an SM clock stuck far below its maximum with no reason (a leftover
    clock lock), is not a valid measurement.  sw_power_cap is kept."""
    reasons = clocks.get("reasons") or []
    if any(r in reasons for r in REJECTED_REASONS):
        return True
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    return bool(sm and mx and sm < 0.6 * mx and "sw_power_cap" not in reasons)


def measured_window(local, step, timed, k, world):
    """clock_window, re-measured once if its clock record is rejected; the
    first record is kept beside the second (`rejected_first`)."""
    ms, clocks = clock_window(local, step, timed, k, world)
    if clocks_rejected(clocks):
        first = clocks
        ms, clocks = clock_window(local, step, timed, k, world)
        clocks = dict(clocks, rejected_first=first)
    return ms, clocks


def clock_window(local, step, timed, k, world, pad_s=0.3):
    """Run the timed steps inside a sampling window of nvidia-smi: at least
    `pad_s` of untimed steps of the same workload before and after them keep
    the GPU under the same load while the 200 ms sampler records clocks, so a
    timed region of a few milliseconds still gets samples."""
    def pad():
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        n = 1  # grow the batch of steps between clock checks, so long steps pad by one or two steps
        while time.perf_counter() - t0 < pad_s:
            for _ in range(n):
                step()
            torch.cuda.synchronize()
            n = min(2 * n, 64)
    t0 = time.perf_counter()
    with Clocks(local) as clk:
        pad()
        barrier(world)  # the timed steps are bracketed by a barrier and a synchronize on both sides
        torch.cuda.synchronize()
        ms = timed(step, k)  # synchronizes at its end
        barrier(world)
        pad()
    summary = clk.summary()
    summary["window_s"] = round(time.perf_counter() - t0, 3)
    summary["timed_s"] = round(sum(ms) / 1e3, 4)
    return ms, summary


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def sum_over_ranks(x, world):
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# Configs that are one model's whole set of matrices: with N ranks each matrix
# is updated by one owner (strong scaling).  The other configs are a batch per
# rank (weak scaling).
OWNER_PLACED = ("c3", "c4")


def shard(work, rank, world):
    """This rank's part of the workload and the scaling it implies.  Placement
    is the library's LPT over its cost model, computed identically on every
    rank (no communication)."""
    if world <= 1 or work.name not in OWNER_PLACED:
        return work, "weak"
    import dataclasses
    import newton_schulz_04_gb300 as pkg
    mine = pkg.owned(work.shapes, rank, world, steps=work.steps, dtype=work.dtype)
    sub = dataclasses.replace(work, shapes=[work.shapes[i] for i in mine],
                              grads=[work.grads[i] for i in mine] if work.grads else [],
                              weights=[work.weights[i] for i in mine] if work.weights else [])
    return sub, "strong"


def max_over_ranks(x, world):
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def host_copy_gbs(dev, nbytes=1 << 30):
    """This box's pinned host <-> device copy rates in GB/s, best of 3 copies of
    1 GiB: each direction alone, and the total of both directions at once (as
    the end-to-end pass runs them).  The end-to-end figure is bound by them
    when a step's copies take longer than its compute."""
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def h2d():
        d_in.copy_(h_in, non_blocking=True)

    def d2h():
        h_out.copy_(d_out, non_blocking=True)

    def both():
        with torch.cuda.stream(s_in):
            h2d()
        with torch.cuda.stream(s_out):
            d2h()

    out = {}
    for name, fn, moved in (("h2d", h2d, nbytes), ("d2h", d2h, nbytes), ("both_total", both, 2 * nbytes)):
        best = float("inf")
        for _ in range(3):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            best = min(best, time.perf_counter() - t0)
        out[name] = moved / best / 1e9
    del h_in, h_out, d_in, d_out
    return out


def step_copy_gbs(dev, host_in, dev_in, host_out, dev_out):
    """The copy rates of one step's own buffers (all gradients in, all weights
    out), each direction alone and both at once, in GB/s: what the
    end-to-end pass can reach on this machine and these allocations."""
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    nin = sum(t.numel() * t.element_size() for t in host_in)
    nout = sum(t.numel() * t.element_size() for t in host_out)

    def h2d():
        with torch.cuda.stream(s_in):
            for d, h in zip(dev_in, host_in):
                d.copy_(h, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s_out):
            for h, d in zip(host_out, dev_out):
                h.copy_(d, non_blocking=True)

    out = {}
    for name, fns, moved in (("step_h2d", (h2d,), nin), ("step_d2h", (d2h,), nout), ("step_both_total", (h2d, d2h),
                                                                                       nin + nout)):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for fn in fns:
            fn()
        torch.cuda.synchronize(dev)
        out[name] = moved / (time.perf_counter() - t0) / 1e9
    return out


def cpu_baseline(work, budget_s=15.0, max_mats=None, start=0, of=None):
    """The fp64 oracle, as it stands, on a bounded sample of the workload
    (matrices from index `start` on, cyclically; `of` describes the whole
    workload the sample comes from)."""
    import oracle
    flops = 0.0
    done = 0
    t0 = time.perf_counter()
    n_all = len(work.shapes)
    order = [(start + k) % n_all for k in range(n_all)]
    for i in order:
        if max_mats is not None and done >= max_mats:
            break
        g = work.grads[i].detach().to("cpu")
        w = work.weights[i].detach().to("cpu")
        m, n = work.shapes[i]
        oracle.muon_update(w, g, np.zeros((m, n)), work.beta, work.lr, work.steps, work.coeffs)
        s, l = min(m, n), max(m, n)
        flops += 3.0 * s * s * l + (4 * work.steps - 3) * float(s) ** 3
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    cores = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info
        cores = max(int(x.get("num_threads", 1)) for x in threadpool_info()) or cores
    except Exception:
        pass
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} of {of or f'{n_all} matrices of the same workload'}, fp64 numpy, {dt:.1f} s",
            "seconds": dt, "matrices": done}


def c3_sample(work):
    """One matrix of each bucket of the model: layer 0's q (4096x4096) and down
    (14336x4096), drawn exactly as in the full workload (same seeded streams)."""
    pick = [i for i in (0, 6) if i < len(work.shapes)]
    return synth.Workload("c3_sample", [work.shapes[i] for i in pick], [work.grads[i].cpu() for i in pick],
                          [work.weights[i].cpu() for i in pick])


def run_reference(args, world, rank):
    if rank != 0:
        return
    of = None
    if args.config.startswith("c3"):
        # the model's first layer holds one matrix of each bucket; the oracle
        # takes one of them per step, in turn
        work = c3_sample(synth.c3("cpu", layers=1))
        of = f"sampled matrices (4096x4096 and 14336x4096) of {workload_desc(args.config)}"
        per_step = dict(max_mats=1)
    else:
        work = make_workload(args.config, "cpu")
        per_step = dict(budget_s=max(5.0, 60.0 / max(args.steps, 1)))
    steps = []
    for _ in range(args.warmup):
        cpu_baseline(synth.c1(), budget_s=1.0, max_mats=1)
    vals = []
    t_all = time.perf_counter()
    for k in range(args.steps):
        r = cpu_baseline(work, start=k, of=of, **per_step)
        vals.append(r)
        steps.append(r["seconds"])
    tot_flops = sum(v["value"] * 1e12 * v["seconds"] for v in vals)
    tot_s = sum(steps)
    value = tot_flops / tot_s / 1e12
    line = {
        "impl": "reference", "metric": "Muon update TFLOP/s (algorithmic, symmetric Gram count)", "value": value,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_s / max(args.steps, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(args.config), "name": args.config,
                   "sample": vals[0]["sample"]},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": vals[0]["cores"], "kind": "oracle",
                         "sample": vals[0]["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": time.perf_counter() - t_all,
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import newton_schulz_04_gb300 as pkg
    pkg.load(build_if_missing=True)
    dev = torch.device("cuda", local)
    work = make_workload(args.config, dev if args.config.startswith("c3") else "cpu")
    work, scaling = shard(work, rank, world)
    if not work.shapes:
        raise SystemExit(f"rank {rank} owns no matrix of {args.config} at world size {world}")
    shapes = work.shapes
    count = len(shapes)
    W = [w.to(dev) for w in work.weights]
    G = [g.to(dev) for g in work.grads]
    # The end-to-end pass's buffers come first, before the workspace and the
    # timed work: on a box whose GPU memory earlier processes have used, host
    # copies into and out of buffers allocated later ran slower (c3 end to end
    # 785-794 TFLOP/s against 879-932 allocated here; the same on a fresh box).
    G2 = [g.clone() for g in G]  # the second gradient buffer of the end-to-end pass
    Gh = [torch.empty(g.shape, dtype=g.dtype).pin_memory() for g in G]
    for gh, g in zip(Gh, G):
        gh.copy_(g)
    Wh = [torch.empty(w.shape, dtype=w.dtype).pin_memory() for w in W]
    # With one shape group nothing else computes while its weights leave, so
    # the copy-out reads a device snapshot and the next step starts at once.
    # With several groups the later groups cover the copy-out, and a snapshot
    # only adds work (measured: c3 1025 -> 996 TFLOP/s end to end, c4 244 -> 215).
    snapshot = len({(min(a, b), max(a, b)) for a, b in work.shapes}) == 1
    Ws = [torch.empty_like(w) for w in W] if snapshot else W
    if not args.config.startswith("c3"):
        cpu_work = work
    else:
        cpu_work = None
    t_tune = time.perf_counter()
    # largest groups first: the end-to-end pass copies each group's weights out
    # while the groups after it compute
    upd = pkg.MuonUpdater(W, work.beta, work.lr, work.steps, work.coeffs, args.schedule, use_graph=not args.no_graph,
                          group_order="largest_first")
    t_tune = time.perf_counter() - t_tune
    Mo = upd.moms
    flops_step = work.flop_count()
    flops_all = sum_over_ranks(flops_step, world)  # = world x flops_step under weak scaling
    count_all = sum_over_ranks(count, world)
    in_bytes = sum(g.numel() * g.element_size() for g in G) + sum(m.numel() * 4 for m in Mo) * 2 + \
        sum(w.numel() * w.element_size() for w in W) * 2
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if in_bytes < 4 * L2_BYTES else None
    st = torch.cuda.current_stream(dev)

    def step():
        upd.step(G)

    def step_eager():
        upd._eager(G, st)

    def timed(fn, k):
        out = []
        for _ in range(k):
            if flush is not None:
                flush.zero_()  # evict L2 between timed steps (outside the events)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(st)
            fn()
            b.record(st)
            out.append((a, b))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in out]

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert pkg.device_status(upd.workspace) == 0
    # ---- timed region: device-resident inputs, one replay (or call) per step
    barrier(world)
    torch.cuda.synchronize()
    ms, clocks = measured_window(local, step, timed, args.steps, world)
    barrier(world)
    # ---- a second pass of the same steps, called directly with a CUDA-event
    # pair around every library launch, gives the per-kernel times (events
    # between kernels stop launches from overlapping, so this pass is slower)
    pkg.profile_enable(True)
    ms_eager = timed(step_eager, args.steps)
    pkg.profile_enable(False)
    recs = pkg.profile_records()
    assert pkg.device_status(upd.workspace) == 0
    t_total = max_over_ranks(sum(ms) / 1e3, world)
    ms_step = 1e3 * t_total / args.steps
    value = flops_all * args.steps / t_total / 1e12
    value_eager = flops_all * args.steps / max_over_ranks(sum(ms_eager) / 1e3, world) / 1e12
    # per-launch-label totals of the profiled pass, then per kernel family
    # (tc_syrk / tc_sym / tc_rect / tc_program are launches of one kernel)
    by = {}
    for k, t, fl, byt in recs:
        d = by.setdefault(k, [0.0, 0, 0.0, 0.0])
        d[0] += t
        d[1] += 1
        d[2] += fl
        d[3] += byt
    fam = {}
    for k, v in by.items():
        d = fam.setdefault(family_of(k), [0.0, 0, 0.0, 0.0])
        for i in range(4):
            d[i] += v[i]
    dom = max(fam, key=lambda k: fam[k][0])
    pk = peaks()
    # a kernel inside a seconds-long step runs under the power cap: sustained peak
    sustained = ms_step >= 100.0
    tc_peak = pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]
    traffic = recorded_traffic(args.config, dom)
    tot_launch_ms = sum(v[0] for v in by.values())
    t_dom = fam[dom][0] / 1e3
    common = {"kernel": dom, "traffic": traffic, "launches": fam[dom][1], "avg_launch_ms": fam[dom][0] / fam[dom][1],
              "share_of_launch_time": fam[dom][0] / tot_launch_ms,
              "launch_labels": sorted(k for k in by if family_of(k) == dom)}
    if dom in ("tc_gemm", "simt_gemm"):
        # achieved: the method's algorithmic count (symmetric Gram form,
        # 3 s^2 l + (4T - 3) s^3 per matrix) of the steps the profiled pass ran,
        # over the family's summed launch time; executed: the products the
        # schedule actually ran (lower tiles of symmetric outputs counted once)
        achieved = flops_step * args.steps / t_dom / 1e12
        executed = fam[dom][2] / t_dom / 1e12
        if dom == "simt_gemm":
            mhz = clocks.get("sm_mhz") or 2070.0
            peak = fp32_alu_peak_tflops(mhz)
            roof = dict(bound="alu", achieved=achieved, peak=peak, unit="TFLOP/s", frac=achieved / peak,
                        executed_tflops=executed, executed_frac=executed / peak,
                        peak_source=f"152 SMs x 128 FP32 lanes x 2 flops x {mhz:.0f} MHz (sampled median, else max)")
        else:
            roof = dict(bound="tensor", achieved=achieved, peak=tc_peak, unit="TFLOP/s", frac=achieved / tc_peak,
                        executed_tflops=executed, executed_frac=executed / tc_peak,
                        peak_source=pk["source"] + (" sustained" if sustained else " burst"))
    else:
        achieved = fam[dom][3] / t_dom / 1e9
        roof = dict(bound="hbm", achieved=achieved, peak=pk["hbm_gbs"], unit="GB/s", frac=achieved / pk["hbm_gbs"],
                    peak_source=pk["source"])
    roof.update(common)
    kernels = {k: {"launches": v[1], "ms_total": v[0], "share": v[0] / tot_launch_ms,
                   "executed_tflops": (v[2] / (v[0] / 1e3) / 1e12) if v[2] else None,
                   "gbs": (v[3] / (v[0] / 1e3) / 1e9) if v[3] else None} for k, v in by.items()}
    # ---- end to end through the C ABI with host buffers (pinned).  Every step
    # copies its gradients in from pinned host memory and the updated weights
    # back out.  The copy of step k+1's gradients runs on a second stream into
    # the other of two device gradient buffers while step k computes.  As soon
    # as a shape group's update is done, a third stream copies its weights out
    # to the host while the later groups compute; the group's next update
    # waits for that copy (or, with a single group, only for a device
    # snapshot that the host copy then reads).
    h2d = sum(g.numel() * g.element_size() for g in Gh)
    d2h = sum(w.numel() * w.element_size() for w in Wh)
    Gsets = [G, G2]
    cs = torch.cuda.Stream(dev)
    cs_out = torch.cuda.Stream(dev)
    ngroups = len(upd.groups)
    link = host_copy_gbs(dev)
    link.update(step_copy_gbs(dev, Gh, Gsets[1], Wh, W))

    def e2e_run(k):
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_used = [torch.cuda.Event(), torch.cuda.Event()]
        ev_snap = [torch.cuda.Event() for _ in range(ngroups)]  # group g's weights are snapshotted
        ev_out = [torch.cuda.Event() for _ in range(ngroups)]  # group g's weights are on the host

        def copy_in(i):
            with torch.cuda.stream(cs):
                cs.wait_event(ev_used[i])  # the step that last read buffer i is done
                for g, gh in zip(Gsets[i], Gh):
                    g.copy_(gh, non_blocking=True)
                ev_in[i].record(cs)

        def before_group(gi, idx, s):
            s.wait_event(ev_snap[gi])  # the previous step's weights of this group are snapshotted

        def after_group(gi, idx, s):
            done = torch.cuda.Event()
            done.record(s)
            with torch.cuda.stream(cs_out):
                cs_out.wait_event(done)
                if snapshot:
                    for q in idx:
                        Ws[q].copy_(W[q], non_blocking=True)
                    ev_snap[gi].record(cs_out)
                for q in idx:
                    Wh[q].copy_(Ws[q], non_blocking=True)
                if not snapshot:
                    ev_snap[gi].record(cs_out)  # the group's next update waits for the copy itself
                ev_out[gi].record(cs_out)

        if flush is not None:
            flush.zero_()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for i in (0, 1):
            ev_used[i].record(st)
        for e in ev_snap + ev_out:
            e.record(st)
        copy_in(0)
        for s_ in range(k):
            i = s_ % 2
            if s_ + 1 < k:
                copy_in(1 - i)
            st.wait_event(ev_in[i])
            if args.no_graph:
                upd._eager(Gsets[i], st, before_group, after_group)
            else:
                upd.step(Gsets[i], st, before_group, after_group)
            ev_used[i].record(st)
        for e in ev_out:  # the last step's weights are all on the host
            st.wait_event(e)
        b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    e2e_run(max(args.warmup, 2))  # both gradient buffers get their graphs here
    with Clocks(local) as e2e_clk:  # the copies draw power too: the clocks of this pass, reported beside it
        e2e_ms = e2e_run(args.steps)
    e2e_t = max_over_ranks(e2e_ms / 1e3, world)
    e2e_val = flops_all * args.steps / e2e_t / 1e12
    launches_per_step = len(recs) / args.steps
    line = {
        "metric": "Muon update TFLOP/s (algorithmic, symmetric Gram count)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": scaling, "vs_baseline": None,
        "dtype": ("fp16x2" if any(c.startswith("orig_f16x3") for c in upd.chosen.values()) else
                  "fp32" if work.dtype == torch.float32 else "bf16+fp16"),
        "operands": operands_desc(work.dtype, next(iter(upd.chosen.values()))),
        "data": "synthetic",
        "config": {"workload": workload_desc(args.config), "name": args.config,
                   "matrices_per_gpu": count, "l2": "flushed between timed steps" if flush is not None
                   else "inputs larger than L2",
                   "parallelism": "1 gpu" if world == 1 else
                   (f"owner placement over {world} ranks (LPT), no data-path collective" if scaling == "strong"
                    else f"one batch per rank x{world}")},
        "schedules": {f"{a}x{b}": sc for (a, b), sc in sorted(upd.chosen.items())},
        "schedule_arg": args.schedule,
        "matrices_per_s": count_all * args.steps / t_total,
        "pct_of_bf16_peak": 100.0 * value / pk["bf16_tflops"],
        "value_without_graph": value_eager,
        "launch_path": "CUDA graph replay of the C-ABI calls, one graph per shape group" if not args.no_graph
                       else "direct C-ABI calls",
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "roofline_timing": "per-launch CUDA events in a second pass of the same steps",
        "roofline": roof,
        "kernels": kernels,
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelining": "step k+1's gradient copy-in overlaps step k on a second stream; each shape group's "
                              "weights are copied out on a third stream while the later groups compute (largest "
                              "groups first); with a single group, from a device snapshot while the next step "
                              "computes",
                "ms_per_step": 1e3 * e2e_t / args.steps,
                "host_copy_gbs": link, "clocks": e2e_clk.summary()},
        "clocks": clocks,
        "peaks": pk,
    }
    if args.schedule == "tuned":
        line["tuning_s"] = t_tune
    if rank == 0 and world == 1 and not args.no_cpu_baseline and cpu_work is not None:
        line["cpu_baseline"] = cpu_baseline(cpu_work, budget_s=args.cpu_budget)
    elif rank == 0 and world == 1 and not args.no_cpu_baseline:
        small = c3_sample(work)
        line["cpu_baseline"] = cpu_baseline(small, budget_s=args.cpu_budget, max_mats=len(small.shapes),
                                            of=f"2 sampled matrices (4096x4096 and 14336x4096) of the {count} "
                                               f"matrices of the workload")
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- AdamW tail
TAIL_DESC = {
    "tail": "AdamW tail: 2048 1-D tensors, lengths log-uniform in [1024, 131072] (seed 5), bf16 params and grads "
            "N(0,1) / N(0,1e-4), fp32 moments",
    "tail_c3": "AdamW tail of the 32-layer d=4096 model: 65 RMSNorm weight vectors of 4096, bf16",
}
TAIL_HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def tail_sizes(name):
    if name == "tail_c3":
        return [4096] * 65
    g = torch.Generator().manual_seed(5)
    return [int(1024 * 2.0 ** (7.0 * float(u))) for u in torch.rand(2048, generator=g)]


def tail_cpu_baseline(sizes, budget_s):
    """The fp64 oracle, as it stands, on a bounded sample of the tail."""
    import oracle
    g = torch.Generator().manual_seed(6)
    done_el = 0
    done = 0
    dt = 0.0  # time inside the oracle only (inputs are drawn outside it)
    for k in sizes:
        p = torch.randn(k, generator=g).to(torch.bfloat16).double().numpy()
        gr = (torch.randn(k, generator=g) * 1e-2).to(torch.bfloat16).double().numpy()
        m, v = np.zeros(k), np.zeros(k)
        t0 = time.perf_counter()
        oracle.adamw.adamw_step(p, gr, m, v, step=1, **TAIL_HP)
        dt += time.perf_counter() - t0
        done_el += k
        done += 1
        if dt > budget_s:
            break
    return {"value": done_el * 22.0 / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} of {len(sizes)} tensors ({done_el} elements), fp64 numpy, one step, {dt:.1f} s",
            "seconds": dt}


def run_tail(args, world, rank, local):
    import newton_schulz_04_gb300 as pkg
    pkg.load(build_if_missing=True)
    dev = torch.device("cuda", local)
    sizes = tail_sizes(args.config)
    gen = torch.Generator().manual_seed(7 + rank)
    # the tail packed into flat buffers (one per array), each tensor a view
    # starting on an 8-element (16-byte) boundary
    offs, off = [], 0
    for k in sizes:
        offs.append(off)
        off += (k + 7) // 8 * 8
    n_el = sum(sizes)
    flat_p = torch.zeros(off, dtype=torch.bfloat16, device=dev)
    flat_g = torch.zeros(off, dtype=torch.bfloat16, device=dev)
    flat_m = torch.zeros(off, dtype=torch.float32, device=dev)
    flat_v = torch.zeros(off, dtype=torch.float32, device=dev)
    for o, k in zip(offs, sizes):
        flat_p[o:o + k] = torch.randn(k, generator=gen).to(torch.bfloat16).to(dev)
        flat_g[o:o + k] = (torch.randn(k, generator=gen) * 1e-2).to(torch.bfloat16).to(dev)
    view = lambda t: [t[o:o + k] for o, k in zip(offs, sizes)]  # noqa: E731
    P, G, M, V = view(flat_p), view(flat_g), view(flat_m), view(flat_v)
    bytes_step = 22.0 * n_el  # read p, g (bf16), m, v (fp32); write p, m, v
    st = torch.cuda.current_stream(dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if bytes_step < 4 * L2_BYTES else None
    opt = pkg.AdamwTail(P, G, M, V, lr=TAIL_HP["lr"], betas=(TAIL_HP["beta1"], TAIL_HP["beta2"]), eps=TAIL_HP["eps"],
                        weight_decay=TAIL_HP["weight_decay"])

    def step():
        opt.step(st)

    def timed(fn, k):
        out = []
        for _ in range(k):
            if flush is not None:
                flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(st)
            fn()
            b.record(st)
            out.append((a, b))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in out]

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    ms, clocks = measured_window(local, step, timed, args.steps, world)
    barrier(world)
    t_total = max_over_ranks(sum(ms) / 1e3, world)
    value = world * bytes_step * args.steps / t_total / 1e9
    pk = peaks()
    launches = (len(sizes) + 511) // 512
    # end to end: the packed gradients from pinned host memory in, the packed
    # parameters back out, every step
    Gh = flat_g.cpu().pin_memory()
    Ph = torch.empty(flat_p.shape, dtype=flat_p.dtype).pin_memory()
    h2d = Gh.numel() * 2
    d2h = Ph.numel() * 2

    def e2e_step():
        flat_g.copy_(Gh, non_blocking=True)
        step()
        Ph.copy_(flat_p, non_blocking=True)

    e2e_ms = timed(e2e_step, args.steps)
    e2e_t = max_over_ranks(sum(e2e_ms) / 1e3, world)
    line = {
        "metric": "AdamW tail update GB/s (algorithmic bytes: 22 per bf16 element)", "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 params, fp32 math",
        "data": "synthetic",
        "config": {"workload": TAIL_DESC[args.config], "name": args.config, "tensors": len(sizes), "elements": n_el,
                   "l2": "flushed between timed steps" if flush is not None else "inputs larger than L2",
                   "parallelism": "1 gpu" if world == 1 else f"one tail per rank x{world}"},
        "gpu_launches": launches * args.steps,
        "roofline": {"bound": "hbm", "kernel": "adamw_tail", "achieved": value / world, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": value / world / pk["hbm_gbs"],
                     "traffic": recorded_traffic(args.config, "adamw_tail"), "peak_source": pk["source"]},
        "e2e": {"value": world * bytes_step * args.steps / e2e_t / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * e2e_t / args.steps},
        "clocks": clocks,
        "peaks": pk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = tail_cpu_baseline(sizes, min(args.cpu_budget, 15.0))
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_tail_reference(args, world, rank):
    if rank != 0:
        return
    sizes = tail_sizes(args.config)
    for _ in range(args.warmup):
        tail_cpu_baseline(sizes[:4], 1.0)
    vals = [tail_cpu_baseline(sizes, max(5.0, 60.0 / max(args.steps, 1))) for _ in range(args.steps)]
    tot_bytes = sum(v["value"] * 1e9 * v["seconds"] for v in vals)
    tot_s = sum(v["seconds"] for v in vals)
    value = tot_bytes / tot_s / 1e9
    print(json.dumps({
        "impl": "reference", "metric": "AdamW tail update GB/s (algorithmic bytes: 22 per bf16 element)",
        "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_s / max(args.steps, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": TAIL_DESC[args.config], "name": args.config, "sample": vals[0]["sample"]},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": vals[0]["sample"]},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c3")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="call the C ABI per step instead of replaying a graph")
    ap.add_argument("--schedule", default="auto", help="NS schedule (auto, orig, gram_r2, orig_f16x3, ..., with an "
                    "optional +shared / +separate launch mode), or tuned: the fastest per shape group, measured")
    ap.add_argument("--record-traffic", metavar="CSV", help="store the DRAM traffic of an ncu metrics log taken on "
                    "--config in profiles/dram_traffic.json (no GPU work)")
    ap.add_argument("--traffic-scale", type=float, default=1.0, help="with --record-traffic: the factor from the "
                    "captured workload's launches to --traffic-workload's")
    ap.add_argument("--traffic-workload", help="with --record-traffic: the workload the rows are for (default --config)")
    ap.add_argument("--traffic-command", default="", help="with --record-traffic: the command that made the log")
    args = ap.parse_args()
    if args.record_traffic:
        wl = args.traffic_workload or args.config
        note = "" if wl == args.config else f"captured on {args.config}, scaled by {args.traffic_scale:g}"
        doc = record_traffic(args.record_traffic, wl, args.traffic_command, args.traffic_scale, note)
        print(json.dumps([r for r in doc["rows"] if r["workload"] == wl]))
        return
    world, rank, local = dist_setup(args.gpus)
    tail = args.config in TAIL_DESC
    if args.impl == "reference":
        (run_tail_reference if tail else run_reference)(args, world, rank)
    else:
        (run_tail if tail else run_ours)(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
