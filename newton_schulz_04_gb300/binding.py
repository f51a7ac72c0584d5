"""ctypes binding of libmuon_ns.so (argument marshalling only).

Every step of the update runs in the library's CUDA kernels.  PyTorch is used
here only to own device memory (the workspace, outputs) and to name the CUDA
stream.  There is no fallback: if the library is missing or the device is not
an sm_103 GPU the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

import torch

from . import build as _build

OK, ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED = range(8)
STATUS_NAMES = ["OK", "ERR_ARG", "ERR_SHAPE", "ERR_ALIGN", "ERR_WORKSPACE", "ERR_CUDA", "ERR_TIMEOUT",
                "ERR_UNSUPPORTED"]
BF16, FP32, FP16 = 0, 1, 2  # FP16: muon_debug_gemm only
F16_LO_SCALE = 2048.0  # an fp16 pair stores lo = fp16((v - hi) * 2^11)
SCHED = {"auto": 0, "gram_x3": 1, "gram_x1": 2, "orig": 3, "orig_bf16": 4, "orig_f16x3": 5, "gram_r2": 6}
SCHED_NAMES = {v: k for k, v in SCHED.items()}
LAUNCH = {"": 0, "shared": 0x100, "separate": 0x200}  # "+shared" / "+separate" suffixes of a schedule name


def sched_code(name: str) -> int:
    """C-ABI value of a schedule name, optionally with a launch-mode suffix
    ("gram_r2+shared", "orig+separate")."""
    base, _, mode = name.partition("+")
    if base not in SCHED or mode not in LAUNCH:
        raise ValueError(f"unknown schedule {name!r}")
    return SCHED[base] | LAUNCH[mode]
WS_ALIGN = 256

_lib = None


class MuonError(RuntimeError):
    def __init__(self, status: int, msg: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES[status] if 0 <= status < 8 else status}: {msg}")


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load the in-tree shared library (optionally building it first)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"{path} is missing: run newton_schulz_04_gb300.build.build() first")
        _build.build()
    lib = ctypes.CDLL(path)
    vp, sz, i32, i64, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    fptr = ctypes.POINTER(ctypes.c_float)
    lib.muon_ns_batched.argtypes = [vp, i32, i32, i32, i32, fptr, vp, i32, i32, vp, sz, vp]
    lib.muon_ns_batched.restype = i32
    lib.muon_step.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i64), i32,
                              f32, f32, i32, fptr, i32, i32, vp, sz, vp]
    lib.muon_step.restype = i32
    lib.muon_workspace_bytes.argtypes = [ctypes.POINTER(i64), i32, i32, i32, i32]
    lib.muon_workspace_bytes.restype = sz
    lib.muon_resolve_schedule.argtypes = [i64, i64, i32, i32, i32]
    lib.muon_resolve_schedule.restype = i32
    lib.muon_bucket_plan.argtypes = [ctypes.POINTER(i64), i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.muon_bucket_plan.restype = i32
    lib.muon_device_status.argtypes = [vp, vp]
    lib.muon_device_status.restype = i32
    lib.muon_debug_bounded_wait.argtypes = [vp, ctypes.c_longlong, vp]
    lib.muon_debug_bounded_wait.restype = i32
    lib.muon_debug_gemm.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, sz, vp]
    lib.muon_debug_gemm.restype = i32
    lib.muon_profile_enable.argtypes = [i32]
    lib.muon_profile_enable.restype = None
    lib.muon_profile_count.argtypes = []
    lib.muon_profile_count.restype = i32
    lib.muon_profile_get.argtypes = [i32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float),
                                     ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
    lib.muon_profile_get.restype = i32
    lib.muon_ns_batched_static.argtypes = [vp, i32, i32, i32, i32, fptr, vp, i32, i32, vp]
    lib.muon_ns_batched_static.restype = i32
    lib.muon_static_scratch_bytes.argtypes = []
    lib.muon_static_scratch_bytes.restype = sz
    lib.muon_static_status.argtypes = [vp]
    lib.muon_static_status.restype = i32
    lib.muon_debug_bounded_wait_static.argtypes = [ctypes.c_longlong, vp]
    lib.muon_debug_bounded_wait_static.restype = i32
    lib.muon_adamw_tail.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                                    ctypes.POINTER(i64), i32, f32, f32, f32, f32, f32, i32, i32, vp]
    lib.muon_adamw_tail.restype = i32
    lib.muon_cost_estimate.argtypes = [ctypes.POINTER(i64), i32, i32, i32, i32, ctypes.POINTER(ctypes.c_double)]
    lib.muon_cost_estimate.restype = i32
    lib.muon_partition.argtypes = [ctypes.POINTER(ctypes.c_double), i32, i32, i32, ctypes.POINTER(i32),
                                   ctypes.POINTER(ctypes.c_double)]
    lib.muon_partition.restype = i32
    lib.muon_last_error.argtypes = []
    lib.muon_last_error.restype = ctypes.c_char_p
    lib.muon_version.argtypes = []
    lib.muon_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int):
    if status != OK:
        raise MuonError(status, load().muon_last_error().decode())


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return BF16
    if dt == torch.float32:
        return FP32
    raise TypeError(f"unsupported dtype {dt}: bfloat16 or float32")


def _shapes_arr(shapes):
    flat = [int(v) for mn in shapes for v in mn]
    return (ctypes.c_int64 * max(len(flat), 1))(*flat)


def _coeffs(coeffs):
    if coeffs is None:
        return None
    return (ctypes.c_float * 3)(*[float(c) for c in coeffs])


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def workspace_bytes(shapes, steps=5, dtype=torch.bfloat16, schedule="auto") -> int:
    lib = load()
    n = lib.muon_workspace_bytes(_shapes_arr(shapes), len(shapes), int(steps), _dtype_code(dtype), sched_code(schedule))
    if n == 0:
        raise MuonError(ERR_ARG, lib.muon_last_error().decode())
    return int(n)


def resolve_schedule(m, n, steps=5, dtype=torch.bfloat16, schedule="auto") -> str:
    return SCHED_NAMES[load().muon_resolve_schedule(int(m), int(n), int(steps), _dtype_code(dtype),
                                                    sched_code(schedule))]


def bucket_plan(shapes):
    """(order, group_start) exactly as the library groups the matrices."""
    lib = load()
    n = len(shapes)
    order = (ctypes.c_int * max(n, 1))()
    start = (ctypes.c_int * (n + 1))()
    g = lib.muon_bucket_plan(_shapes_arr(shapes), n, order, start)
    if g < 0:
        raise MuonError(ERR_ARG, "bad shapes")
    return list(order[:n]), list(start[:g + 1])


def adamw_tail(params, grads, exp_avgs, exp_avg_sqs, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01,
               step=1, stream=None) -> None:
    """In place: one AdamW step over a list of tensors of any shape (C-ABI
    muon_adamw_tail).  params / grads share one dtype (bfloat16 or float32);
    the moments are float32 tensors of the same sizes."""
    lib = load()
    count = len(params)
    if not (len(grads) == count == len(exp_avgs) == len(exp_avg_sqs)):
        raise ValueError("params, grads and both moment lists must have the same length")
    if count == 0:
        return
    dtype = params[0].dtype
    for p, g, m, v in zip(params, grads, exp_avgs, exp_avg_sqs):
        if p.dtype != dtype or g.dtype != dtype or m.dtype != torch.float32 or v.dtype != torch.float32:
            raise TypeError("params and grads share one dtype; moments are float32")
        if not (p.numel() == g.numel() == m.numel() == v.numel()):
            raise ValueError("each param, grad and moment must have the same number of elements")
        if not (p.is_contiguous() and g.is_contiguous() and m.is_contiguous() and v.is_contiguous()):
            raise ValueError("tensors must be contiguous")
    P = ctypes.c_void_p * count
    n = (ctypes.c_int64 * count)(*[p.numel() for p in params])
    _check(lib.muon_adamw_tail(P(*[p.data_ptr() for p in params]), P(*[g.data_ptr() for g in grads]),
                               P(*[m.data_ptr() for m in exp_avgs]), P(*[v.data_ptr() for v in exp_avg_sqs]), n,
                               count, float(lr), float(betas[0]), float(betas[1]), float(eps), float(weight_decay),
                               int(step), _dtype_code(dtype), ctypes.c_void_p(_stream_ptr(stream))))


class AdamwTail:
    """AdamW over a fixed list of tensors (the non-matrix tail), with the
    pointer tables built once and the step count kept here; `step()` is one
    C-ABI call (one launch per 512 tensors)."""

    def __init__(self, params, grads, exp_avgs, exp_avg_sqs, lr=1e-3, betas=(0.9, 0.999), eps=1e-8,
                 weight_decay=0.01):
        lib = load()
        self._lib = lib
        self.count = len(params)
        if not (len(grads) == self.count == len(exp_avgs) == len(exp_avg_sqs)):
            raise ValueError("params, grads and both moment lists must have the same length")
        dtype = params[0].dtype if self.count else torch.float32
        for p, g, m, v in zip(params, grads, exp_avgs, exp_avg_sqs):
            if p.dtype != dtype or g.dtype != dtype or m.dtype != torch.float32 or v.dtype != torch.float32:
                raise TypeError("params and grads share one dtype; moments are float32")
            if not (p.numel() == g.numel() == m.numel() == v.numel()):
                raise ValueError("each param, grad and moment must have the same number of elements")
            if not (p.is_contiguous() and g.is_contiguous() and m.is_contiguous() and v.is_contiguous()):
                raise ValueError("tensors must be contiguous")
        self._keep = (list(params), list(grads), list(exp_avgs), list(exp_avg_sqs))
        P = ctypes.c_void_p * max(self.count, 1)
        self._p = P(*[t.data_ptr() for t in params])
        self._g = P(*[t.data_ptr() for t in grads])
        self._m = P(*[t.data_ptr() for t in exp_avgs])
        self._v = P(*[t.data_ptr() for t in exp_avg_sqs])
        self._n = (ctypes.c_int64 * max(self.count, 1))(*[t.numel() for t in params])
        self._dt = _dtype_code(dtype) if self.count else FP32
        self.lr, self.betas, self.eps, self.weight_decay = lr, betas, eps, weight_decay
        self.t = 0

    def step(self, stream=None) -> None:
        self.t += 1
        _check(self._lib.muon_adamw_tail(self._p, self._g, self._m, self._v, self._n, self.count, float(self.lr),
                                         float(self.betas[0]), float(self.betas[1]), float(self.eps),
                                         float(self.weight_decay), self.t, self._dt,
                                         ctypes.c_void_p(_stream_ptr(stream))))


def cost_estimate(shapes, steps=5, dtype=torch.bfloat16, schedule="auto") -> list:
    """Predicted device seconds of each matrix's update (the library's cost model)."""
    lib = load()
    n = len(shapes)
    out = (ctypes.c_double * max(n, 1))()
    _check(lib.muon_cost_estimate(_shapes_arr(shapes), n, int(steps), _dtype_code(dtype), sched_code(schedule), out))
    return list(out[:n])


PARTITION_EXACT_MAX = 24


def partition(costs, world: int, exact_limit: int = 12):
    """(owner per matrix, total cost per owner): greedy LPT, solved exactly when
    len(costs) <= exact_limit.  Same answer on every rank for the same costs."""
    lib = load()
    n = len(costs)
    c = (ctypes.c_double * max(n, 1))(*[float(x) for x in costs])
    owner = (ctypes.c_int32 * max(n, 1))()
    load_ = (ctypes.c_double * max(int(world), 1))()
    _check(lib.muon_partition(c, n, int(world), int(exact_limit), owner, load_))
    return list(owner[:n]), list(load_[:int(world)])


def measure_costs(shapes, steps=5, dtype=torch.bfloat16, schedule="auto", repeats=3, cache=None, device=None):
    """Measured device seconds per matrix, per shape group, for placement.

    Each distinct (short, long) group of `shapes` runs muon_step on synthetic
    data at its real batch width; the time per call (CUDA events, after one
    warm-up) divided by the width is that group's per-matrix cost.  `cache`
    (a dict, e.g. loaded from and saved to JSON by the caller) keeps results
    keyed by "s,l,dtype,steps,schedule,width" across calls.
    """
    dev = device or torch.device("cuda")
    groups = {}
    for i, (m, n) in enumerate(shapes):
        groups.setdefault((min(m, n), max(m, n)), []).append(i)
    out = [0.0] * len(shapes)
    gen = torch.Generator(device="cpu").manual_seed(0)
    for (s_, l_), idx in sorted(groups.items()):
        key = f"{s_},{l_},{str(dtype).split('.')[-1]},{steps},{schedule},{len(idx)}"
        if cache is not None and key in cache:
            per = float(cache[key])
        else:
            W = [torch.zeros(s_, l_, dtype=dtype, device=dev) for _ in idx]
            G = [torch.randn(s_, l_, generator=gen).to(dtype).to(dev) for _ in idx]
            M = [torch.zeros(s_, l_, dtype=torch.float32, device=dev) for _ in idx]
            ws = new_workspace(workspace_bytes([(s_, l_)] * len(idx), steps, dtype, schedule), dev)
            muon_step(W, G, M, 0.0, 0.0, steps, None, schedule, ws)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(repeats):
                muon_step(W, G, M, 0.0, 0.0, steps, None, schedule, ws)
            b.record()
            b.synchronize()
            per = a.elapsed_time(b) / 1e3 / repeats / len(idx)
            del W, G, M, ws
            if cache is not None:
                cache[key] = per
        for i in idx:
            out[i] = per
    return out


def schedule_candidates(dtype=torch.bfloat16, steps=5):
    """What a measured choice may pick from: schedules whose accuracy meets
    the dtype's tolerance on every input kind measured (bf16: original space,
    or the Gram recurrence restarted every two steps, and past 10 steps the
    fp16-pair schedule; fp32: the tensor-core fp16-pair schedule up to 6
    steps, FFMA restarted Gram or original space), each tensor-core one with
    shared or separate launches."""
    if dtype == torch.bfloat16:
        if steps > 10:
            base = ["orig_f16x3"]
        else:
            base = ["orig", "gram_r2"] if steps >= 3 else ["orig"]
        return [f"{b}+{mode}" for b in base for mode in ("shared", "separate")]
    if steps <= 6:
        return ["orig_f16x3+shared", "orig_f16x3+separate", "orig", "gram_r2"]
    return ["gram_r2", "orig"]


def tune_schedules(shapes, steps=5, dtype=torch.bfloat16, candidates=None, repeats=3, cache=None, device=None):
    """Measured schedule choice per shape group.

    For each distinct (short, long) group of `shapes`, at its real batch width,
    every candidate schedule (schedule_candidates by default) runs muon_step on
    one set of synthetic tensors drawn on the device (one warm-up call, then
    `repeats` calls timed with CUDA events), and the fastest wins.  Returns
    {(s, l): schedule}.  `cache` (a dict, e.g. loaded from and saved to JSON by
    the caller) keeps, per key "s,l,dtype,steps,width", the chosen schedule and
    every candidate's milliseconds, so later calls measure nothing.
    """
    dev = device or torch.device("cuda")
    cands = list(candidates or schedule_candidates(dtype, steps))
    groups = {}
    for (m, n) in shapes:
        key = (min(m, n), max(m, n))
        groups[key] = groups.get(key, 0) + 1
    out = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    for (s_, l_), width in sorted(groups.items()):
        key = f"{s_},{l_},{str(dtype).split('.')[-1]},{steps},{width}"
        if cache is not None and key in cache:
            out[(s_, l_)] = cache[key]["best"]
            continue
        W = [torch.zeros(s_, l_, dtype=dtype, device=dev) for _ in range(width)]
        G = [torch.randn(s_, l_, generator=gen, device=dev).to(dtype) for _ in range(width)]
        M = [torch.zeros(s_, l_, dtype=torch.float32, device=dev) for _ in range(width)]
        ws = new_workspace(max(workspace_bytes([(s_, l_)] * width, steps, dtype, sc) for sc in cands), dev)
        ms = {}
        for sc in cands:
            muon_step(W, G, M, 0.0, 0.0, steps, None, sc, ws)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(repeats):
                muon_step(W, G, M, 0.0, 0.0, steps, None, sc, ws)
            b.record()
            b.synchronize()
            ms[sc] = a.elapsed_time(b) / repeats
        del W, G, M, ws
        entry = {"best": min(ms, key=ms.get), "ms": ms}
        if cache is not None:
            cache[key] = entry
        out[(s_, l_)] = entry["best"]
    return out


def owned(shapes, rank: int, world: int, costs=None, steps=5, dtype=torch.bfloat16, schedule="auto",
          exact_limit: int = 12):
    """Indices of the matrices `rank` owns out of `world` owners (model costs
    unless measured `costs` are given)."""
    if costs is None:
        costs = cost_estimate(shapes, steps, dtype, schedule)
    owner, _ = partition(costs, world, exact_limit)
    return [i for i, r in enumerate(owner) if r == rank]


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """Caller-owned workspace (uint8, 256-byte aligned, status word zeroed)."""
    ws = torch.empty(int(nbytes) + WS_ALIGN, dtype=torch.uint8, device=device or "cuda")
    off = (-ws.data_ptr()) % WS_ALIGN
    ws = ws[off:off + int(nbytes)]
    ws[:16].zero_()
    return ws


def ns_batched(X: torch.Tensor, steps: int = 5, coeffs=None, schedule: str = "auto", out=None,
               workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """O_i = NS(X_i) for a [B, m, n] bf16/fp32 CUDA tensor (C-ABI muon_ns_batched)."""
    lib = load()
    if X.dim() != 3 or not X.is_cuda or not X.is_contiguous():
        raise ValueError("X must be a contiguous [B, m, n] CUDA tensor")
    B, m, n = X.shape
    dt = _dtype_code(X.dtype)
    if out is None:
        out = torch.empty_like(X)
    if workspace is None:
        workspace = new_workspace(workspace_bytes([(m, n)] * max(B, 1), steps, X.dtype, schedule), X.device)
    st = lib.muon_ns_batched(ctypes.c_void_p(X.data_ptr()), B, m, n, int(steps), _coeffs(coeffs),
                             ctypes.c_void_p(out.data_ptr()), dt, sched_code(schedule),
                             ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                             ctypes.c_void_p(_stream_ptr(stream)))
    _check(st)
    return out


def ns_batched_static(X: torch.Tensor, steps: int = 5, coeffs=None, schedule: str = "auto", out=None,
                      stream=None) -> torch.Tensor:
    """As ns_batched, through the entry point that allocates nothing (the
    library's fixed device scratch; see muon_ns_batched_static)."""
    lib = load()
    if X.dim() != 3 or not X.is_cuda or not X.is_contiguous():
        raise ValueError("X must be a contiguous [B, m, n] CUDA tensor")
    B, m, n = X.shape
    if out is None:
        out = torch.empty_like(X)
    _check(lib.muon_ns_batched_static(ctypes.c_void_p(X.data_ptr()), B, m, n, int(steps), _coeffs(coeffs),
                                      ctypes.c_void_p(out.data_ptr()), _dtype_code(X.dtype), sched_code(schedule),
                                      ctypes.c_void_p(_stream_ptr(stream))))
    return out


def static_status(stream=None) -> int:
    """Synchronise and read/clear the status word of the static scratch that
    ns_batched_static runs in (OK or ERR_TIMEOUT)."""
    return load().muon_static_status(ctypes.c_void_p(_stream_ptr(stream)))


def debug_bounded_wait_static(max_cycles: int, stream=None) -> None:
    _check(load().muon_debug_bounded_wait_static(int(max_cycles), ctypes.c_void_p(_stream_ptr(stream))))


def muon_step(weights: Sequence[torch.Tensor], grads: Sequence[torch.Tensor], moms: Sequence[torch.Tensor],
              beta: float = 0.95, lr: float = 0.02, steps: int = 5, coeffs=None, schedule: str = "auto",
              workspace: torch.Tensor | None = None, stream=None) -> None:
    """In place: mom <- beta mom + grad; W <- W - lr NS(mom) (C-ABI muon_step)."""
    lib = load()
    count = len(weights)
    if not (len(grads) == count == len(moms)):
        raise ValueError("weights, grads and moms must have the same length")
    if count == 0:
        return
    dtype = weights[0].dtype
    for w, g, mo in zip(weights, grads, moms):
        if w.dim() != 2 or w.shape != g.shape or w.shape != mo.shape:
            raise ValueError("each weight, grad and momentum must be 2-D of one shape")
        if w.dtype != dtype or g.dtype != dtype or mo.dtype != torch.float32:
            raise TypeError("weights and grads share one dtype; momentum is float32")
        if not (w.is_contiguous() and g.is_contiguous() and mo.is_contiguous()):
            raise ValueError("tensors must be contiguous")
    shapes = [tuple(w.shape) for w in weights]
    if workspace is None:
        workspace = new_workspace(workspace_bytes(shapes, steps, dtype, schedule), weights[0].device)
    P = ctypes.c_void_p * count
    st = lib.muon_step(P(*[w.data_ptr() for w in weights]), P(*[g.data_ptr() for g in grads]),
                       P(*[m.data_ptr() for m in moms]), _shapes_arr(shapes), count, float(beta), float(lr),
                       int(steps), _coeffs(coeffs), _dtype_code(dtype), sched_code(schedule),
                       ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                       ctypes.c_void_p(_stream_ptr(stream)))
    _check(st)


def device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise and read/clear the workspace status word (OK or ERR_TIMEOUT)."""
    return load().muon_device_status(ctypes.c_void_p(workspace.data_ptr()), ctypes.c_void_p(_stream_ptr(stream)))


def debug_bounded_wait(workspace: torch.Tensor, max_cycles: int, stream=None) -> None:
    _check(load().muon_debug_bounded_wait(ctypes.c_void_p(workspace.data_ptr()), int(max_cycles),
                                          ctypes.c_void_p(_stream_ptr(stream))))


def debug_gemm(A, B, A_lo=None, B_lo=None, split=1, b_mn=False, sym=False, a_sym=False, b_sym=False,
               workspace=None, stream=None):
    """Test hook: out[b] = A[b] @ (B[b] if b_mn else B[b]^T) through one library kernel.

    bf16 (or fp16) operands run the tensor-core kernel and return the fp32
    value of the bf16 (fp16) head/residual pair it writes (with sym, only the
    256 x 256 blocks on or below the diagonal are written); a_sym / b_sym
    declare operands given in that block-lower storage.  split=4 (fp16,
    b_mn, square A) adds B_lo / 2^11 through the diagonal K segment; split=5
    (fp16) multiplies the pairs A + A_lo / 2^11 and B + B_lo / 2^11 (the low
    parts stored scaled by 2^11).  fp32 operands run the FFMA kernel."""
    lib = load()
    batch, M, K = A.shape
    N = B.shape[2] if b_mn else B.shape[1]
    if workspace is None:
        workspace = new_workspace(1024 + 131072 if split == 4 else 4096, A.device)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    if A.dtype == torch.float32:
        out = torch.zeros(batch, M, N, dtype=torch.float32, device=A.device)
        lo = None
    else:
        out = torch.zeros(batch, M, N, dtype=A.dtype, device=A.device)
        lo = torch.zeros_like(out)
    flags = int(sym) | (int(a_sym) << 1) | (int(b_sym) << 2)
    code = FP16 if A.dtype == torch.float16 else _dtype_code(A.dtype)
    _check(lib.muon_debug_gemm(ptr(A), ptr(A_lo), ptr(B), ptr(B_lo), batch, M, N, K, split, int(b_mn), flags,
                               code, ptr(out), ptr(lo), ptr(workspace), workspace.numel(),
                               ctypes.c_void_p(_stream_ptr(stream))))
    if lo is None:
        return out
    if A.dtype == torch.float16:
        return out.float() + lo.float() / F16_LO_SCALE
    return out.float() + lo.float()


def profile_enable(on: bool = True) -> None:
    """Start (clearing old records) or stop per-launch CUDA-event timing."""
    load().muon_profile_enable(1 if on else 0)


def profile_records():
    """[(kind, ms, flops, bytes)] for every launch recorded since profile_enable(True)."""
    lib = load()
    out = []
    for i in range(lib.muon_profile_count()):
        k, ms, fl, by = ctypes.c_char_p(), ctypes.c_float(), ctypes.c_double(), ctypes.c_double()
        _check(lib.muon_profile_get(i, ctypes.byref(k), ctypes.byref(ms), ctypes.byref(fl), ctypes.byref(by)))
        out.append((k.value.decode(), ms.value, fl.value, by.value))
    return out


class MuonUpdater:
    """Owner-side Muon step over a fixed list of 2-D parameters.

    Holds the fp32 momentum buffers and one caller-side workspace sized for the
    parameter shapes.  `step(grads)` makes one C-ABI call per shape group (the
    library's bucket grouping); the groups are independent, so their order
    does not change any result.  `group_order="largest_first"` runs the groups
    with the most parameter bytes first, which lets a caller that copies each
    group's weights out (the `after_group` hook of `step`) overlap those copies
    with the groups that follow.  With `schedule="tuned"` each group runs the
    schedule that measured fastest for it (tune_schedules, at construction;
    `tune_cache` is passed through).  With `use_graph=True` the first step
    with a given set of gradient tensors runs eagerly and is captured, one
    CUDA graph per group; later steps with the same tensors replay them.
    Graphs are kept for up to `max_graphs` sets of gradient tensors (e.g. two
    buffers that alternate while the next step's gradients are copied in).
    """

    def __init__(self, params: Sequence[torch.Tensor], beta=0.95, lr=0.02, steps=5, coeffs=None,
                 schedule="auto", workspace_limit: int | None = None, use_graph: bool = False, max_graphs: int = 4,
                 tune_cache=None, group_order: str = "library"):
        if group_order not in ("library", "largest_first"):
            raise ValueError("group_order is 'library' or 'largest_first'")
        self.params = list(params)
        self.beta, self.lr, self.steps, self.coeffs, self.schedule = beta, lr, steps, coeffs, schedule
        self.moms = [torch.zeros(p.shape, dtype=torch.float32, device=p.device) for p in self.params]
        shapes = [tuple(p.shape) for p in self.params]
        dtype = self.params[0].dtype
        if schedule == "tuned":
            self.chosen = tune_schedules(shapes, steps, dtype, cache=tune_cache, device=self.params[0].device)
        else:
            self.chosen = {(min(sh), max(sh)): resolve_schedule(sh[0], sh[1], steps, dtype, schedule) for sh in shapes}
        order, start = bucket_plan(shapes)
        self._groups = []
        for k in range(len(start) - 1):
            idx = order[start[k]:start[k + 1]]
            s_, l_ = min(shapes[idx[0]]), max(shapes[idx[0]])
            self._groups.append((idx, self.chosen[(s_, l_)] if schedule == "tuned" else schedule))
        if group_order == "largest_first":
            nbytes = [sum(self.params[i].numel() * self.params[i].element_size() for i in idx) for idx, _ in self._groups]
            self._groups = [g for _, g in sorted(zip(nbytes, self._groups), key=lambda t: -t[0])]
        need = max((workspace_bytes([shapes[i] for i in idx], steps, dtype, sc) for idx, sc in self._groups), default=0)
        if workspace_limit is not None:
            need = min(need, int(workspace_limit))
        self.workspace = new_workspace(need, self.params[0].device)
        self.use_graph = use_graph
        self.max_graphs = max_graphs
        self._graphs = {}  # tuple of gradient data pointers -> one CUDAGraph per group

    @property
    def groups(self):
        """The shape groups in the order `step` runs them: (parameter indices, schedule)."""
        return [(list(idx), sc) for idx, sc in self._groups]

    def _run_group(self, gi, grads, stream):
        idx, sc = self._groups[gi]
        muon_step([self.params[i] for i in idx], [grads[i] for i in idx], [self.moms[i] for i in idx], self.beta,
                  self.lr, self.steps, self.coeffs, sc, self.workspace, stream)

    def _eager(self, grads, stream=None, before_group=None, after_group=None):
        st = stream if stream is not None else torch.cuda.current_stream()
        for gi, (idx, _) in enumerate(self._groups):
            if before_group is not None:
                before_group(gi, idx, st)
            self._run_group(gi, grads, st)
            if after_group is not None:
                after_group(gi, idx, st)

    def step(self, grads: Sequence[torch.Tensor], stream=None, before_group=None, after_group=None):
        """One step on `stream` (the current stream if None).

        `before_group(gi, indices, stream)` and `after_group(gi, indices,
        stream)`, if given, are called on the host just before and just after
        group `gi`'s work is enqueued on the stream, e.g. to make the stream
        wait for an earlier copy of those weights, or to record an event and
        start copying them out."""
        if not self.use_graph:
            self._eager(grads, stream, before_group, after_group)
            return
        key = tuple(g.data_ptr() for g in grads)
        graphs = self._graphs.get(key)
        if graphs is not None:
            st = stream if stream is not None else torch.cuda.current_stream()
            with torch.cuda.stream(st):
                for gi, (idx, _) in enumerate(self._groups):
                    if before_group is not None:
                        before_group(gi, idx, st)
                    graphs[gi].replay()
                    if after_group is not None:
                        after_group(gi, idx, st)
            return
        # this call's update runs eagerly (and sets up per-device state); the same
        # launch sequence is then captured, group by group, for the following calls
        self._eager(grads, stream, before_group, after_group)
        (stream if stream is not None else torch.cuda.current_stream()).synchronize()
        graphs = []
        side = torch.cuda.Stream()
        for gi in range(len(self._groups)):
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                self._run_group(gi, grads, side)
            graphs.append(graph)
        if len(self._graphs) >= self.max_graphs:
            self._graphs.pop(next(iter(self._graphs)))
        self._graphs[key] = graphs
