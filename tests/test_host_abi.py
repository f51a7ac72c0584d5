"""Host-side tests of the C ABI: the library loads on a CPU-only host, exports
every entry point the header declares, validates arguments before touching
the GPU, and groups matrices exactly like the reference grouping."""
import ctypes
import os
import re

import pytest
import torch

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from newton_schulz_04_gb300 import build as b
    b.build()
    import newton_schulz_04_gb300 as m
    return m.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "muon_ns.h")).read()
    return sorted(set(re.findall(r"MUON_API\s+[\w\s\*]*?\b(muon_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    syms = declared_symbols()
    for s in ["muon_ns_batched", "muon_step", "muon_workspace_bytes", "muon_last_error", "muon_device_status"]:
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    for s in declared_symbols():
        assert hasattr(lib, s), s
        assert ctypes.cast(getattr(lib, s), ctypes.c_void_p).value


def test_bucket_plan_matches_reference_grouping(lib):
    import newton_schulz_04_gb300 as m
    g = torch.Generator().manual_seed(0)
    for trial in range(50):
        n = int(torch.randint(1, 40, (1,), generator=g))
        dims = [64, 128, 200, 256]
        shapes = [(dims[int(torch.randint(0, 4, (1,), generator=g))], dims[int(torch.randint(0, 4, (1,), generator=g))])
                  for _ in range(n)]
        order, start = m.bucket_plan(shapes)
        ref = oracle.bucket_order(shapes)
        got = [((min(shapes[order[start[k]]]), max(shapes[order[start[k]]])), order[start[k]:start[k + 1]])
               for k in range(len(start) - 1)]
        assert got == ref


def test_bucket_plan_llama_shapes(lib):
    import newton_schulz_04_gb300 as m
    shapes = synth.c3_shapes()
    order, start = m.bucket_plan(shapes)
    assert start == [0, 128, 224]
    assert order[:4] == [0, 1, 2, 3]
    assert sorted(order) == list(range(len(shapes)))


def test_schedule_choice(lib):
    import newton_schulz_04_gb300 as m
    # bf16 AUTO runs the Gram recurrence restarted every two steps where it
    # executes at most 0.9x ORIG's tensor-core work, else original space;
    # fp32 AUTO takes Gram space whenever l > s, where it never costs more
    for shp in [(1024, 1024), (4096, 4096), (1000, 1100), (1024, 1280)]:
        assert m.resolve_schedule(*shp) == "orig", shp
    for shp in [(1024, 4096), (1024, 8192), (16384, 1024), (4096, 14336), (256, 1024), (1024, 2048)]:
        assert m.resolve_schedule(*shp) == "gram_r2", shp
    assert m.resolve_schedule(4096, 14336, steps=2) == "orig"  # no two-step segment to run
    assert m.resolve_schedule(4096, 14336, steps=3) == "gram_r2"
    assert m.resolve_schedule(1024, 8192, steps=0) == "orig"
    # bf16 past 10 steps: fp16 pairs, whatever the shape
    for shp in [(1024, 1024), (4096, 14336), (256, 1024)]:
        assert m.resolve_schedule(*shp, steps=10) != "orig_f16x3", shp
        assert m.resolve_schedule(*shp, steps=11) == "orig_f16x3", shp
        assert m.resolve_schedule(*shp, steps=100) == "orig_f16x3", shp
    assert m.resolve_schedule(1024, 1024, steps=20, schedule="orig") == "orig"
    assert m.schedule_candidates(torch.bfloat16, 20) == ["orig_f16x3+shared", "orig_f16x3+separate"]
    assert m.resolve_schedule(1024, 8192, schedule="gram_x1") == "gram_x1"
    assert m.resolve_schedule(128, 256, dtype=torch.float32) == "orig_f16x3"
    assert m.resolve_schedule(128, 128, dtype=torch.float32) == "orig_f16x3"
    assert m.resolve_schedule(128, 256, dtype=torch.float32, schedule="gram_x3") == "gram_x3"
    assert m.resolve_schedule(128, 128, dtype=torch.float32, schedule="orig") == "orig"
    assert m.resolve_schedule(128, 128, dtype=torch.float32, schedule="gram_r2") == "gram_r2"  # FFMA segments
    assert m.resolve_schedule(128, 256, dtype=torch.float32, schedule="orig_f16x3") == "orig_f16x3"
    assert m.resolve_schedule(128, 256, schedule="orig_f16x3") == "orig_f16x3"
    # fp32 beyond 6 steps: Gram space only in restarted segments
    assert m.resolve_schedule(1024, 2048, steps=6, dtype=torch.float32) == "orig_f16x3"
    assert m.resolve_schedule(1024, 2048, steps=10, dtype=torch.float32) == "gram_r2"
    assert m.resolve_schedule(1024, 1100, steps=10, dtype=torch.float32) == "orig"
    assert m.resolve_schedule(1024, 2048, steps=10, dtype=torch.float32, schedule="gram_r2") == "gram_r2"


def test_launch_mode_flags(lib):
    import newton_schulz_04_gb300 as m
    assert m.sched_code("gram_r2+shared") == 6 | 0x100
    assert m.sched_code("orig+separate") == 3 | 0x200
    assert m.resolve_schedule(4096, 14336, schedule="orig+separate") == "orig"
    assert m.workspace_bytes([(512, 2048)] * 3, schedule="gram_r2+shared") == m.workspace_bytes([(512, 2048)] * 3)
    big = 1 << 40
    # both flags at once, or an unknown flag, are argument errors
    assert _ns_call(lib, X=big, out=2 * big, sc=6 | 0x300) == 1
    assert _ns_call(lib, X=big, out=2 * big, sc=6 | 0x400) == 1
    with pytest.raises(ValueError):
        m.sched_code("orig+sideways")


def test_gram_r2_work_against_orig(lib):
    """The segment plan's tensor-core work as AUTO counts it: per segment of k
    steps S^2 L (SYRK) + (4k - 3) S^3 + 2 S^2 L; ORIG is k = 1 throughout."""
    def work(plan, S, L):
        return sum(3 * S * S * L + (4 * k - 3) * S ** 3 for k in plan)
    S, L = 4096, 14336
    assert work([1, 2, 2], S, L) / work([1] * 5, S, L) < 0.75  # the c3 rectangular bucket: 26 % less
    assert work([1, 2, 2], S, S) == work([1] * 5, S, S)          # square: the same


def test_workspace_sizes(lib):
    import newton_schulz_04_gb300 as m
    one = m.workspace_bytes([(1024, 1024)])
    many = m.workspace_bytes([(1024, 1024)] * 16)
    assert many > one
    # ORIG bf16 per matrix: two bf16 X pairs + bf16 A pair + bf16 B pair
    assert many >= 16 * 1024 * 1024 * (8 + 4 + 4)
    assert m.workspace_bytes([(1024, 1024)] * 300) == m.workspace_bytes([(1024, 1024)] * 256)


def _ns_call(lib, X=1, B=1, m=8, n=8, steps=5, out=2, dt=0, sc=0, ws=256, wsb=1 << 20, coeffs=None):
    return lib.muon_ns_batched(ctypes.c_void_p(X), B, m, n, steps, coeffs, ctypes.c_void_p(out), dt, sc,
                               ctypes.c_void_p(ws), wsb, None)


def test_argument_errors_before_any_launch(lib):
    E = {"arg": 1, "shape": 2, "align": 3, "ws": 4}
    big = 1 << 40
    assert _ns_call(lib, X=0, out=big) == E["arg"]
    assert _ns_call(lib, B=-1) == E["arg"]
    assert _ns_call(lib, X=big, out=2 * big, m=0) == E["shape"]
    assert _ns_call(lib, X=big, out=2 * big, n=70000) == E["shape"]
    assert _ns_call(lib, X=big, out=2 * big, steps=-1) == E["arg"]
    assert _ns_call(lib, X=big, out=2 * big, steps=1000) == E["arg"]
    assert _ns_call(lib, X=big, out=2 * big, dt=7) == E["arg"]
    assert _ns_call(lib, X=big, out=2 * big, sc=9) == E["arg"]
    assert _ns_call(lib, X=big, out=2 * big, ws=0) == E["arg"]
    assert _ns_call(lib, X=big, out=2 * big, ws=big + 8 * 1024 * 1024 + 3) == E["align"]
    assert _ns_call(lib, X=big + 1, out=2 * big) == E["align"]
    assert _ns_call(lib, X=big, out=big + 64) == E["arg"]  # overlap
    nan = (ctypes.c_float * 3)(float("nan"), 0.0, 0.0)
    assert _ns_call(lib, X=big, out=2 * big, coeffs=nan) == E["arg"]
    # workspace too small for one 4096 x 4096 matrix
    assert _ns_call(lib, X=big, out=2 * big, m=4096, n=4096, ws=4 * big, wsb=1 << 20) == E["ws"]
    assert "workspace" in lib.muon_last_error().decode()


def test_step_argument_errors(lib):
    P = ctypes.c_void_p * 2
    shapes = (ctypes.c_int64 * 4)(8, 8, 8, 8)
    big = 1 << 40
    W = P(big, big + (1 << 20))
    G = P(2 * big, 2 * big + (1 << 20))
    Mm = P(3 * big, 3 * big + (1 << 20))
    ws = ctypes.c_void_p(4 * big)
    if not torch.cuda.is_available():
        # Every argument is valid (the pointers are fake), so this call gets as far
        # as the first CUDA call, which fails cleanly on a host without a GPU.  It
        # is never made where a GPU exists: there it would launch on fake pointers.
        st = lib.muon_step(W, G, Mm, shapes, 2, 0.95, 0.02, 5, None, 0, 0, ws, 1 << 26, None)
        assert st == 5
    bad = P(big, 0)
    assert lib.muon_step(bad, G, Mm, shapes, 2, 0.95, 0.02, 5, None, 0, 0, ws, 1 << 20, None) == 1
    assert lib.muon_step(W, G, Mm, shapes, -1, 0.95, 0.02, 5, None, 0, 0, ws, 1 << 20, None) == 1
    assert lib.muon_step(W, G, Mm, shapes, 2, float("inf"), 0.02, 5, None, 0, 0, ws, 1 << 20, None) == 1
    Wo = P(3 * big, big + (1 << 20))  # W[0] aliases mom[0]
    assert lib.muon_step(Wo, G, Mm, shapes, 2, 0.95, 0.02, 5, None, 0, 0, ws, 1 << 20, None) == 1
    shp_bad = (ctypes.c_int64 * 4)(8, -8, 8, 8)
    assert lib.muon_step(W, G, Mm, shp_bad, 2, 0.95, 0.02, 5, None, 0, 0, ws, 1 << 20, None) == 2


def test_empty_batch_is_a_noop(lib):
    assert _ns_call(lib, X=1 << 40, B=0, out=1 << 41, ws=1 << 42) == 0


def _gemm_call(lib, split=4, dt=2, b_mn=1, M=256, N=256, K=256, B_lo=True, wsb=1024 + 131072, sym=0):
    big = 1 << 40
    p = ctypes.c_void_p
    return lib.muon_debug_gemm(p(big), None, p(2 * big), p(3 * big) if B_lo else None, 1, M, N, K, split, b_mn, sym,
                               dt, p(5 * big), None, p(6 * big), wsb, None)


def test_debug_gemm_diagonal_segment_argument_errors(lib):
    # every case is refused on the host, before any CUDA call
    E = {"arg": 1, "shape": 2, "ws": 4}
    assert _gemm_call(lib, dt=0) == E["arg"]             # bf16: the segment is fp16 only
    assert _gemm_call(lib, B_lo=False) == E["arg"]       # needs B's low part
    assert _gemm_call(lib, b_mn=0) == E["arg"]           # needs an MN-major B
    assert _gemm_call(lib, K=512) == E["arg"]            # D is square: K must equal M
    assert _gemm_call(lib, sym=1) == E["arg"]            # full outputs only
    assert _gemm_call(lib, wsb=1024 + 1000) == E["ws"]   # room for the diagonal table
    assert "workspace" in lib.muon_last_error().decode()
    assert _gemm_call(lib, split=5) == E["arg"]
    assert _gemm_call(lib, M=200, K=200) == E["shape"]   # tiles pair 256 rows


def test_updater_groups_on_the_host(lib):
    """The updater's groups are the library's bucket grouping; largest_first
    orders them by parameter bytes (stable for ties), and an unknown order is
    an argument error.  Built on CPU tensors: nothing here launches."""
    import newton_schulz_04_gb300 as m
    shapes = [(64, 128), (512, 1024), (128, 64), (256, 256), (1024, 512), (64, 64)]
    params = [torch.zeros(s, dtype=torch.bfloat16) for s in shapes]
    lib_order = m.MuonUpdater(params, use_graph=False)
    order, start = m.bucket_plan(shapes)
    assert [idx for idx, _ in lib_order.groups] == [order[start[k]:start[k + 1]] for k in range(len(start) - 1)]
    big = m.MuonUpdater(params, use_graph=False, group_order="largest_first")
    nbytes = [sum(shapes[i][0] * shapes[i][1] for i in idx) for idx, _ in big.groups]
    assert nbytes == sorted(nbytes, reverse=True)
    assert sorted(map(tuple, (idx for idx, _ in big.groups))) == sorted(map(tuple, (idx for idx, _ in lib_order.groups)))
    with pytest.raises(ValueError):
        m.MuonUpdater(params, group_order="smallest_first")
