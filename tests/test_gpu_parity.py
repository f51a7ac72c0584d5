"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Tolerances (fixed for this update): relative Frobenius error of O <= 2e-2 for
bf16 operands and <= 1e-4 for the fp32 path; fp32 momentum within one fp32 ulp
of the fp64 value.  The apply W <- W - lr O is checked in two ways, so that
O_gpu (the orthogonalised momentum the library applies) is itself held to the
O tolerance:

* with W0 = 0 and a power-of-two lr, muon_step's weights must equal
  -lr * muon_ns_batched(G) bit for bit (the fused apply epilogue and the plain
  store epilogue see the same fp32 O; scaling by a power of two commutes with
  rounding to bf16), and muon_ns_batched(G) is compared with the oracle's O;
* with W0 != 0, every weight must be within its own rounding of
  W0 - lr * O_gpu: half a unit in the last place (ulp) of W, plus half an ulp
  of O (O_gpu is known here through muon_ns_batched's bf16 output), plus the
  fp32 rounding of the apply.

At zero NS steps O is known to fp32 accuracy, and the bf16 weight is checked
against RNE(W0 - lr * O_oracle) to one bf16 ulp.  The Gram schedules without
restarts (GRAM_X3 on bf16 pairs, GRAM_X1 on plain bf16: the pages' form, kept
on request for comparison) are not held to 2e-2 on rank-deficient inputs;
their errors there are measured and bounded as documented.  Every default
(AUTO) schedule is held to the tolerances above.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_FP32 = 1e-4
# The C ABI takes beta as fp32; the oracle is given that same value (widened).
BETA32 = float(np.float32(0.95))


def _m():
    import newton_schulz_04_gb300 as m
    m.load(build_if_missing=True)
    return m


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def bf16_ulp(v):
    v = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def oracle_O(x, steps=5, coeffs=oracle.QUINTIC):
    return oracle.newton_schulz(x.detach().cpu().double().numpy(), steps, coeffs)


SHAPES_BF16 = [(256, 512), (512, 256), (200, 328), (328, 200), (256, 256), (130, 1000)]


@pytest.mark.parametrize("sched", ["orig", "orig_bf16", "gram_x3", "gram_r2", "orig_f16x3"])
@pytest.mark.parametrize("shape", SHAPES_BF16)
def test_ns_batched_bf16(sched, shape):
    m = _m()
    B = 3
    X = torch.stack([synth.random_matrix(*shape, seed=40 + i) for i in range(B)]).to(torch.bfloat16).cuda()
    O = m.ns_batched(X, steps=5, schedule=sched)
    torch.cuda.synchronize()
    for i in range(B):
        e = rel(O[i].float().cpu(), oracle_O(X[i]))
        assert e < TOL_BF16, (sched, shape, i, e)


@pytest.mark.parametrize("shape", [(256, 1024), (512, 2048), (768, 3072), (1024, 8192)])
def test_ill_conditioned_low_rank_bf16(shape):
    # The rank-8 + noise recipe of the many-small-matrices workload.  The
    # default schedule (the restarted Gram recurrence, GRAM_R2, at these
    # aspects) and every accurate schedule must meet the bf16 tolerance.  Split
    # Gram space without restarts (GRAM_X3, kept for comparison) amplifies G's
    # rounding in the directions of small singular values over its 5 steps: its
    # error here is bounded, not held to 2e-2.
    m = _m()
    X = torch.stack([synth.low_rank(*shape, 8, 1e-4, seed=60 + i) for i in range(2)]).to(torch.bfloat16).cuda()
    for sched, tol in [("auto", TOL_BF16), ("orig", TOL_BF16), ("orig_bf16", TOL_BF16), ("gram_r2", TOL_BF16),
                       ("orig_f16x3", TOL_BF16), ("gram_x3", 0.1)]:
        O = m.ns_batched(X, steps=5, schedule=sched)
        torch.cuda.synchronize()
        for i in range(2):
            e = rel(O[i].float().cpu(), oracle_O(X[i]))
            assert e < tol, (sched, shape, i, e)


def _inputs_of_every_kind():
    yield "gaussian 256x768", synth.random_matrix(256, 768, seed=41)
    yield "gaussian 512x512", synth.random_matrix(512, 512, seed=42)
    yield "rank-8 768x3072", synth.low_rank(768, 3072, 8, 1e-4, seed=60)
    x = synth.random_matrix(512, 2048, seed=43)
    x[0] *= 100
    yield "row-scaled 512x2048", x


def test_orig_fp16_operands_keep_a_wide_margin():
    """ORIG multiplies fp16 operands after step 0 and carries X as an fp16 pair.
    A CPU emulation puts its error at <= 1.8e-3 on these inputs.  The bf16 split
    schedule reaches ~1e-2, so ORIG must stay well inside 2e-2."""
    m = _m()
    for name, x in _inputs_of_every_kind():
        X = x[None].to(torch.bfloat16).cuda()
        ref = oracle_O(X[0])
        e16 = rel(m.ns_batched(X, steps=5, schedule="orig")[0].float().cpu(), ref)
        ebf = rel(m.ns_batched(X, steps=5, schedule="orig_bf16")[0].float().cpu(), ref)
        assert e16 < 5e-3, (name, e16)
        assert ebf < TOL_BF16, (name, ebf)


def test_gram_r2_keeps_a_margin():
    """The Gram recurrence restarted every two steps on fp16 operands: a CPU
    emulation (fp32-exact accumulation, which the tensor cores match on these
    products) puts its worst error over rank-1 to rank-32, Gaussian,
    row-scaled and fp32-momentum inputs at 8.2e-3 before the bf16 output
    rounding, against 4.1e-3 for ORIG.  It must stay within 1.2e-2 here."""
    m = _m()
    for name, x in _inputs_of_every_kind():
        X = x[None].to(torch.bfloat16).cuda()
        e = rel(m.ns_batched(X, steps=5, schedule="gram_r2")[0].float().cpu(), oracle_O(X[0]))
        assert e < 1.2e-2, (name, e)


def test_auto_runs_gram_r2_where_it_saves_work():
    m = _m()
    assert m.resolve_schedule(4096, 14336) == "gram_r2"
    assert m.resolve_schedule(4096, 4096) == "orig"
    X = torch.stack([synth.random_matrix(256, 1024, seed=830 + i) for i in range(2)]).to(torch.bfloat16).cuda()
    a = m.ns_batched(X, steps=5)
    b = m.ns_batched(X, steps=5, schedule="gram_r2")
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_coefficients_outside_the_fp16_range_run_the_bf16_schedule():
    """The quintic scaled by 1.05 peaks at 1.26 on [0, 1.25] (over the fp16
    check's 1.25) but its iterates stay bounded.  ORIG must then run the
    bf16 split schedule, bit-identical to ORIG_BF16.  Its steeper slopes
    amplify bf16 rounding beyond the quintic's (2.7e-2 measured, against
    about 1e-2 for the quintic), so the bound here is 4e-2."""
    m = _m()
    co = tuple(1.05 * c for c in oracle.QUINTIC)
    X = torch.stack([synth.random_matrix(256, 512, seed=44 + i) for i in range(2)]).to(torch.bfloat16).cuda()
    a = m.ns_batched(X, steps=5, coeffs=co, schedule="orig")
    b = m.ns_batched(X, steps=5, coeffs=co, schedule="orig_bf16")
    q = m.ns_batched(X, steps=5, schedule="orig")
    qb = m.ns_batched(X, steps=5, schedule="orig_bf16")
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert not torch.equal(q, qb)  # the quintic itself takes the fp16 operands
    for i in range(2):
        assert rel(a[i].float().cpu(), oracle_O(X[i], 5, co)) < 4e-2


def test_unrestarted_gram_schedules_as_documented():
    """GRAM_X1 and GRAM_X3 run the Gram recurrence for all steps without
    restarts (the pages' form, kept for comparison).  On full-rank Gaussian
    inputs GRAM_X3 stays at the bf16 output rounding and plain-bf16 GRAM_X1
    is coarser.  On a rank-8 input GRAM_X1 diverges (the rounding of G grows
    in the directions of small singular values), GRAM_X3 reaches ~2e-2, and
    the restarted GRAM_R2 that AUTO uses stays within 1.2e-2."""
    m = _m()
    X = torch.stack([synth.random_matrix(256, 1024, seed=70 + i) for i in range(2)]).to(torch.bfloat16).cuda()
    O1 = m.ns_batched(X, steps=5, schedule="gram_x1")
    O3 = m.ns_batched(X, steps=5, schedule="gram_x3")
    torch.cuda.synchronize()
    for i in range(2):
        ref = oracle_O(X[i])
        e1, e3 = rel(O1[i].float().cpu(), ref), rel(O3[i].float().cpu(), ref)
        assert e3 < 4e-3, e3
        assert np.isfinite(e1) and e3 < e1 < 0.5, (e1, e3)
    L = synth.low_rank(768, 3072, 8, 1e-4, seed=60)[None].to(torch.bfloat16).cuda()
    ref = oracle_O(L[0])
    e1 = rel(m.ns_batched(L, steps=5, schedule="gram_x1")[0].float().cpu(), ref)
    e3 = rel(m.ns_batched(L, steps=5, schedule="gram_x3")[0].float().cpu(), ref)
    er = rel(m.ns_batched(L, steps=5, schedule="gram_r2")[0].float().cpu(), ref)
    assert e1 > 1.0, e1
    assert 5e-3 < e3 < 5e-2, e3
    assert er < 1.2e-2, er


@pytest.mark.parametrize("sched", ["orig", "gram_x3", "gram_r2", "orig_f16x3"])
@pytest.mark.parametrize("shape", [(128, 256), (256, 128), (200, 328), (384, 384)])
def test_ns_batched_fp32(sched, shape):
    m = _m()
    X = torch.stack([synth.random_matrix(*shape, seed=80 + i) for i in range(2)]).cuda()
    O = m.ns_batched(X, steps=5, schedule=sched)
    torch.cuda.synchronize()
    for i in range(2):
        e = rel(O[i].cpu(), oracle_O(X[i]))
        assert e < TOL_FP32, (sched, shape, i, e)


def test_c1_single_fp32_matrix_full_step():
    """Workload c1: one 128x256 fp32 matrix N(0,1) seed 0, quintic, 5 steps,
    beta 0.95 from a zero state, lr 0.02."""
    m = _m()
    w = synth.c1()
    W = w.weights[0].clone().cuda()
    G = w.grads[0].clone().cuda()
    M = torch.zeros_like(G)
    m.muon_step([W], [G], [M], beta=w.beta, lr=w.lr, steps=5)
    torch.cuda.synchronize()
    Wn, Mn, O = oracle.muon_update(w.weights[0], w.grads[0], np.zeros((128, 256)), w.beta, w.lr, 5)
    assert np.array_equal(M.cpu().double().numpy(), Mn)  # M = G exactly from a zero state
    dO = (w.weights[0].double().numpy() - W.cpu().double().numpy()) / w.lr
    assert rel(dO, O) < TOL_FP32


def _ulp(v, dtype):
    if dtype == torch.bfloat16:
        return bf16_ulp(v)
    return np.spacing(np.abs(np.asarray(v, dtype=np.float64)).astype(np.float32)).astype(np.float64)


def _check_apply(W0, Wg, O_gpu, lr, dtype):
    """Elementwise: Wg is W0 - lr * O_gpu up to the rounding of the apply (half
    an ulp of W), of O_gpu's stored copy (half an ulp of O) and of fp32."""
    W0 = np.asarray(W0, dtype=np.float64)
    Wg = np.asarray(Wg, dtype=np.float64)
    O_gpu = np.asarray(O_gpu, dtype=np.float64)
    exact = W0 - lr * O_gpu
    tol = _ulp(Wg, dtype) / 2 + lr * _ulp(O_gpu, dtype) / 2 + 2.0 ** -23 * (np.abs(W0) + lr * np.abs(O_gpu))
    bad = np.abs(Wg - exact) > tol * (1 + 1e-6)
    assert not bad.any(), (int(bad.sum()), float(np.max(np.abs(Wg - exact) / np.maximum(tol, 1e-300))))


def _check_step(shapes, dtype=torch.bfloat16, seed=0, sched="auto", steps=5, mom_init=False, ws_limit=None):
    m = _m()
    Ws, Gs, Ms = [], [], []
    for i, (a, b) in enumerate(shapes):
        # with a nonzero momentum state O_gpu cannot be recomputed through
        # muon_ns_batched, so W0 = 0 and a large lr make W show O to 2^-9
        Ws.append(torch.zeros(a, b, dtype=dtype) if mom_init else
                  synth.random_matrix(a, b, seed=seed + 1000 + i, std=0.02).to(dtype))
        Gs.append(synth.random_matrix(a, b, seed=seed + i).to(dtype))
        Ms.append(synth.random_matrix(a, b, seed=seed + 500 + i) if mom_init else torch.zeros(a, b))
    W = [w.clone().cuda() for w in Ws]
    G = [g.clone().cuda() for g in Gs]
    M = [x.clone().cuda() for x in Ms]
    ws = None
    if ws_limit is not None:
        ws = m.new_workspace(ws_limit)
    lr = 0.5 if mom_init else 0.02
    m.muon_step(W, G, M, beta=0.95, lr=lr, steps=steps, schedule=sched, workspace=ws)
    torch.cuda.synchronize()
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_FP32
    for i in range(len(shapes)):
        Wn, Mn, O = oracle.muon_update(Ws[i], Gs[i], Ms[i], BETA32, lr, steps)
        Mg = M[i].cpu().double().numpy()
        # fp32 momentum within one ulp of the fp64 value
        ulp = np.spacing(np.abs(Mn).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(Mg - Mn) <= ulp), i
        Wg = W[i].cpu().double().numpy()
        W0 = Ws[i].double().numpy()
        if not mom_init:
            # from a zero state M = G, so muon_ns_batched(G) is the O the step applied
            O_gpu = m.ns_batched(G[i][None], steps=steps, schedule=sched)[0]
            torch.cuda.synchronize()
            O_gpu = O_gpu.double().cpu().numpy()
            assert rel(O_gpu, O) < tol, (i, rel(O_gpu, O))
            _check_apply(W0, Wg, O_gpu, lr, dtype)
        else:
            # W_gpu = round(-lr O_gpu): rounding adds at most 2^-9 (bf16) relative
            e = rel(-Wg / lr, O)
            assert e < tol + (2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -23), (i, e)


def _check_zero_weight_apply(m, G, O_ref, steps=5, sched="auto", lr=2.0 ** -5, idx=None, tol=TOL_BF16):
    """W0 = 0 and a power-of-two lr: W after muon_step must be -lr times
    muon_ns_batched's output bit for bit, and that output must match the
    oracle's O (given for the indices in `idx`)."""
    W = [torch.zeros_like(g) for g in G]
    M = [torch.zeros(g.shape, dtype=torch.float32, device=g.device) for g in G]
    m.muon_step(W, G, M, beta=0.95, lr=lr, steps=steps, schedule=sched)
    torch.cuda.synchronize()
    for i in (idx if idx is not None else range(len(G))):
        O_gpu = m.ns_batched(G[i][None], steps=steps, schedule=sched)[0]
        torch.cuda.synchronize()
        assert torch.equal(W[i], -lr * O_gpu), i
        if O_ref is not None and i in O_ref:
            e = rel(O_gpu.double().cpu().numpy(), O_ref[i])
            assert e < tol, (i, e)
        assert torch.count_nonzero(W[i]).item() > 0.99 * W[i].numel()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_apply_epilogue_exact_at_five_steps(dtype):
    """The fused apply at T = 5 on both orientations and ragged shapes: the
    weights equal -lr * O_gpu exactly (W0 = 0, lr = 2^-5), and O_gpu matches
    the oracle within the dtype's tolerance."""
    m = _m()
    shapes = [(256, 512), (512, 256), (200, 328), (328, 200), (256, 256)]
    Gc = [synth.random_matrix(a, b, seed=2300 + i).to(dtype) for i, (a, b) in enumerate(shapes)]
    O_ref = {i: oracle_O(g) for i, g in enumerate(Gc)}
    _check_zero_weight_apply(m, [g.cuda() for g in Gc], O_ref, tol=TOL_BF16 if dtype == torch.bfloat16 else TOL_FP32)


def test_apply_with_nonzero_momentum_large_lr():
    """Nonzero momentum state (M = beta M0 + G is not a bf16 value), W0 = 0 and
    lr = 0.5, so the weight's own rounding adds at most 2^-9 to the implied O's
    relative error."""
    m = _m()
    shapes = [(256, 512), (512, 256), (200, 328)]
    Gs = [synth.random_matrix(a, b, seed=2400 + i).to(torch.bfloat16) for i, (a, b) in enumerate(shapes)]
    Ms = [synth.random_matrix(a, b, seed=2500 + i) for i, (a, b) in enumerate(shapes)]
    W = [torch.zeros(a, b, dtype=torch.bfloat16, device="cuda") for (a, b) in shapes]
    G = [g.cuda() for g in Gs]
    M = [x.clone().cuda() for x in Ms]
    lr = 0.5
    m.muon_step(W, G, M, beta=0.95, lr=lr, steps=5)
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        _, _, O = oracle.muon_update(torch.zeros(shapes[i]), Gs[i], Ms[i], BETA32, lr, 5)
        e = rel(-W[i].cpu().double().numpy() / lr, O)
        assert e < TOL_BF16 + 2.0 ** -8, (i, e)


def test_apply_and_momentum_exact_at_zero_steps():
    """With zero NS steps O = M / (||M||_F + eps) is known to fp32 accuracy, so
    the bf16 weight must be within one bf16 ulp of RNE(W0 - lr O) and the fp32
    momentum within one fp32 ulp of beta*M0 + G."""
    m = _m()
    shapes = [(256, 512), (512, 256), (200, 328)]
    Ws = [synth.random_matrix(a, b, seed=2000 + i, std=0.02).to(torch.bfloat16) for i, (a, b) in enumerate(shapes)]
    Gs = [synth.random_matrix(a, b, seed=2100 + i).to(torch.bfloat16) for i, (a, b) in enumerate(shapes)]
    Ms = [synth.random_matrix(a, b, seed=2200 + i) for i, (a, b) in enumerate(shapes)]
    W = [w.clone().cuda() for w in Ws]
    G = [g.clone().cuda() for g in Gs]
    M = [x.clone().cuda() for x in Ms]
    lr = 0.5  # large, so O is visible above W's rounding
    m.muon_step(W, G, M, beta=0.95, lr=lr, steps=0)
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        Wn, Mn, O = oracle.muon_update(Ws[i], Gs[i], Ms[i], BETA32, lr, 0)
        ulp = np.spacing(np.abs(Mn).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(M[i].cpu().double().numpy() - Mn) <= ulp), i
        ref = oracle.bf16_round(Wn)
        # one bf16 ulp, plus the rounding of the fp32 apply W0 - lr O, which shows
        # where the two terms nearly cancel
        W0 = Ws[i].double().numpy()
        tol = bf16_ulp(ref) + 2.0 ** -22 * (np.abs(W0) + lr * np.abs(O))
        assert np.all(np.abs(W[i].cpu().double().numpy() - ref) <= tol), i


def test_muon_step_mixed_shapes_and_orientations():
    # one bucket holds 256x512 and 512x256 members (transposed on the fly)
    _check_step([(256, 512), (512, 256), (256, 256), (256, 512), (200, 328), (328, 200)])


def test_muon_step_nonzero_momentum_state():
    _check_step([(256, 512), (512, 256)], mom_init=True, seed=7)


def test_muon_step_small_workspace_chunks_the_batch():
    m = _m()
    shapes = [(256, 512)] * 5
    one = m.workspace_bytes(shapes[:1])
    _check_step(shapes, ws_limit=one + one // 2, seed=11)


def test_muon_step_fp32():
    _check_step([(128, 256), (256, 128), (384, 384)], dtype=torch.float32, seed=13)


def test_steps_zero_returns_normalised_input():
    m = _m()
    X = torch.stack([synth.random_matrix(200, 328, seed=90 + i) for i in range(2)]).to(torch.bfloat16).cuda()
    O = m.ns_batched(X, steps=0)
    torch.cuda.synchronize()
    for i in range(2):
        ref = oracle_O(X[i], steps=0)
        assert rel(O[i].float().cpu(), ref) < 4e-3  # bf16 output rounding only


def test_zero_matrix_gives_zero():
    m = _m()
    X = torch.zeros(2, 256, 512, dtype=torch.bfloat16, device="cuda")
    for sched in ["orig", "gram_x3", "gram_x1"]:
        O = m.ns_batched(X, steps=5, schedule=sched)
        torch.cuda.synchronize()
        assert torch.count_nonzero(O).item() == 0


def test_custom_coefficients_cubic():
    m = _m()
    X = torch.stack([synth.random_matrix(256, 512, seed=95)]).cuda()
    cub = (1.5, -0.5, 0.0)
    O = m.ns_batched(X, steps=12, coeffs=cub)
    torch.cuda.synchronize()
    assert rel(O[0].cpu(), oracle_O(X[0], 12, cub)) < TOL_FP32


def test_determinism_bitwise():
    m = _m()
    X = torch.stack([synth.random_matrix(512, 1024, seed=97 + i) for i in range(3)]).to(torch.bfloat16).cuda()
    for sched in ["orig", "orig_bf16", "gram_x3", "gram_r2", "orig_f16x3"]:
        a = m.ns_batched(X, steps=5, schedule=sched)
        b = m.ns_batched(X, steps=5, schedule=sched)
        torch.cuda.synchronize()
        assert torch.equal(a, b)


def test_c2_full_size_sampled():
    """Workload c2 at full size in the benchmark's launch configuration: 16
    square 1024x1024 bf16 grads N(0, 0.02^2), zero momentum, 5 steps.  O_gpu
    (muon_ns_batched on the same grads) is checked against the oracle on two
    sampled matrices, every weight elementwise against W0 - lr O_gpu, all 16
    outputs for finiteness and the singular-value band of the map (sigma_out
    <= 1.2024 for every input); then the zero-weight run pins the apply
    epilogue bit for bit."""
    m = _m()
    w = synth.c2()
    W = [x.clone().cuda() for x in w.weights]
    G = [x.clone().cuda() for x in w.grads]
    M = [torch.zeros(x.shape, dtype=torch.float32, device="cuda") for x in w.grads]
    m.muon_step(W, G, M, beta=w.beta, lr=w.lr, steps=5)
    O = m.ns_batched(torch.stack(G), steps=5)
    torch.cuda.synchronize()
    O_ref = {}
    for i in [0, 13]:
        Wn, Mn, Oo = oracle.muon_update(w.weights[i], w.grads[i], np.zeros((1024, 1024)), w.beta, w.lr, 5)
        O_ref[i] = Oo
        assert rel(O[i].double().cpu().numpy(), Oo) < TOL_BF16
        assert np.array_equal(M[i].cpu().double().numpy(), Mn)
    for i in range(16):
        _check_apply(w.weights[i].double().numpy(), W[i].cpu().double().numpy(), O[i].double().cpu().numpy(), w.lr,
                     torch.bfloat16)
    sv = torch.linalg.svdvals(O.float())
    assert torch.isfinite(sv).all() and sv.max().item() < 1.2024 * 1.02
    _check_zero_weight_apply(m, G, O_ref)


@pytest.mark.parametrize("n", [8192])
def test_aspect_sweep_gram_auto(n):
    """Workload c5 at n = 8192: 2 of the 8 matrices, row 0 scaled by 100 to
    skew the spectrum, through the default schedule and split Gram space."""
    m = _m()
    w = synth.c5(n=n, batch=2)
    X = torch.stack(w.grads).cuda()
    for sched in ["auto", "gram_x3"]:
        O = m.ns_batched(X, steps=5, schedule=sched)
        torch.cuda.synchronize()
        for i in range(2):
            assert rel(O[i].float().cpu(), oracle_O(w.grads[i])) < TOL_BF16, sched


def test_c3_one_layer_full_size():
    """One layer of the 32-layer d=4096 / ffn=14336 model at full size (q, k, v,
    o 4096x4096; gate, up 4096x14336; down 14336x4096), bf16 grads N(0, 1e-6),
    zero momentum, 5 steps, in the benchmark's launch configuration.  The o
    projection (4096x4096) and the down projection (14336x4096, run transposed)
    are checked against the oracle through muon_ns_batched; every weight is
    checked elementwise against W0 - lr O_gpu; the zero-weight run pins the
    apply epilogue bit for bit on all seven matrices."""
    m = _m()
    w = synth.c3(device="cuda", layers=1)
    W = [x.clone() for x in w.weights]
    G = [x.clone() for x in w.grads]
    M = [torch.zeros(x.shape, dtype=torch.float32, device="cuda") for x in w.grads]
    W0 = [x.cpu() for x in w.weights]
    m.muon_step(W, G, M, beta=w.beta, lr=w.lr, steps=5)
    torch.cuda.synchronize()
    O_ref = {}
    for i in range(7):
        O_gpu = m.ns_batched(G[i][None], steps=5)[0]
        torch.cuda.synchronize()
        O_np = O_gpu.double().cpu().numpy()
        if i in (3, 6):
            g = w.grads[i].cpu()
            Wn, Mn, Oo = oracle.muon_update(W0[i], g, np.zeros(tuple(g.shape)), w.beta, w.lr, 5)
            O_ref[i] = Oo
            e = rel(O_np, Oo)
            assert e < TOL_BF16, (i, e)
            assert np.array_equal(M[i].cpu().double().numpy(), Mn)
        _check_apply(W0[i].double().numpy(), W[i].cpu().double().numpy(), O_np, w.lr, torch.bfloat16)
    _check_zero_weight_apply(m, G, O_ref)


def test_c4_many_small_matrices_sampled():
    """The 512-matrix workload of shapes {256x1024, 512x2048, 768x3072} with
    rank-8 + noise grads, run as one muon_step; one matrix of each shape is
    checked against the oracle (O through muon_ns_batched, W elementwise)."""
    m = _m()
    w = synth.c4()
    W = [x.cuda() for x in w.weights]
    G = [x.cuda() for x in w.grads]
    M = [torch.zeros(x.shape, dtype=torch.float32, device="cuda") for x in w.grads]
    m.muon_step(W, G, M, beta=w.beta, lr=w.lr, steps=5)
    torch.cuda.synchronize()
    picked = {}
    for i, shp in enumerate(w.shapes):
        picked.setdefault(shp, i)
    assert len(picked) == 3
    for shp, i in picked.items():
        Wn, Mn, O = oracle.muon_update(w.weights[i], w.grads[i], np.zeros(shp), w.beta, w.lr, 5)
        O_gpu = m.ns_batched(G[i][None], steps=5)[0]
        torch.cuda.synchronize()
        O_gpu = O_gpu.double().cpu().numpy()
        e = rel(O_gpu, O)
        assert e < TOL_BF16, (shp, e)
        _check_apply(w.weights[i].double().numpy(), W[i].cpu().double().numpy(), O_gpu, w.lr, torch.bfloat16)


@pytest.mark.parametrize("sched", ["auto", "gram_r2", "orig_f16x3"])
@pytest.mark.parametrize("n", [1024, 2048, 4096])
def test_c5_aspect_sweep_fp32(n, sched):
    """The aspect-ratio sweep on the fp32 path (m = 1024, row 0 scaled by 100),
    2 of the 8 matrices per shape, 5 and 10 steps: FFMA (AUTO: Gram space at
    5 steps, two-step Gram segments or original space at 10) and the
    tensor-core fp16-pair schedule."""
    m = _m()
    for steps in (5, 10):
        w = synth.c5(n=n, batch=2, dtype=torch.float32, steps=steps)
        X = torch.stack(w.grads).cuda()
        O = m.ns_batched(X, steps=steps, schedule=sched)
        torch.cuda.synchronize()
        for i in range(2):
            e = rel(O[i].cpu(), oracle_O(w.grads[i], steps))
            assert e < TOL_FP32, (n, steps, i, e)


@pytest.mark.parametrize("sched", ["auto", "orig", "gram_r2"])
@pytest.mark.parametrize("steps", [5, 10])
def test_fp32_rank_deficient_inputs_stay_bounded(sched, steps):
    """fp32 rank-1 and rank-8 + noise inputs (not rounded to bf16).  fp32
    rounding of A = X X^T is far above the squared noise singular values here,
    so even FFMA in original space misses 1e-4 (measured: up to 2.2e-4 at 5
    steps, 3.3e-3 at 10).  Every fp32 schedule AUTO uses must stay finite and
    within 5e-4 (5 steps) or 5e-3 (10 steps).  (Gram space without restarts
    diverged on these inputs at 10 steps, which is why AUTO never runs it
    beyond 6.)"""
    m = _m()
    for shape, r in [((256, 1024), 8), ((768, 3072), 8), ((768, 3072), 1)]:
        X = torch.stack([synth.low_rank(*shape, r, 1e-4, seed=860 + i) for i in range(2)]).cuda()
        O = m.ns_batched(X, steps=steps, schedule=sched)
        torch.cuda.synchronize()
        assert torch.isfinite(O).all(), (sched, shape, r)
        for i in range(2):
            e = rel(O[i].cpu(), oracle_O(X[i], steps))
            assert e < (5e-4 if steps <= 6 else 5e-3), (sched, shape, r, i, e)


def test_fp32_pair_schedule_full_step():
    """muon_step on fp32 data through the tensor-core fp32 schedule: the c1
    matrix and both orientations of a ragged shape, momentum within one fp32
    ulp, weights elementwise against W0 - lr O_gpu."""
    _check_step([(128, 256), (256, 128), (200, 328)], dtype=torch.float32, seed=17, sched="orig_f16x3")
    _check_step([(256, 512)], dtype=torch.float32, seed=19, sched="orig_f16x3", mom_init=True)


def test_fp32_restarted_gram_full_step():
    _check_step([(128, 512), (512, 128), (200, 600)], dtype=torch.float32, seed=23, sched="gram_r2", steps=10)


def test_updater_graphs_for_alternating_gradient_buffers():
    """MuonUpdater keeps one CUDA graph per set of gradient tensors, so two
    buffers used in turn (the next step's gradients copied in while this step
    runs) replay their own graphs.  Four steps must equal four direct calls
    bit for bit, including the momentum."""
    m = _m()
    shapes = [(256, 512), (512, 256), (256, 768)]
    W0 = [synth.random_matrix(a, b, seed=600 + i, std=0.02).to(torch.bfloat16) for i, (a, b) in enumerate(shapes)]
    Gs = [[synth.random_matrix(a, b, seed=700 + 10 * k + i).to(torch.bfloat16).cuda() for i, (a, b) in enumerate(shapes)]
          for k in range(2)]
    Wg = [w.clone().cuda() for w in W0]
    We = [w.clone().cuda() for w in W0]
    upd = m.MuonUpdater(Wg, 0.95, 0.02, 5, use_graph=True)
    ref = m.MuonUpdater(We, 0.95, 0.02, 5, use_graph=False)
    for k in range(4):
        upd.step(Gs[k % 2])
        ref.step(Gs[k % 2])
    torch.cuda.synchronize()
    assert len(upd._graphs) == 2
    for a, b in zip(Wg, We):
        assert torch.equal(a, b)
    for a, b in zip(upd.moms, ref.moms):
        assert torch.equal(a, b)


def test_updater_group_order_and_hooks():
    """Running the shape groups largest first, with a per-group copy-out of the
    weights on another stream (the end-to-end pattern), gives the same weights
    and momentum, bit for bit, as the library order without hooks; the hooks
    see every group once, in the order the updater reports."""
    m = _m()
    shapes = [(256, 512), (1024, 256), (256, 768), (512, 256), (256, 1024)]
    W0 = [synth.random_matrix(a, b, seed=900 + i, std=0.02).to(torch.bfloat16) for i, (a, b) in enumerate(shapes)]
    Gs = [[synth.random_matrix(a, b, seed=950 + 10 * k + i).to(torch.bfloat16).cuda() for i, (a, b) in enumerate(shapes)]
          for k in range(2)]
    Wa = [w.clone().cuda() for w in W0]
    Wb = [w.clone().cuda() for w in W0]
    upd = m.MuonUpdater(Wa, 0.95, 0.02, 5, use_graph=True, group_order="largest_first")
    ref = m.MuonUpdater(Wb, 0.95, 0.02, 5, use_graph=False)
    sizes = [sum(shapes[i][0] * shapes[i][1] for i in idx) for idx, _ in upd.groups]
    assert sizes == sorted(sizes, reverse=True)
    assert sorted(i for idx, _ in upd.groups for i in idx) == list(range(len(shapes)))
    host = [torch.empty(w.shape, dtype=w.dtype).pin_memory() for w in Wa]
    out = torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in upd.groups]
    for e in copied:
        e.record()
    seen = []

    def before(gi, idx, st):
        st.wait_event(copied[gi])  # the previous copy of these weights has left

    def after(gi, idx, st):
        seen.append((gi, list(idx)))
        ev = torch.cuda.Event()
        ev.record(st)
        with torch.cuda.stream(out):
            out.wait_event(ev)
            for q in idx:
                host[q].copy_(Wa[q], non_blocking=True)
            copied[gi].record(out)

    for k in range(3):
        upd.step(Gs[k % 2], before_group=before, after_group=after)
        ref.step(Gs[k % 2])
    torch.cuda.synchronize()
    assert seen[:len(upd.groups)] == [(gi, idx) for gi, (idx, _) in enumerate(upd.groups)]
    assert len(seen) == 3 * len(upd.groups)
    for a, b, h in zip(Wa, Wb, host):
        assert torch.equal(a, b)
        assert torch.equal(h, a.cpu())
    for a, b in zip(upd.moms, ref.moms):
        assert torch.equal(a, b)


@pytest.mark.parametrize("sched,dtype", [("orig", torch.bfloat16), ("gram_x3", torch.bfloat16),
                                         ("gram_r2", torch.bfloat16), ("orig", torch.float32),
                                         ("gram_x3", torch.float32), ("orig_f16x3", torch.float32),
                                         ("gram_r2", torch.float32)])
@pytest.mark.parametrize("steps", [1, 2, 3])
def test_each_product_through_few_steps(sched, dtype, steps):
    """One step is O = P_0 X_0 with P_0 = a I + b G_0 + c G_0^2 (the SYRK, the
    polynomial and the projection); two steps add the Q and G updates (Gram)
    or a second X update (original).  Checking T = 1, 2, 3 against the oracle
    pins each product's contribution, on a ragged shape (200 x 328)."""
    m = _m()
    X = torch.stack([synth.random_matrix(200, 328, seed=810 + i) for i in range(2)]).to(dtype).cuda()
    O = m.ns_batched(X, steps=steps, schedule=sched)
    torch.cuda.synchronize()
    tol = TOL_FP32 if dtype == torch.float32 else TOL_BF16
    for i in range(2):
        e = rel(O[i].float().cpu(), oracle_O(X[i], steps))
        assert e < tol, (sched, dtype, steps, i, e)


@pytest.mark.parametrize("sched,steps,coeffs", [("orig", 7, None), ("gram_x3", 7, None), ("orig_bf16", 7, None),
                                                ("orig", 12, (1.5, -0.5, 0.0)), ("gram_r2", 7, None),
                                                ("gram_r2", 10, None), ("gram_r2", 12, (1.5, -0.5, 0.0))])
def test_more_products_than_one_shared_launch(sched, steps, coeffs):
    """A short chunk runs up to 16 consecutive products in one launch; 7 or 12
    steps need several such launches, chained on the same per-matrix counters."""
    m = _m()
    X = torch.stack([synth.random_matrix(256, 512, seed=820 + i) for i in range(3)]).to(torch.bfloat16).cuda()
    O = m.ns_batched(X, steps=steps, schedule=sched, coeffs=coeffs)
    torch.cuda.synchronize()
    for i in range(3):
        e = rel(O[i].float().cpu(), oracle_O(X[i], steps, coeffs or oracle.QUINTIC))
        assert e < TOL_BF16, (sched, steps, i, e)


def test_longest_side_at_the_maximum():
    """The largest accepted dimension (65536) as the long side, in both
    orientations, through muon_step with the default schedule (the restarted
    Gram recurrence at this aspect); W checked elementwise against
    W0 - lr O_gpu and O_gpu against the oracle on each matrix."""
    m = _m()
    shapes = [(256, 65536), (65536, 256)]
    Gs = [synth.random_matrix(a, b, seed=2700 + i).to(torch.bfloat16) for i, (a, b) in enumerate(shapes)]
    Ws = [synth.random_matrix(a, b, seed=2800 + i, std=0.02).to(torch.bfloat16) for i, (a, b) in enumerate(shapes)]
    W = [w.cuda() for w in Ws]
    G = [g.cuda() for g in Gs]
    M = [torch.zeros(g.shape, dtype=torch.float32, device="cuda") for g in Gs]
    assert m.resolve_schedule(256, 65536) == "gram_r2"
    m.muon_step(W, G, M, beta=0.95, lr=0.02, steps=5)
    torch.cuda.synchronize()
    for i in range(2):
        O_gpu = m.ns_batched(G[i][None], steps=5)[0].double().cpu().numpy()
        e = rel(O_gpu, oracle_O(Gs[i]))
        assert e < TOL_BF16, (i, e)
        _check_apply(Ws[i].double().numpy(), W[i].cpu().double().numpy(), O_gpu, 0.02, torch.bfloat16)


def test_transposed_apply_with_unaligned_rows():
    """A matrix stored transposed to its packed form whose rows (the short
    side, 130 bf16 values = 260 bytes) are not 16-byte multiples takes the
    per-element final path; its neighbour with aligned rows (the block path)
    runs in the same call."""
    _check_step([(1000, 130), (600, 200)], seed=31)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_pair_schedule_falls_back_outside_the_fp16_range(dtype):
    """Coefficients whose polynomial leaves [-1.25, 1.25] on [0, 1.25] (the
    quintic scaled by 1.05) cannot run on fp16 pairs: ORIG_F16X3 then runs
    the bf16 split schedule (bf16 data) or FFMA original space (fp32 data),
    bit for bit."""
    m = _m()
    co = tuple(1.05 * c for c in oracle.QUINTIC)
    X = torch.stack([synth.random_matrix(256, 512, seed=2900 + i) for i in range(2)]).to(dtype).cuda()
    a = m.ns_batched(X, steps=5, coeffs=co, schedule="orig_f16x3")
    b = m.ns_batched(X, steps=5, coeffs=co, schedule="orig_bf16" if dtype == torch.bfloat16 else "orig")
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("steps", [4, 6])
def test_restarted_gram_plans_with_a_final_single_step(steps):
    """GRAM_R2 splits T steps as 1, 2, 2, ..., with a last single step when
    T - 1 is odd (4 steps: 1, 2, 1; 6 steps: 1, 2, 2, 1)."""
    m = _m()
    X = torch.stack([synth.random_matrix(256, 1024, seed=2950 + i) for i in range(2)]).to(torch.bfloat16).cuda()
    O = m.ns_batched(X, steps=steps, schedule="gram_r2")
    torch.cuda.synchronize()
    for i in range(2):
        e = rel(O[i].float().cpu(), oracle_O(X[i], steps))
        assert e < 1.2e-2, (steps, i, e)


@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
@pytest.mark.parametrize("sched", ["auto", "orig", "gram_r2"])
def test_nonfinite_input_stays_in_its_matrix(bad, sched):
    """A NaN or Inf in one matrix of a batch is not checked: it propagates into
    that matrix's output (its norm is not finite), and the other matrices of
    the same launches come out bit for bit as without it."""
    m = _m()
    X = torch.stack([synth.random_matrix(256, 768, seed=3000 + i) for i in range(3)]).to(torch.bfloat16).cuda()
    ref = m.ns_batched(X, steps=5, schedule=sched)
    Xb = X.clone()
    Xb[1, 17, 100] = bad
    out = m.ns_batched(Xb, steps=5, schedule=sched)
    torch.cuda.synchronize()
    assert not torch.isfinite(out[1].float()).all()
    assert torch.equal(out[0], ref[0]) and torch.equal(out[2], ref[2])


@pytest.mark.parametrize("sched", ["auto", "orig"])
def test_rows_spanning_six_decades(sched):
    """Row norms spread log-uniformly over 1e-3 .. 1e3 (bf16 data): after the
    Frobenius normalisation most rows sit far below fp16's normal range, where
    the fp16 pair keeps their low part; the result must still meet the bf16
    tolerance."""
    m = _m()
    g = torch.Generator().manual_seed(3100)
    X = torch.randn(2, 512, 2048, generator=g)
    X *= (10.0 ** (6.0 * torch.rand(2, 512, 1, generator=g) - 3.0))
    X = X.to(torch.bfloat16).cuda()
    O = m.ns_batched(X, steps=5, schedule=sched)
    torch.cuda.synchronize()
    for i in range(2):
        e = rel(O[i].float().cpu(), oracle_O(X[i]))
        assert e < TOL_BF16, (sched, i, e)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_degenerate_shapes(dtype):
    """Single rows, single columns, 1 x 1 and tiny matrices: a 1 x n matrix has
    one singular value, so O is x / |x| mapped by the scalar polynomial; each
    pads to one 256 x 256 tile pair.  Checked through muon_step against the
    oracle, in one call with every shape."""
    _check_step([(1, 1), (1, 300), (300, 1), (2, 2), (17, 5), (5, 17), (1, 4096)], dtype=dtype, seed=41)


def test_muon_step_more_matrices_than_one_chunk():
    """300 matrices of one shape group (both orientations) exceed the 256
    matrices a chunk takes: the group runs as two chunks through the same
    workspace, and every matrix's update still matches the oracle."""
    shapes = [(64, 128) if i % 3 else (128, 64) for i in range(300)]
    _check_step(shapes, seed=47)


def test_ns_batched_more_matrices_than_one_chunk():
    """muon_ns_batched with B = 300 (over the 256 a chunk takes): sampled
    matrices from both chunks against the oracle, and every output finite."""
    m = _m()
    g = torch.Generator().manual_seed(49)
    X = torch.randn(300, 64, 128, generator=g).to(torch.bfloat16).cuda()
    O = m.ns_batched(X, steps=5)
    torch.cuda.synchronize()
    assert torch.isfinite(O.float()).all()
    for i in (0, 131, 255, 256, 299):
        e = rel(O[i].float().cpu(), oracle_O(X[i]))
        assert e < TOL_BF16, (i, e)


@pytest.mark.parametrize("steps", [6, 7])
def test_fp32_at_the_pair_schedule_threshold(steps):
    """fp32 AUTO runs the tensor-core fp16 pairs up to 6 steps and FFMA from
    7: both sides of the switch meet 1e-4 on Gaussian and row-scaled inputs."""
    m = _m()
    assert m.resolve_schedule(512, 2048, steps=steps, dtype=torch.float32) == ("orig_f16x3" if steps <= 6 else "gram_r2")
    x = synth.random_matrix(512, 2048, seed=53)
    y = synth.random_matrix(512, 2048, seed=54)
    y[0] *= 100
    X = torch.stack([x, y]).cuda()
    O = m.ns_batched(X, steps=steps)
    torch.cuda.synchronize()
    for i in range(2):
        e = rel(O[i].cpu(), oracle_O(X[i], steps))
        assert e < TOL_FP32, (steps, i, e)


@pytest.mark.parametrize("sched", ["auto", "orig", "gram_r2", "orig_bf16"])
def test_identity_coefficients_return_the_normalised_input(sched):
    """With (a, b, c) = (1, 0, 0) every step maps X to itself, so O is
    X / (||X||_F + eps) whatever the schedule: the polynomial epilogues, the
    Gram segments and the low-part bookkeeping must add nothing."""
    m = _m()
    X = torch.stack([synth.random_matrix(256, 768, seed=57 + i) for i in range(2)]).to(torch.bfloat16).cuda()
    O = m.ns_batched(X, steps=3, coeffs=(1.0, 0.0, 0.0), schedule=sched)
    torch.cuda.synchronize()
    for i in range(2):
        x = X[i].double().cpu().numpy()
        ref = x / (np.linalg.norm(x) + oracle.EPS)
        assert rel(O[i].float().cpu(), ref) < 2e-3, (sched, i)  # the bf16 output rounding only
        assert rel(oracle_O(X[i], 3, (1.0, 0.0, 0.0)), ref) < 1e-12


@pytest.mark.parametrize("shape", [(4096, 14336), (200, 328), (1000, 130), (300, 72)])
def test_transpose_equivariance_bitwise(shape):
    """NS(X^T) = NS(X)^T.  The library packs the short side first and sums each
    packed tile's squares in packed order, so X and X^T run the same products
    on the same packed matrix and norm: the outputs agree bit for bit.  This
    pins the transposed pack, the norm, and the transposed output path (the
    4096 x 14336 case is the full-size down projection; 1000 x 130 and
    300 x 72 pair the 8-wide pack kernel with the per-element one)."""
    m = _m()
    X = synth.random_matrix(*shape, seed=59).to(torch.bfloat16).cuda()[None]
    Xt = X.transpose(1, 2).contiguous()
    O = m.ns_batched(X, steps=5)
    Ot = m.ns_batched(Xt, steps=5)
    torch.cuda.synchronize()
    assert torch.equal(Ot, O.transpose(1, 2))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_result_independent_of_batch_company(dtype):
    """A matrix's output does not depend on what else is in the call: alone,
    in a batch of 7 (another launch mode and tile schedule), or in a muon_step
    with other shape groups, it is bit for bit the same."""
    m = _m()
    X = synth.random_matrix(256, 1024, seed=61).to(dtype).cuda()
    others = torch.stack([synth.random_matrix(256, 1024, seed=62 + i) for i in range(6)]).to(dtype).cuda()
    alone = m.ns_batched(X[None], steps=5)[0]
    batch = m.ns_batched(torch.cat([others[:3], X[None], others[3:]]), steps=5)[3]
    torch.cuda.synchronize()
    assert torch.equal(alone, batch)
    # through muon_step: W = 0, lr = 2^-5, so W = -lr O exactly (see the apply tests)
    shapes = [(256, 1024), (512, 512), (1024, 256), (300, 200)]
    Ws = [torch.zeros(s, dtype=dtype, device="cuda") for s in shapes]
    Gs = [X] + [synth.random_matrix(*s, seed=70 + i).to(dtype).cuda() for i, s in enumerate(shapes[1:])]
    Ms = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in shapes]
    m.muon_step(Ws, Gs, Ms, beta=0.95, lr=2.0 ** -5, steps=5)
    W1 = torch.zeros_like(X)
    m.muon_step([W1], [X], [torch.zeros(X.shape, dtype=torch.float32, device="cuda")], beta=0.95, lr=2.0 ** -5,
                steps=5)
    torch.cuda.synchronize()
    assert torch.equal(Ws[0], W1)


@pytest.mark.parametrize("steps", [12, 20, 100])
def test_bf16_long_runs_meet_the_tolerance(steps):
    """The quintic does not contract inside its band, so single fp16 operands
    drift past 2e-2 beyond about 12 steps; AUTO then runs fp16 pairs, which
    stay near the bf16 output rounding.  Checked up to the maximum step count
    on the inputs where the drift was largest."""
    m = _m()
    y = synth.random_matrix(512, 2048, seed=84)
    y[0] *= 100
    for name, x in (("gauss 256x512", synth.random_matrix(256, 512, seed=80)), ("rowx100 512x2048", y)):
        X = x[None].to(torch.bfloat16).cuda()
        O = m.ns_batched(X, steps=steps)
        torch.cuda.synchronize()
        e = rel(O[0].float().cpu(), oracle_O(X[0], steps))
        assert e < 1e-2, (steps, name, e)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_large_ragged_shapes(dtype):
    """Large shapes that are not multiples of the 256 tile: 2000 x 3000 pads to
    2048 x 3072, so every product's last tile row and column, the symmetric
    products' diagonal tiles and the apply all run partly on padding."""
    _check_step([(2000, 3000), (3000, 2000)], dtype=dtype, seed=91)


def test_seeded_fuzz_of_shapes_steps_and_schedules():
    """150 seeded draws of (m, n) in [1, 1200], dtype, 1-14 steps and an
    accurate schedule (or AUTO), each through muon_ns_batched with a batch of
    1-3 matrices, against the oracle at the dtype's tolerance (Gaussian
    inputs)."""
    m = _m()
    rng = np.random.default_rng(2024)
    bf16_scheds = ["auto", "orig", "gram_r2", "orig_f16x3"]
    fp32_scheds = ["auto", "orig", "gram_r2", "orig_f16x3"]
    for case in range(150):
        a, b = (int(v) for v in rng.integers(1, 1201, size=2))
        dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
        steps = int(rng.integers(1, 15))
        scheds = bf16_scheds if dtype == torch.bfloat16 else fp32_scheds
        sched = scheds[int(rng.integers(0, len(scheds)))]
        if dtype == torch.bfloat16 and steps > 10 and sched in ("orig", "gram_r2"):
            sched = "auto"  # single fp16 operands are documented to drift past 10 steps
        if dtype == torch.float32 and steps > 6 and sched == "orig_f16x3":
            sched = "auto"  # fp16 pairs on fp32 data are for up to 6 steps
        B = int(rng.integers(1, 4))
        X = torch.stack([synth.random_matrix(a, b, seed=5000 + 10 * case + i) for i in range(B)]).to(dtype).cuda()
        O = m.ns_batched(X, steps=steps, schedule=sched)
        torch.cuda.synchronize()
        tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_FP32
        for i in range(B):
            e = rel(O[i].float().cpu(), oracle_O(X[i], steps))
            assert e < tol, (case, (a, b), str(dtype), steps, sched, i, e)


def test_seeded_fuzz_of_muon_step_calls():
    """12 seeded muon_step calls, each over 2-6 matrices of random shapes (so
    several shape groups, both orientations) in one dtype, checked matrix by
    matrix: momentum to one fp32 ulp, O against the oracle, W elementwise."""
    rng = np.random.default_rng(2025)
    for call in range(12):
        dtype = torch.bfloat16 if call % 3 else torch.float32
        shapes = [tuple(int(v) for v in rng.integers(1, 700, size=2)) for _ in range(int(rng.integers(2, 7)))]
        _check_step(shapes, dtype=dtype, seed=6000 + 100 * call, steps=int(rng.integers(1, 9)))
