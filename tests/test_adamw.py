"""AdamW on the non-matrix tail: the oracle's pins (CPU), the C ABI's argument
checks (CPU), and the CUDA kernel against the oracle (GPU)."""
import math

import numpy as np
import pytest
import torch

from oracle import adamw as A

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


# ---------------------------------------------------------------- oracle pins

def test_constant_gradient_closed_form():
    """With a constant g from zero moments, m_t = (1 - b1^t) g and
    v_t = (1 - b2^t) g^2, so every bias-corrected step is lr g / (|g| + eps)."""
    rng = np.random.default_rng(0)
    g = rng.standard_normal(257) * 1e-2
    p0 = rng.standard_normal(257)
    p, m, v = p0.copy(), np.zeros(257), np.zeros(257)
    hp = dict(HP, weight_decay=0.0)
    for t in range(1, 8):
        p, m, v = A.adamw_step(p, g, m, v, step=t, **hp)
        np.testing.assert_allclose(m, (1 - 0.9 ** t) * g, rtol=1e-13)
        np.testing.assert_allclose(v, (1 - 0.999 ** t) * g * g, rtol=1e-12)
    expect = p0 - 7 * 1e-3 * g / (np.abs(g) + 1e-8)
    np.testing.assert_allclose(p, expect, rtol=0, atol=1e-14)  # 7 steps of fp64 rounding on |p| ~ 2


def test_zero_gradient_is_pure_decoupled_decay():
    p0 = np.linspace(-2, 2, 101)
    p, m, v = p0.copy(), np.zeros(101), np.zeros(101)
    for t in range(1, 6):
        p, m, v = A.adamw_step(p, np.zeros(101), m, v, step=t, **HP)
    np.testing.assert_allclose(p, p0 * (1 - 1e-3 * 0.01) ** 5, rtol=1e-15)
    assert not m.any() and not v.any()


def test_matches_torch_adamw_in_float64():
    torch.manual_seed(1)
    shape = (3, 41)
    p0 = torch.randn(shape, dtype=torch.float64)
    param = torch.nn.Parameter(p0.clone())
    opt = torch.optim.AdamW([param], lr=3e-3, betas=(0.8, 0.95), eps=1e-3, weight_decay=0.1, foreach=False)
    p, m, v = p0.numpy().copy(), np.zeros(shape), np.zeros(shape)
    for t in range(1, 6):
        g = torch.randn(shape, dtype=torch.float64)
        param.grad = g.clone()
        opt.step()
        p, m, v = A.adamw_step(p, g.numpy(), m, v, lr=3e-3, beta1=0.8, beta2=0.95, eps=1e-3, weight_decay=0.1,
                               step=t)
    np.testing.assert_allclose(p, param.detach().numpy(), rtol=1e-13, atol=1e-15)
    st = opt.state[param]
    np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-13)
    np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-13)


def _coupled(p, g, m, v, lr, beta1, beta2, eps, weight_decay, step):  # planted slip: L2 decay in the gradient
    return A.adamw_step(p, np.asarray(g) + weight_decay * np.asarray(p), m, v, lr, beta1, beta2, eps, 0.0, step)


def _no_bias_correction(p, g, m, v, lr, beta1, beta2, eps, weight_decay, step):  # planted slip
    return A.adamw_step(p, g, m, v, lr, beta1, beta2, eps, weight_decay, step=10 ** 9)


@pytest.mark.parametrize("slip", [_coupled, _no_bias_correction])
def test_planted_slips_break_a_pin(slip):
    p0 = np.linspace(-2, 2, 11)
    g = np.full(11, 1e-2)
    p1, m1, v1 = slip(p0, np.zeros(11), np.zeros(11), np.zeros(11), step=1, **HP)
    p2, _, _ = slip(p0, g, np.zeros(11), np.zeros(11), step=1, **dict(HP, weight_decay=0.0))
    decay_ok = np.allclose(p1, p0 * (1 - 1e-5), rtol=1e-15)
    step_ok = np.allclose(p2, p0 - 1e-3 * g / (np.abs(g) + 1e-8), rtol=0, atol=1e-15)
    assert not (decay_ok and step_ok)


# ---------------------------------------------------------------- ABI (CPU)

def _lib():
    import newton_schulz_04_gb300 as mm
    from newton_schulz_04_gb300 import build as b
    b.build()
    return mm


def test_adamw_abi_rejects_bad_arguments_before_launch():
    import ctypes
    mm = _lib()
    lib = mm.load()
    P = ctypes.c_void_p * 1
    fake = P(ctypes.c_void_p(256))
    n = (ctypes.c_int64 * 1)(8)
    call = lambda **kw: lib.muon_adamw_tail(  # noqa: E731
        kw.get("p", fake), fake, fake, fake, kw.get("n", n), kw.get("count", 1), kw.get("lr", 1e-3), kw.get("b1", 0.9),
        0.999, kw.get("eps", 1e-8), 0.0, kw.get("step", 1), kw.get("dt", 0), None)
    assert call(count=0) == 0                                 # empty tail: nothing to do
    assert call(count=-1) == 1                                # MUON_ERR_ARG
    assert call(step=0) == 1
    assert call(lr=math.nan) == 1
    assert call(b1=1.0) == 1
    assert call(eps=-1.0) == 1
    assert call(dt=7) == 1
    assert call(n=(ctypes.c_int64 * 1)(-1)) == 2             # MUON_ERR_SHAPE
    assert call(p=P(ctypes.c_void_p(257))) == 3               # MUON_ERR_ALIGN (bf16 at an odd address)
    assert call(p=P(None)) == 1                               # NULL pointer of a non-empty tensor
    assert call(n=(ctypes.c_int64 * 1)(0)) == 0               # all tensors empty: nothing launched


# ---------------------------------------------------------------- GPU parity

def _tail(dtype, sizes, seed, offset_elems=0):
    g = torch.Generator().manual_seed(seed)
    out = []
    for k in sizes:
        buf = lambda std: (torch.randn(k + offset_elems, generator=g) * std)  # noqa: E731
        p = buf(1.0).to(dtype)[offset_elems:]
        gr = buf(1e-2).to(dtype)[offset_elems:]
        out.append((p, gr))
    return out


def _check_against_oracle(dtype, sizes, steps, seed, offset_elems=0, hp=None):
    mm = _lib()
    # the C ABI takes the hyperparameters as fp32; the oracle gets those same values, widened
    hp = {k: float(np.float32(v)) for k, v in (hp or HP).items()}
    tail = _tail(dtype, sizes, seed, offset_elems)
    P = [p.cuda() for p, _ in tail]
    G = [g.cuda() for _, g in tail]
    M = [torch.zeros(p.numel(), dtype=torch.float32, device="cuda") for p in P]
    V = [torch.zeros(p.numel(), dtype=torch.float32, device="cuda") for p in P]
    ref = [(p.double().numpy(), np.zeros(p.numel()), np.zeros(p.numel())) for p, _ in tail]
    for t in range(1, steps + 1):
        mm.adamw_tail(P, G, M, V, lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
                      weight_decay=hp["weight_decay"], step=t)
        nref = []
        for (rp, rm, rv), (_, gr) in zip(ref, tail):
            rp, rm, rv = A.adamw_step(rp, gr.double().numpy(), rm, rv, step=t, **hp)
            if dtype == torch.bfloat16:  # the device keeps p in bf16 between steps
                rp = torch.from_numpy(rp).to(torch.bfloat16).double().numpy()
            nref.append((rp, rm, rv))
        ref = nref
    torch.cuda.synchronize()
    for i, (rp, rm, rv) in enumerate(ref):
        gp = P[i].double().cpu().numpy()
        if dtype == torch.bfloat16:
            # one bf16 rounding of an fp32 result: within one bf16 ulp of the rounded fp64 value
            ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(rp), 1e-30))) - 7)
            assert np.all(np.abs(gp - rp) <= ulp), i
        else:
            np.testing.assert_allclose(gp, rp, rtol=2e-6, atol=1e-9)
        np.testing.assert_allclose(M[i].double().cpu().numpy(), rm, rtol=2e-6, atol=1e-12)
        np.testing.assert_allclose(V[i].double().cpu().numpy(), rv, rtol=2e-6, atol=1e-15)


SIZES = [0, 1, 7, 8, 9, 4096, 4099, 65536 + 3, 300001]


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_adamw_tail_matches_oracle(dtype):
    _check_against_oracle(dtype, SIZES, steps=4, seed=11)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_adamw_tail_unaligned_tensors_take_the_scalar_path(dtype):
    _check_against_oracle(dtype, [5, 64, 1000, 33333], steps=2, seed=12, offset_elems=1)


@pytest.mark.gpu
def test_adamw_tail_more_tensors_than_one_launch_holds():
    sizes = [(7 * i) % 513 + 1 for i in range(300)]  # 300 tensors -> 3 launches of up to 128
    _check_against_oracle(torch.float32, sizes, steps=2, seed=13,
                          hp=dict(lr=2e-3, beta1=0.8, beta2=0.95, eps=1e-6, weight_decay=0.1))


@pytest.mark.gpu
def test_adamw_tail_of_the_32_layer_model():
    """The 1-D tail of the 32-layer d=4096 model: two RMSNorm weights per
    layer and a final norm, 65 vectors of 4096, bf16, 3 steps."""
    _check_against_oracle(torch.bfloat16, [4096] * 65, steps=3, seed=14)


@pytest.mark.gpu
def test_adamw_tail_object_matches_the_function_bitwise():
    """AdamwTail (pointer tables built once, step counted inside) runs the same
    kernel as adamw_tail, so three steps give identical bits; 600 tensors take
    two launches."""
    mm = _lib()
    sizes = [(13 * i) % 700 + 1 for i in range(600)]
    a = [(p.cuda(), g.cuda()) for p, g in _tail(torch.bfloat16, sizes, 15)]
    b = [(p.clone(), g) for p, g in a]
    mk = lambda: [torch.zeros(p.numel(), dtype=torch.float32, device="cuda") for p, _ in a]  # noqa: E731
    Ma, Va, Mb, Vb = mk(), mk(), mk(), mk()
    opt = mm.AdamwTail([p for p, _ in a], [g for _, g in a], Ma, Va, lr=2e-3, weight_decay=0.05)
    for t in range(1, 4):
        opt.step()
        mm.adamw_tail([p for p, _ in b], [g for _, g in b], Mb, Vb, lr=2e-3, weight_decay=0.05, step=t)
    torch.cuda.synchronize()
    assert opt.t == 3
    for (pa, _), (pb, _), ma, mb, va, vb in zip(a, b, Ma, Mb, Va, Vb):
        assert torch.equal(pa, pb) and torch.equal(ma, mb) and torch.equal(va, vb)
