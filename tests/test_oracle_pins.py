"""Pins of the fp64 CPU oracle to things other than itself.

The pages print no worked example, so each pin is a closed form, a library
routine that computes the same mathematical object another way, an invariant
of the iteration, or brute force on a tiny input.  Each one is chosen so that a
plausible slip in the oracle (a dropped polynomial term, a wrong sign, X^T X in
place of X X^T, a missing normalisation, a wrong orientation) fails it.
"""
import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
import synth

A5, B5, C5 = 3.4445, -4.7750, 2.0315


def scalar_map(sig, steps, a=A5, b=B5, c=C5):
    """The NS polynomial applied to one singular value, written independently
    of the oracle: sigma <- sigma * (a + b sigma^2 + c sigma^4)."""
    sig = np.array(sig, dtype=np.float64)
    for _ in range(steps):
        s2 = sig * sig
        sig = sig * (a + s2 * (b + c * s2))
    return sig


def svd_closed_form(M, steps, coeffs=(A5, B5, C5), eps=1e-7):
    """U diag(p^T(sigma)) V^T from LAPACK's SVD of M / (||M||_F + eps)."""
    M = np.asarray(M, dtype=np.float64)
    s = np.linalg.norm(M, "fro") + eps
    U, S, Vt = np.linalg.svd(M / s, full_matrices=False)
    return (U * scalar_map(S, steps, *coeffs)) @ Vt


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


CASES = [
    ("c1", lambda: synth.c1().grads[0].double().numpy()),
    ("wide17x40", lambda: synth.random_matrix(17, 40, 11).double().numpy()),
    ("tall50x20", lambda: synth.random_matrix(50, 20, 12).double().numpy()),
    ("square32", lambda: synth.random_matrix(32, 32, 13).double().numpy()),
    ("lowrank24x64", lambda: synth.low_rank(24, 64, 3, 1e-3, 14).double().numpy()),
]


@pytest.mark.parametrize("name,make", CASES)
@pytest.mark.parametrize("steps", [1, 2, 5])
def test_original_space_matches_svd_closed_form(name, make, steps):
    M = make()
    O = oracle.newton_schulz(M, steps)
    assert O.shape == M.shape
    assert rel(O, svd_closed_form(M, steps)) < 1e-12


@pytest.mark.parametrize("name,make", CASES)
def test_gram_space_matches_svd_closed_form(name, make):
    M = make()
    O = oracle.newton_schulz(M, 5, space="gram")
    assert rel(O, svd_closed_form(M, 5)) < 1e-12


@pytest.mark.parametrize("name,make", CASES[:4])
def test_cubic_converges_to_polar_factor(name, make):
    # (1.5, -0.5, 0) maps (0, sqrt(3)) into itself and converges to 1, so the
    # iteration tends to the orthogonal polar factor, computed here by scipy.
    M = make()
    O = oracle.newton_schulz(M, 60, coeffs=oracle.CUBIC)
    side = "right"
    U, _ = scipy.linalg.polar(M, side=side)
    assert rel(O, U) < 1e-10


@pytest.mark.parametrize("shape", [(6, 9), (9, 6), (16, 16), (3, 40)])
@pytest.mark.parametrize("steps", [1, 2, 3, 5, 10])
def test_gram_and_original_agree(shape, steps):
    M = synth.random_matrix(*shape, seed=100 + steps).double().numpy()
    Og = oracle.newton_schulz(M, steps, space="gram")
    Oo = oracle.newton_schulz(M, steps, space="original")
    # fp64 rounding is amplified by up to a^T (a = 3.4445) in small singular
    # directions: 2e-12 was seen at T = 10, so allow 1e-10 there.
    assert rel(Og, Oo) < (1e-12 if steps <= 5 else 1e-10)


def test_gram_intermediates_are_gram_matrices_of_the_iterates():
    # G_k must equal X_k X_k^T where X_k is the k-th original-space iterate,
    # and Q X0 must equal X_T: this pins the recurrence G_{k+1} = P G P.
    M = synth.random_matrix(12, 30, 7).double().numpy()
    X0, _ = oracle.frob_normalize(M)
    T = 4
    g = oracle.ns_gram(X0, T)
    for k in range(T):
        Xk = oracle.ns_original(X0, k)
        assert rel(g["G"][k], Xk @ Xk.T) < 1e-12
    assert rel(g["Q"] @ X0, oracle.ns_original(X0, T)) < 1e-12
    # G0 by brute-force dot products
    G0 = np.array([[sum(X0[i, t] * X0[j, t] for t in range(30)) for j in range(12)]
                   for i in range(12)])
    assert rel(g["G0"], G0) < 1e-14


def test_singular_values_lie_in_band_of_the_map():
    M = synth.c1().grads[0].double().numpy()
    O = oracle.newton_schulz(M, 5)
    s_in = np.linalg.svd(M / (np.linalg.norm(M) + 1e-7), compute_uv=False)
    s_out = np.linalg.svd(O, compute_uv=False)
    grid = np.linspace(s_in.min(), s_in.max(), 200001)
    img = scalar_map(grid, 5)
    assert s_out.min() >= img.min() - 1e-9
    assert s_out.max() <= img.max() + 1e-9
    # Over all of (0, 1] the quintic with five steps never exceeds ~1.2024.
    glob = scalar_map(np.linspace(1e-6, 1.0, 400001), 5).max()
    assert 1.20 < glob < 1.21
    assert s_out.max() <= glob
    # each output singular value is the map of the matching input one
    assert np.allclose(np.sort(s_out), np.sort(scalar_map(s_in, 5)), rtol=1e-11, atol=1e-12)


def test_transpose_equivariance():
    M = synth.random_matrix(20, 33, 21).double().numpy()
    assert rel(oracle.newton_schulz(M.T, 5), oracle.newton_schulz(M, 5).T) < 1e-14


def test_orthogonal_equivariance():
    M = synth.random_matrix(10, 14, 22).double().numpy()
    rng = np.random.default_rng(5)
    U, _ = np.linalg.qr(rng.standard_normal((10, 10)))
    V, _ = np.linalg.qr(rng.standard_normal((14, 14)))
    lhs = oracle.newton_schulz(U @ M @ V, 5)
    rhs = U @ oracle.newton_schulz(M, 5) @ V
    assert rel(lhs, rhs) < 1e-12


def test_scale_invariance():
    M = synth.random_matrix(16, 24, 23).double().numpy()
    assert rel(oracle.newton_schulz(3.7 * M, 5), oracle.newton_schulz(M, 5)) < 1e-6


def test_diagonal_reduces_to_scalar_map():
    d = np.array([3.0, 1.0, 0.5, 0.25])
    M = np.zeros((4, 7))
    M[np.arange(4), np.arange(4)] = d
    s = np.sqrt(np.sum(d * d)) + 1e-7
    O = oracle.newton_schulz(M, 5)
    E = np.zeros_like(M)
    E[np.arange(4), np.arange(4)] = scalar_map(d / s, 5)
    assert np.max(np.abs(O - E)) < 1e-14


@pytest.mark.parametrize("shape", [(1, 300), (300, 1), (1, 1)])
def test_single_row_or_column_reduces_to_scalar_map(shape):
    """A 1 x n (or n x 1) matrix has one singular value, |x| / (|x| + eps):
    O is x / |x| times the scalar map of it, whichever side is short."""
    x = np.random.default_rng(12).standard_normal(shape)
    nx = np.linalg.norm(x)
    O = oracle.newton_schulz(x, 5)
    assert np.max(np.abs(O - x / nx * scalar_map(np.array([nx / (nx + 1e-7)]), 5)[0])) < 1e-14


def test_worked_example_by_hand():
    # M = [[3,0,0],[0,4,0]]: ||M||_F = 5, singular values 0.6 and 0.8 after
    # normalisation.  One quintic step by hand:
    #   0.6: 3.4445*0.6 - 4.775*0.216 + 2.0315*0.07776 = 1.19326944
    #   0.8: 3.4445*0.8 - 4.775*0.512 + 2.0315*0.32768 = 0.97648192
    M = np.array([[3.0, 0.0, 0.0], [0.0, 4.0, 0.0]])
    O = oracle.newton_schulz(M, 1)
    assert abs(O[0, 0] - 1.19326944) < 1e-6
    assert abs(O[1, 1] - 0.97648192) < 1e-6
    assert np.max(np.abs(O - np.diag(np.diag(O[:, :2])) @ np.eye(2, 3))) == 0.0


def test_zero_input_gives_zero():
    O = oracle.newton_schulz(np.zeros((8, 12)), 5)
    assert np.all(O == 0)


def test_steps_zero_returns_normalised_input():
    M = synth.random_matrix(5, 9, 3).double().numpy()
    O = oracle.newton_schulz(M, 0)
    assert rel(O, M / (np.linalg.norm(M) + 1e-7)) < 1e-15


def test_momentum_from_zero_state_and_dampening_equivalence():
    g = synth.random_matrix(6, 10, 4, dtype=torch.bfloat16)
    M = oracle.momentum_update(np.zeros((6, 10)), g, 0.95)
    assert np.array_equal(M, g.double().numpy())
    M2 = oracle.momentum_update(M, g, 0.95)
    assert np.allclose(M2, 1.95 * g.double().numpy(), rtol=1e-15, atol=0)
    # a dampened momentum (1-beta)M from a zero state gives the same NS output
    assert rel(oracle.newton_schulz(0.05 * M, 5), oracle.newton_schulz(M, 5)) < 1e-6


def test_muon_update_applies_minus_lr_times_O():
    g = synth.random_matrix(8, 16, 5)
    W = synth.random_matrix(8, 16, 6)
    Wn, Mn, O = oracle.muon_update(W, g, np.zeros((8, 16)), 0.95, 0.02, 5)
    assert rel(Wn, W.double().numpy() - 0.02 * svd_closed_form(g.double().numpy(), 5)) < 1e-12


def test_bf16_round_matches_torch_cast_on_fp32_values():
    x = torch.randn(100000, generator=torch.Generator().manual_seed(9)) * 3
    ties = torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130, 3.0e38])
    x = torch.cat([x, ties])
    ref = x.to(torch.bfloat16).double().numpy()
    got = oracle.bf16_round(x.double().numpy())
    assert np.array_equal(got, ref)


def test_bucket_order_small_example():
    shapes = [(4, 8), (8, 4), (2, 2), (4, 8), (3, 5)]
    assert oracle.bucket_order(shapes) == [((2, 2), [2]), ((3, 5), [4]), ((4, 8), [0, 1, 3])]


def _mutant_original(X0, steps, coeffs, mutation):
    """A copy of the original-space iteration with one planted slip."""
    a, b, c = coeffs
    X = np.array(X0, dtype=np.float64)
    for _ in range(steps):
        A = X.T @ X if mutation == "gram_side" else X @ X.T
        if mutation == "gram_side":  # X^T X multiplied from the left (square X)
            X = a * X + (b * A + c * (A @ A)) @ X
        elif mutation == "drop_c":
            X = a * X + (b * A) @ X
        elif mutation == "sign_b":
            X = a * X + (-b * A + c * (A @ A)) @ X
        elif mutation == "no_cube":
            X = a * X + (b * A + c * A) @ X
    return X


@pytest.mark.parametrize("mutation", ["gram_side", "drop_c", "sign_b", "no_cube"])
def test_planted_slips_fail_the_svd_pin(mutation):
    # The closed-form pin must be sensitive to each of these mistakes.
    M = synth.random_matrix(24, 24, 31).double().numpy()
    X0 = M / (np.linalg.norm(M) + 1e-7)
    bad = _mutant_original(X0, 5, (A5, B5, C5), mutation)
    assert rel(bad, svd_closed_form(M, 5)) > 1e-3
    good = oracle.ns_original(X0, 5)
    assert rel(good, svd_closed_form(M, 5)) < 1e-12


def test_golden_c1_fixture():
    """tests/golden/c1.json: SHA-256 of the seeded c1 input and a summary of
    the oracle's output for it (written by tests/golden/make_golden.py, which
    calls only synth/ and oracle/)."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "c1.json")
    gold = json.load(open(path))
    g = synth.c1().grads[0]
    assert synth.sha256_of(g) == gold["input_sha256"]
    O = oracle.newton_schulz(g.double().numpy(), gold["steps"])
    assert abs(np.linalg.norm(O) - gold["O_fro"]) < 1e-12
    assert np.allclose(O.ravel()[:8], gold["O_first8"], rtol=0, atol=1e-14)
    sv = np.linalg.svd(O, compute_uv=False)
    assert abs(sv.min() - gold["O_sigma_min"]) < 1e-12
    assert abs(sv.max() - gold["O_sigma_max"]) < 1e-12
