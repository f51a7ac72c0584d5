"""Plain fp64 CPU oracle of the owner-side Muon update.

TEST INFRASTRUCTURE ONLY.  This file is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``; the
CUDA library never imports, links or calls it, and it shares no code, table or
constant generator with the library.  Inputs come from the seeded generators
in ``synth/`` (random numbers only).

What it computes, step by step, in the order the pages describe it:

* DMuon technical summary (gist.science 2606.27153), §1 "Definizione del
  Problema": Muon applies Newton-Schulz (NS) iterations to the
  momentum-aggregated gradient of each weight matrix; the iteration needs the
  product X X^T of the whole matrix.
* same page, §2.2 "Iterazione Gram Newton-Schulz Efficiente": the iteration can
  instead be run in the m x m Gram space G = X X^T (m < n), G is symmetric.
* same page, §5: the Gram formulation does not change the update rule, so the
  Gram recurrence must reproduce the original-space result exactly (up to
  rounding).

Readings where the pages are silent:

* momentum is heavy-ball, M <- beta*M + G (no Nesterov, no dampening);
* X0 = X / (||X||_F + eps), eps = 1e-7;
* the matrix is oriented so the short side comes first (transpose if m > n);
* one coefficient triple (a, b, c) is used for every step, the iteration being
  X <- a X + b (X X^T) X + c (X X^T)^2 X;
* the apply is W <- W - lr * O, no shape factor and no weight decay.

Parity: every function here is pinned by ``tests/test_oracle_pins.py`` against
an SVD closed form, a library polar decomposition, invariants and brute force.
"""
from __future__ import annotations

import numpy as np

QUINTIC = (3.4445, -4.7750, 2.0315)
CUBIC = (1.5, -0.5, 0.0)
EPS = 1e-7


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor: exact widening of its stored values
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def momentum_update(mom, grad, beta):
    """M <- beta*M + G in fp64 (heavy-ball reading of "momentum-aggregated
    gradients", DMuon summary §1)."""
    return float(beta) * _f64(mom) + _f64(grad)


def orient(M):
    """Short side first: return (X, transposed) with X = M^T when m > n, so the
    Gram matrix X X^T is the small one (DMuon summary §2.2, which assumes m < n)."""
    M = _f64(M)
    if M.shape[0] > M.shape[1]:
        return M.T.copy(), True
    return M, False


def frob_normalize(X, eps=EPS):
    """X0 = X / s with s = ||X||_F + eps; returns (X0, s)."""
    X = _f64(X)
    s = float(np.sqrt(np.sum(X * X))) + eps
    return X / s, s


def ns_original(X0, steps, coeffs=QUINTIC):
    """Original-space NS: repeat `steps` times A = X X^T ; X <- a X + (b A + c A A) X."""
    a, b, c = (float(v) for v in coeffs)
    X = _f64(X0).copy()
    for _ in range(int(steps)):
        A = X @ X.T
        X = a * X + (b * A + c * (A @ A)) @ X
    return X


def ns_gram(X0, steps, coeffs=QUINTIC):
    """Gram-space NS (DMuon summary §2.2): everything is done on G = X0 X0^T.

    With P_k = a I + b G_k + c G_k^2 every step is X_{k+1} = P_k X_k.  All P_k
    and G_k are polynomials in G_0, so they commute, which gives
    G_{k+1} = X_{k+1} X_{k+1}^T = P_k G_k P_k and X_T = (P_{T-1} ... P_0) X0.
    Returns a dict with the intermediates G0, P (list), Q = P_{T-1}...P_0 and O.
    """
    a, b, c = (float(v) for v in coeffs)
    X0 = _f64(X0)
    s = X0.shape[0]
    I = np.eye(s)
    G = X0 @ X0.T
    out = {"G0": G.copy(), "P": [], "G": [G.copy()]}
    Q = I.copy()
    for k in range(int(steps)):
        P = a * I + b * G + c * (G @ G)
        out["P"].append(P)
        Q = P @ Q
        if k + 1 < steps:
            H = P @ G
            G = P @ H
            out["G"].append(G.copy())
    out["Q"] = Q
    out["O"] = Q @ X0
    return out


def newton_schulz(M, steps, coeffs=QUINTIC, eps=EPS, space="original"):
    """Orient, normalise, iterate, and un-orient.  Returns O with M's shape."""
    X, tr = orient(M)
    X0, _ = frob_normalize(X, eps)
    if space == "original":
        O = ns_original(X0, steps, coeffs)
    elif space == "gram":
        O = ns_gram(X0, steps, coeffs)["O"]
    else:
        raise ValueError(space)
    return O.T.copy() if tr else O


def muon_update(W, grad, mom, beta, lr, steps, coeffs=QUINTIC, eps=EPS):
    """One owner-side Muon step on one matrix.

    Returns (W_new, M_new, O), all fp64: M_new = beta*mom + grad,
    O = NS(M_new), W_new = W - lr * O.
    """
    M = momentum_update(mom, grad, beta)
    O = newton_schulz(M, steps, coeffs, eps)
    return _f64(W) - float(lr) * O, M, O


def bf16_round(x):
    """Round fp64 values to the nearest bfloat16 value, ties to even, in one
    rounding (bfloat16 keeps 8 significant bits and fp32's exponent range).
    Used to form the expected bf16 weight from the fp64 update."""
    x = _f64(x)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    f, e = np.frexp(x[nz])           # x = f * 2**e, 0.5 <= |f| < 1
    e = np.maximum(e, -125)          # below the smallest normal the quantum stays 2**-133
    q = np.ldexp(1.0, e - 8)         # spacing of 8-significant-bit values at this exponent
    out[nz] = np.rint(x[nz] / q) * q  # numpy rint rounds half to even
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out


def bucket_order(shapes):
    """Reference grouping of matrices by shape key (short side, long side):
    buckets in increasing key order, members in input order.  Returns a list
    of ((s, l), [indices]).  Written as a brute-force scan, independent of the
    library's sort."""
    keys = []
    for (m, n) in shapes:
        k = (min(m, n), max(m, n))
        if k not in keys:
            keys.append(k)
    keys.sort()
    return [(k, [i for i, (m, n) in enumerate(shapes) if (min(m, n), max(m, n)) == k])
            for k in keys]
