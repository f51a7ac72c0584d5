"""Plain fp64 CPU oracle of the AdamW step on the non-matrix tail
(test infrastructure only: imported by ``tests/`` and the CPU-baseline leg
of ``bench.py``; the library never calls it and shares no code with it).

MatrixFSDP technical summary (gist.science 2607.05895), "Metodologia" §1:
1-D vectors and other non-matrix tensors form a tail that one owner updates
with standard AdamW.  The pages give no formula.  The reading here is AdamW
with decoupled weight decay, the usual library form:

    p <- p (1 - lr wd)
    m <- b1 m + (1 - b1) g
    v <- b2 v + (1 - b2) g^2
    p <- p - lr / (1 - b1^t) * m / (sqrt(v) / sqrt(1 - b2^t) + eps)

Pinned in ``tests/test_adamw.py`` by closed forms (constant gradient: the
bias-corrected moments equal g and g^2 exactly at every step; zero gradient:
pure exponential decay) and by torch.optim.AdamW in float64.
"""
from __future__ import annotations

import numpy as np


def adamw_step(p, g, m, v, lr, beta1, beta2, eps, weight_decay, step):
    """One step on one tensor; returns (p, m, v) in float64."""
    p = np.asarray(p, dtype=np.float64) * (1.0 - lr * weight_decay)
    g = np.asarray(g, dtype=np.float64)
    m = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    p = p - (lr / bc1) * m / (np.sqrt(v) / np.sqrt(bc2) + eps)
    return p, m, v
