"""Oracle for RMSNorm, forward and backward (fp64).

Test infrastructure: see the package docstring.

[Troverld] §II.III lists a fused LayerNorm / RMSNorm among the token-wise ops
that tensor parallelism must treat specially, and §III.III allows pre- or
post-norm; no formula is printed.  The standard definition is taken:

    rstd_t = 1 / sqrt(mean_j(x_tj²) + ε),   y_tj = x_tj · rstd_t · γ_j

Backward (chain rule, g = dy ⊙ γ):
    dx_t = rstd_t·g_t − x_t · rstd_t³ · (g_t · x_t) / h,   dγ = Σ_t dy_t ⊙ x_t · rstd_t
plus an optional residual gradient added to dx.

Pins (tests/test_oracle_norm.py): the output of a row has unit RMS when γ = 1
and ε = 0; y is invariant to scaling a row by c > 0 when ε = 0; central finite
differences of dx and dγ.
"""

import numpy as np


def rmsnorm_forward(x, gamma, eps=1e-5):
    x = np.asarray(x, np.float64)
    rstd = 1.0 / np.sqrt((x * x).mean(axis=1) + eps)
    return {"y": x * rstd[:, None] * np.asarray(gamma, np.float64),
            "rstd": rstd}


def rmsnorm_backward(dy, x, gamma, eps=1e-5, dres=None):
    dy = np.asarray(dy, np.float64)
    x = np.asarray(x, np.float64)
    gamma = np.asarray(gamma, np.float64)
    h = x.shape[1]
    rstd = 1.0 / np.sqrt((x * x).mean(axis=1) + eps)
    g = dy * gamma
    dot = (g * x).sum(axis=1)
    dx = rstd[:, None] * g - x * (rstd ** 3 * dot / h)[:, None]
    if dres is not None:
        dx = dx + dres
    dgamma = (dy * x * rstd[:, None]).sum(axis=0)
    return {"dx": dx, "dgamma": dgamma}
