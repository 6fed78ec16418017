"""Error metrics of the GPU-vs-oracle parity tests.

bf16 workloads (fp32 accumulation): per tensor ‖g − o‖_F / ‖o‖_F ≤ 1e-2 and
max|g − o| / rms(o) ≤ 3e-2.  fp32 workloads: max|g − o| / max|o| ≤ 1e-4.
"""

import numpy as np
import torch

BF16_FRO = 1e-2
BF16_MAXRMS = 3e-2
F32_MAXREL = 1e-4


def f64(t):
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def errors(g, o):
    g, o = f64(g), f64(o)
    d = g - o
    fro = np.linalg.norm(d) / max(np.linalg.norm(o), 1e-300)
    rms = np.sqrt(np.mean(o * o)) if o.size else 0.0
    maxrms = np.abs(d).max() / max(rms, 1e-300) if d.size else 0.0
    maxrel = np.abs(d).max() / max(np.abs(o).max(), 1e-300) if d.size else 0.0
    return fro, maxrms, maxrel


def check(g, o, name, dtype="bf16"):
    fro, maxrms, maxrel = errors(g, o)
    if dtype == "f32":
        assert maxrel <= F32_MAXREL, f"{name}: max rel {maxrel:.3e}"
    else:
        assert fro <= BF16_FRO and maxrms <= BF16_MAXRMS, \
            f"{name}: fro {fro:.3e}, max/rms {maxrms:.3e}"
    return fro, maxrms, maxrel
