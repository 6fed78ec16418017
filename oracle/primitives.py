"""Elementwise primitives of the oracle (fp64) and the dropout-mask generator.

Test infrastructure: see the package docstring.

* GeLU is named by [hjcheng-TP] (MLP: Out = Dropout(GeLU(X W1) W2)) and by
  [adu-TP] (Y = GELU(XA)) without a formula; the exact form
  0.5·x·(1 + erf(x/√2)) = x·Φ(x) is taken.  Pinned by Φ(±1), Φ(±2) table values
  and by finite differences of ``gelu`` against ``gelu_grad``.
* SiLU appears in [Grasp-TP] §3 (SwiGLU: gate / up / down projections, the
  formula itself missing from the page); SiLU(x) = x·σ(x) is taken.
* The pages give no random-number generator for dropout ([Troverld] §I.III
  draws "Dropout" after the g all-reduce; [hjcheng-TP] 单卡backward gives the
  backward dZ = dOut ⊙ mask / (1 − p)).  The mask here is one splitmix64 stream
  (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014; constants as in Vigna's public-domain splitmix64.c) seeded with
  the dropout seed, one draw per element of the reduced [T, h] output in
  row-major order: draw e (0-based) = mix(seed + (e + 1)·γ).  The top 24 bits
  of the draw are compared with an integer threshold.  Pinned by the published
  first outputs for seed 1234567.
"""

import math

import numpy as np
from scipy.special import erf

_SQRT2 = math.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)

# splitmix64 constants (the golden-ratio increment and the two finaliser
# multipliers of the published generator).
SPLITMIX_GAMMA = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1


def gelu(x):
    """GeLU(x) = x·Φ(x) = 0.5·x·(1 + erf(x/√2)), elementwise, fp64."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + erf(x / _SQRT2))


def gelu_grad(x):
    """d GeLU / dx = Φ(x) + x·φ(x), with φ the standard normal density."""
    x = np.asarray(x, dtype=np.float64)
    cdf = 0.5 * (1.0 + erf(x / _SQRT2))
    pdf = _INV_SQRT_2PI * np.exp(-0.5 * x * x)
    return cdf + x * pdf


def sigmoid(x):
    """Logistic σ(x) = 1 / (1 + e^(−x)), evaluated without overflow."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-x[pos]))
    ex = np.exp(x[~pos])
    out[~pos] = ex / (1.0 + ex)
    return out


def silu(x):
    """SiLU(x) = x·σ(x)."""
    x = np.asarray(x, dtype=np.float64)
    return x * sigmoid(x)


def silu_grad(x):
    """d SiLU / dx = σ(x)·(1 + x·(1 − σ(x)))."""
    x = np.asarray(x, dtype=np.float64)
    s = sigmoid(x)
    return s * (1.0 + x * (1.0 - s))


def splitmix64_mix(z):
    """The splitmix64 output finaliser on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_MIX1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_MIX2)
    return z ^ (z >> np.uint64(31))


def splitmix64_stream(seed, count):
    """First ``count`` outputs of splitmix64 seeded with ``seed``, as Python ints.

    Written with Python integers (not numpy) so that it is an independent
    statement of the generator: state += γ (mod 2^64), then mix the state.
    """
    out = []
    state = seed & _MASK64
    for _ in range(count):
        state = (state + SPLITMIX_GAMMA) & _MASK64
        z = state
        z = ((z ^ (z >> 30)) * _MIX1) & _MASK64
        z = ((z ^ (z >> 27)) * _MIX2) & _MASK64
        out.append(z ^ (z >> 31))
    return out


def dropout_threshold(p):
    """Integer threshold thr = round(p·2^24), ties to even; keep iff draw24 ≥ thr."""
    if not (0.0 <= p < 1.0):
        raise ValueError("dropout probability must lie in [0, 1)")
    return int(round(p * float(1 << 24)))


def dropout_keep(seed, rows, cols, p, row0=0):
    """Boolean keep-mask for rows [row0, row0+rows) of a [*, cols] output.

    Element (t, j) uses draw e = t·cols + j of the splitmix64 stream seeded
    with ``seed``: k = mix(seed + (e + 1)·γ) >> 40 (the top 24 bits); the
    element is kept when k ≥ ``dropout_threshold(p)``.
    """
    thr = dropout_threshold(p)
    t = np.arange(row0, row0 + rows, dtype=np.uint64)[:, None]
    j = np.arange(cols, dtype=np.uint64)[None, :]
    e = t * np.uint64(cols) + j
    with np.errstate(over="ignore"):
        z = np.uint64(seed & _MASK64) + (e + np.uint64(1)) * np.uint64(SPLITMIX_GAMMA)
        k = splitmix64_mix(z) >> np.uint64(40)
    return k >= np.uint64(thr)
