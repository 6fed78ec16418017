"""Oracle for the FP8 path: per-tensor scaled E4M3 quantization and the
quantize → GEMM → dequantize product (numpy).

Test infrastructure: see the package docstring.

[Troverld] §II.III names an "FP8 fused kernel" (quantize + compute +
dequantize) among the token-wise operators, and [Grasp-TP] §6 asks for
all-reduces of FP8 buffers; neither page gives a format or a scaling rule.
The plainest reading, taken here:

* format E4M3: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
  normal values (1 + m/8)·2^(e−7) for e = 1..15 except the all-ones code
  S.1111.111 (NaN), subnormals (m/8)·2^−6 for e = 0; largest finite value
  1.75·2^8 = 448, no infinities;
* per-tensor scale s = 448 / amax(|x|) in fp32 (s = 1 when amax = 0), codes
  q = round-to-nearest-even(x·s) with the product x·s rounded to fp32 first
  and values beyond ±448 saturated to ±448;
* a GEMM of two quantized operands accumulates decode(qa)·decode(qb) and
  divides by sa·sb.

Pins (tests/test_oracle_fp8.py): decoding all 254 finite codes gives the
format's values (the table written from the definition above, and
monotone); every finite value (−0 included) encodes to its own code; halfway
points go to the even code; tiny negatives keep their sign; saturation;
scale and amax on small hand-worked tensors.
"""

import numpy as np

E4M3_MAX = 448.0


def e4m3_value(code):
    """The value of one E4M3 code (int 0..255); NaN for S.1111.111."""
    code = int(code)
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_FINITE = np.array([c for c in range(256) if not (c & 0x7F) == 0x7F],
                   dtype=np.int64)
_VALUES = np.array([e4m3_value(c) for c in _FINITE])
# the non-negative finite codes in increasing value (0x00 … 0x7E)
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = np.array([e4m3_value(c) for c in _POS_CODES])


def e4m3_decode(codes):
    """Values of an array of codes (uint8), as float64."""
    table = np.array([e4m3_value(c) for c in range(256)])
    return table[np.asarray(codes, dtype=np.int64)]


def e4m3_encode(x):
    """Round-to-nearest-even E4M3 codes (uint8) of float values, saturating
    finite values beyond ±448 to ±448; negative values that round to zero
    give −0 (0x80).  Input must be finite."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # the neighbours below and above |x| among the non-negative values
    hi = np.searchsorted(_POS_VALUES, a, side="left")      # first value ≥ a
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    vlo, vhi = _POS_VALUES[lo], _POS_VALUES[hi]
    exact = vhi == a
    dlo, dhi = a - vlo, vhi - a
    # nearer neighbour; on a tie the even code (mantissa LSB 0)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((_POS_CODES[hi] & 1) == 0))
    mag = np.where(exact, _POS_CODES[hi],
                   np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]))
    # the sign is kept when the magnitude rounds to 0: S.0000.000 with S = 1
    # is −0, as rounding keeps the sign of the value rounded
    sign = np.where(np.signbit(x), 0x80, 0)
    return (mag | sign).astype(np.uint8)


def quantize(x):
    """Per-tensor scaled E4M3 codes of a tensor given exactly (bf16 values).

    Returns (codes uint8, scale float32, amax float32): scale = 448 / amax
    computed in fp32, codes = encode(fp32(x · scale)).
    """
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0.0)
    scale = np.float32(1.0) if amax == 0 else np.float32(E4M3_MAX) / amax
    prod = (x32 * scale).astype(np.float32)
    return e4m3_encode(prod), np.float32(scale), amax


def dequantize(codes, scale):
    return e4m3_decode(codes) / np.float64(scale)


def gemm(qa, sa, qb, sb):
    """C = (decode(qa)·decode(qb)ᵀ) / (sa·sb) in float64; qa [M, K], qb [N, K]."""
    return (e4m3_decode(qa) @ e4m3_decode(qb).T) / (np.float64(sa) *
                                                   np.float64(sb))


def round_bf16(x):
    """x rounded to fp32, then to bf16 (the top 16 bits of the fp32 pattern,
    round to nearest even), returned as float64; finite inputs."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def mlp_forward(X, W1, W2, *, act="swiglu", b1=None, b2=None, R=None, p=0.0,
                seed=0):
    """The MLP forward on the FP8 path: the first projection on quantized X
    and W1 (W1 as one tensor, gate and up rows together), bias and
    activation in fp64, A stored in bf16 then quantized, the second
    projection on quantized A and W2, bias, dropout, residual.  Returns the
    dict of ``oracle.mlp_forward`` (saved G/U/A or H/A in fp64, Z, Out) plus
    the four scales."""
    from .mlp import _activation, _output
    qx, sx, _ = quantize(X)
    qw1, sw1, _ = quantize(W1)
    saved = _activation(dequantize(qx, sx), dequantize(qw1, sw1), b1, act)
    qa, sa, _ = quantize(round_bf16(saved["A"]))
    qw2, sw2, _ = quantize(W2)
    Z = dequantize(qa, sa) @ dequantize(qw2, sw2).T
    out = dict(saved)
    out["Z"] = Z
    out["Out"] = _output(Z, b2, R, p, seed)
    out["scales"] = (sx, sw1, sa, sw2)
    return out


def attention_forward(X, Wq, Wk, Wv, Wo, *, b, s, n_q, n_kv, d, causal=True,
                      bo=None, R=None):
    """The attention block's forward on the FP8 path: the Q, K, V
    projections on quantized X and Wq, Wk, Wv (one scale per tensor), the
    attention core in fp64 on those products, O stored in bf16 then
    quantized, the output projection on quantized O and Wo, bias, residual.
    Returns the dict of ``oracle.attention_forward`` (Q, K, V, O, LSE, Z,
    Out) plus the six scales."""
    from .attention import attention_core
    qx, sx, _ = quantize(X)
    xd = dequantize(qx, sx)
    proj, scales = [], [sx]
    for W in (Wq, Wk, Wv):
        qw, sw, _ = quantize(W)
        proj.append(xd @ dequantize(qw, sw).T)
        scales.append(sw)
    Q, K, V = proj
    O, LSE = attention_core(Q, K, V, b=b, s=s, n_q=n_q, n_kv=n_kv, d=d,
                            causal=causal)
    qo, so, _ = quantize(round_bf16(O))
    qwo, swo, _ = quantize(Wo)
    Z = dequantize(qo, so) @ dequantize(qwo, swo).T
    Out = Z if bo is None else Z + np.asarray(bo, np.float64)
    if R is not None:
        Out = Out + np.asarray(R, np.float64)
    return {"Out": Out, "Q": Q, "K": K, "V": V, "O": O, "LSE": LSE, "Z": Z,
            "scales": tuple(scales) + (so, swo)}
