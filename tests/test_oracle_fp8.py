"""Pins of the FP8 oracle (oracle/fp8.py): the E4M3 format from its
definition, round-to-nearest-even with saturation, and the per-tensor scaled
quantization and GEMM."""

import math
import os

import numpy as np

import oracle
import pytest

from oracle import fp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_values.txt")


def golden():
    out = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            c, v = line.split()
            out.append((int(c, 16), float(v)))
    return out


def test_decode_matches_the_format_table():
    for code, value in golden():
        got = fp8.e4m3_value(code)
        if math.isnan(value):
            assert math.isnan(got)
        else:
            assert got == value and math.copysign(1, got) == math.copysign(1, value)


def test_finite_codes_are_monotone_and_round_trip():
    pos = [fp8.e4m3_value(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(pos, pos[1:]))
    assert pos[-1] == 448.0 and pos[1] == 2.0 ** -9
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])
    vals = fp8.e4m3_decode(codes)
    back = fp8.e4m3_encode(vals)
    assert (back == codes).all()      # −0 included: it keeps its sign


def test_round_to_nearest_even_and_saturation():
    # halfway between 1.0 (0x38, even) and 1.125 (0x39): the even code
    assert fp8.e4m3_encode([1.0625])[0] == 0x38
    # halfway between 1.125 (0x39) and 1.25 (0x3a): 0x3a
    assert fp8.e4m3_encode([1.1875])[0] == 0x3A
    # just above a halfway point rounds up; just below rounds down
    assert fp8.e4m3_encode([1.0626])[0] == 0x39
    assert fp8.e4m3_encode([1.0624])[0] == 0x38
    # subnormal range: 2^-10 is halfway between 0 and 2^-9 → 0 (even)
    assert fp8.e4m3_encode([2.0 ** -10])[0] == 0x00
    assert fp8.e4m3_encode([3 * 2.0 ** -10])[0] == 0x02
    # beyond the largest finite value: saturate to ±448
    assert fp8.e4m3_encode([1000.0])[0] == 0x7E
    assert fp8.e4m3_encode([-465.0])[0] == 0xFE
    assert fp8.e4m3_encode([-1.0])[0] == 0xB8
    # a negative value that rounds to zero keeps its sign: −0
    assert fp8.e4m3_encode([-1e-9])[0] == 0x80
    assert fp8.e4m3_encode([1e-9])[0] == 0x00


def test_quantize_scale_and_codes():
    x = np.array([[0.5, -2.0], [1.0, 0.25]], dtype=np.float32)
    q, s, amax = fp8.quantize(x)
    assert amax == np.float32(2.0)
    assert s == np.float32(224.0)                 # 448 / 2
    # 0.5·224 = 112 = 1.75·2^6 → 0x6e; −2·224 = −448 → 0xfe;
    # 224 = 1.75·2^7 → 0x76; 0.25·224 = 56 = 1.75·2^5 → 0x66
    assert q.tolist() == [[0x6E, 0xFE], [0x76, 0x66]]
    q0, s0, a0 = fp8.quantize(np.zeros((2, 3), dtype=np.float32))
    assert a0 == 0 and s0 == 1 and (q0 == 0).all()


def test_gemm_of_quantized_operands():
    # exactly representable operands: the quantized GEMM is the plain GEMM
    rng = np.random.default_rng(3)
    A = rng.integers(-7, 8, size=(5, 16)).astype(np.float32) / 4
    B = rng.integers(-7, 8, size=(3, 16)).astype(np.float32) / 4
    qa, sa, _ = fp8.quantize(A)
    qb, sb, _ = fp8.quantize(B)
    C = fp8.gemm(qa, sa, qb, sb)
    err = np.abs(C - A.astype(np.float64) @ B.T.astype(np.float64)).max()
    # each operand is within one E4M3 rounding (≤ 2^-4 relative) of its value
    assert err <= 0.15 * np.abs(A).max() * np.abs(B).max() * 16
    # and dequantize(quantize(x)) stays within half an E4M3 step of x
    d = fp8.dequantize(qa, sa)
    assert (np.abs(d - A) <= np.abs(A) * 2.0 ** -4 + 2.0 ** -10).all()


def test_round_bf16_is_round_to_nearest_even():
    # 1 + 2^-8 is halfway between bf16 neighbours 1 and 1 + 2^-7: even → 1
    assert fp8.round_bf16([1.0 + 2.0 ** -8])[0] == 1.0
    assert fp8.round_bf16([1.0 + 3 * 2.0 ** -8])[0] == 1.0 + 2.0 ** -6
    assert fp8.round_bf16([1.0 + 2.0 ** -8 + 2.0 ** -20])[0] == 1.0 + 2.0 ** -7
    assert fp8.round_bf16([-3.0])[0] == -3.0


def test_fp8_mlp_forward_is_the_mlp_on_dequantized_operands():
    # with operands already exact in E4M3 (after scaling) and a bf16-exact A,
    # the FP8 path equals the plain MLP on the dequantized tensors
    import oracle
    rng = np.random.default_rng(5)
    X = rng.integers(-8, 9, size=(6, 32)) / 8.0
    W1 = rng.integers(-8, 9, size=(2 * 16, 32)) / 64.0
    W2 = rng.integers(-8, 9, size=(32, 16)) / 64.0
    o = fp8.mlp_forward(X, W1, W2, act="swiglu")
    sx, sw1, sa, sw2 = o["scales"]
    ref = oracle.mlp_forward(fp8.dequantize(fp8.quantize(X)[0], sx),
                             fp8.dequantize(fp8.quantize(W1)[0], sw1), W2,
                             act="swiglu")
    assert np.allclose(o["G"], ref["G"], rtol=0, atol=1e-12)
    assert np.allclose(o["U"], ref["U"], rtol=0, atol=1e-12)
    # the second projection uses A rounded to bf16, then quantized: within
    # one E4M3 step of A (relative 2^-4) per element
    d = np.abs(o["Z"] - ref["Z"]).max()
    assert d <= 2.0 ** -3 * np.abs(ref["A"]).sum(axis=1).max() * np.abs(W2).max()


def test_fp8_attention_forward_is_attention_on_dequantized_operands():
    # X and the weights take values ±2^-k·amax (exact in E4M3 after the
    # per-tensor scale), so the projections and the attention core equal the
    # plain oracle's exactly; the output projection quantizes O (bf16-rounded)
    # and is within one E4M3 step of it per element
    import oracle
    rng = np.random.default_rng(6)
    b, s, n_q, n_kv, d, h = 2, 5, 4, 2, 8, 16
    pick = lambda shape, unit: (rng.choice([-1.0, -0.5, -0.25, 0.0, 0.25, 0.5,
                                            1.0], size=shape) * unit)
    X = pick((b * s, h), 1.0)
    X[0, 0] = 1.0                                  # amax exactly 1
    Wq, Wk, Wv = (pick((n * d, h), 1 / 16) for n in (n_q, n_kv, n_kv))
    Wo = pick((h, n_q * d), 1 / 16)
    for W in (Wq, Wk, Wv, Wo):
        W[0, 0] = 1 / 16
    kw = dict(b=b, s=s, n_q=n_q, n_kv=n_kv, d=d, causal=True)
    o = fp8.attention_forward(X, Wq, Wk, Wv, Wo, **kw)
    ref = oracle.attention_forward(X, Wq, Wk, Wv, Wo, **kw)
    for k in ("Q", "K", "V", "O", "LSE"):
        assert np.array_equal(o[k], ref[k]), k
    assert o["scales"][0] == np.float32(448.0)
    bound = 2.0 ** -3 * np.abs(ref["O"]).sum(axis=1).max() * np.abs(Wo).max()
    assert np.abs(o["Z"] - ref["Z"]).max() <= bound
    assert np.abs(o["Z"] - ref["Z"]).max() > 0     # O is not exact in E4M3


def test_fp8_attention_forward_bias_and_residual():
    rng = np.random.default_rng(7)
    b, s, n_q, n_kv, d, h = 1, 4, 2, 1, 8, 8
    X = rng.standard_normal((b * s, h))
    Wq, Wk, Wv = (rng.standard_normal((n * d, h)) * 0.1 for n in (n_q, n_kv, n_kv))
    Wo = rng.standard_normal((h, n_q * d)) * 0.1
    bo, R = rng.standard_normal(h), rng.standard_normal((b * s, h))
    kw = dict(b=b, s=s, n_q=n_q, n_kv=n_kv, d=d)
    plain = fp8.attention_forward(X, Wq, Wk, Wv, Wo, **kw)
    full = fp8.attention_forward(X, Wq, Wk, Wv, Wo, bo=bo, R=R, **kw)
    assert np.array_equal(full["Out"], plain["Z"] + bo + R)


# ---------------------------------------------------------------------------
# The FP8 layer (oracle.layer_forward(fp8=True)) on a structured tiny layer
# whose every step has a closed form.  b = 1, s = 2, h = d = h_ffn = 8, one q
# and one kv head, γ1 = γ2 = 1, x = c·σ with sign rows σ0 = (+1)^8 and
# σ1 = (+1)^4 (−1)^4 (σ0·σ1 = 0, both +1 in column 0).
#  * Wq = Wk = 64·I: the two tokens' scores differ by ~1.1e4 ≫ 745, so the
#    causal softmax is exactly one-hot on the diagonal in fp64 and O = V.
#  * Wv = I, Wo = w·I (w a power of two): O and the attention output keep
#    the sign pattern, so each quantized activation has one magnitude a: its
#    E4M3 codes are ±448 and it dequantizes to D(a) = 448 / s(a) with the
#    fp32 scale s(a) = fp32(448 / a).  Every weight is a power of two or 0,
#    which its per-tensor scale maps exactly.
#  * W1 = [64 on column 0 of every gate row; I for the up rows]: G = 64·D2
#    (≥ 37, where σ(G) = 1 in fp64, so SiLU(G) = G), U = D2·σ,
#    A = 64·D2²·σ.  W2 = 2⁻⁶·I.
# With m̂ = bf16(c/√(c² + ε)) the stored first norm output, D1 = D(m̂),
# r1 = c + w·D1 (x1 = r1·σ), m̂2 = bf16(r1/√(r1² + ε)) the stored second norm
# output, D2 = D(m̂2) and D3 = D(64·bf16(D2²)):
#     Out = σ·(r1 + 2⁻⁶·D3).
# Quantizing a norm output before its bf16 rounding would put the unrounded
# magnitude in place of m̂ or m̂2 (ε > 0 makes them differ by ~1e-3), and
# feeding the MLP any tensor other than the stored second norm output breaks
# the closed form.
# ---------------------------------------------------------------------------
def _dequant_uniform(a):
    """The value a tensor of one magnitude a (exact in fp32) dequantizes to."""
    return 448.0 / float(np.float32(448.0) / np.float32(a))


def _structured_layer(c, w, eps, round_norms=True):
    from oracle.fp8 import round_bf16
    rnd = (lambda v: float(round_bf16(v))) if round_norms else float
    h = 8
    sig = np.array([[1.0] * 8, [1.0] * 4 + [-1.0] * 4])
    I8 = np.eye(h)
    Wg = np.zeros((h, h))
    Wg[:, 0] = 64.0
    P = {"g1": np.ones(h), "g2": np.ones(h), "Wq": 64.0 * I8,
         "Wk": 64.0 * I8, "Wv": I8.copy(), "Wo": w * I8,
         "W1": np.concatenate([Wg, I8]), "W2": 2.0 ** -6 * I8}
    x = c * sig
    r1 = c + w * _dequant_uniform(rnd(c / np.sqrt(c * c + eps)))
    d2 = _dequant_uniform(rnd(r1 / np.sqrt(r1 * r1 + eps)))
    d3 = _dequant_uniform(64.0 * float(round_bf16(d2 * d2)))
    closed = sig * (r1 + 2.0 ** -6 * d3)
    shp = dict(b=1, s=2, n_q=1, n_kv=1, d=8, eps=eps)
    return x, P, shp, closed


def test_fp8_layer_equals_the_plain_layer_when_every_quantization_is_exact():
    # ε = 0: every norm output is ±1 (exact in bf16 and E4M3), every weight a
    # power of two or 0, so the FP8 layer is the plain layer: Out = (c+w+1)σ
    x, P, shp, closed = _structured_layer(c=1.0, w=2.0, eps=0.0)
    f8 = oracle.layer_forward(x, P, fp8=True, **shp)
    plain = oracle.layer_forward(x, P, **shp)
    np.testing.assert_allclose(f8["Out"], plain["Out"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(f8["Out"], closed, rtol=0, atol=1e-12)
    np.testing.assert_allclose(closed[:, 0], 4.0)
    # the first block quantized the ±1 norm output: scale 448 / 1
    assert f8["attn"]["scales"][0] == np.float32(448.0)


@pytest.mark.parametrize("c,w,eps", [(1.0, 2.0, 1e-2), (2.0, 0.5, 0.3),
                                     (0.5, 4.0, 1e-3)])
def test_fp8_layer_quantizes_each_norm_output_as_stored_in_bf16(c, w, eps):
    from oracle.fp8 import round_bf16
    x, P, shp, closed = _structured_layer(c, w, eps)
    f8 = oracle.layer_forward(x, P, fp8=True, **shp)
    np.testing.assert_allclose(f8["Out"], closed, rtol=0, atol=1e-12)
    # with the norm outputs quantized unrounded the closed form moves by far
    # more than the tolerance
    _, _, _, unrounded = _structured_layer(c, w, eps, round_norms=False)
    assert np.abs(unrounded - closed).max() > 1e-4
    # per-tensor scale of the quantized first norm output: 448 / bf16(amax)
    m_hat = float(round_bf16(c / np.sqrt(c * c + eps)))
    assert f8["attn"]["scales"][0] == np.float32(448.0) / np.float32(m_hat)
