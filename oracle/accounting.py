"""Oracle for the communication-volume and FLOP accounting (exact integers).

Test infrastructure: see the package docstring.  Python integers throughout,
so nothing overflows and every value is exact.

Communication ([Grasp-TP] §5; [Troverld] §II.II TP row; [adu-TP]
张量并行的通信开销):

* Each tensor-parallel all-reduce carries a logical payload of T·h·δ bytes,
  T = b·s tokens, δ bytes per element (FP32 4, BF16 2: [Troverld] §O.I).
* A ring all-reduce (reduce-scatter then all-gather) moves 2(n−1)/n of the
  payload per rank ([Grasp-TP] §5); kept as an exact reduced fraction.
* [Troverld] §II.II drops the (n−1)/n factor and counts 2·δ·b·S·H per
  all-reduce, 4·δbSH per block, 8·δbSH per layer.
* Counts: an MLP or an attention block has one reduction in forward (g after
  the row-parallel projection) and one in backward (f at the input gradient);
  a layer has four ([Grasp-TP] §5 list, [adu-TP]).

FLOPs ([hjcheng-TP] MLP / Attention 单卡forward, 单卡backward, TP forward):

* GeLU MLP: two GEMMs of 2·T·h·f each → forward 4·T·h·f, backward twice that.
  At f = 4h these are the page's 16·BS·d² and 32·BS·d².
* SwiGLU MLP: three GEMMs → forward 6·T·h·f, backward 12·T·h·f (the same
  2-GEMMs-per-forward-GEMM rule applied to the gate/up/down projections).
* Attention: projections 2·T·h·(n_q + 2·n_kv)·d + 2·T·n_q·d·h, score and
  value products 4·b·n_q·d·C with C = s² for the full mask ([hjcheng-TP]
  table: 8BSd² + 4BS²d for MHA) or C = s(s+1)/2 for the causal mask
  (unmasked pairs only).  Backward is twice forward, as the page concludes
  (flash recompute is not counted).
* A layer is attention + MLP (the norms are not counted).
"""

from fractions import Fraction

DTYPE_BYTES = {"f32": 4, "bf16": 2}
_REDUCTIONS = {"mlp": (1, 1), "attn": (1, 1), "layer": (2, 2)}


def comm_report(scope, T, h, n, dtype):
    """Exact TP communication figures for one microbatch of one scope."""
    delta = DTYPE_BYTES[dtype]
    fwd, bwd = _REDUCTIONS[scope]
    payload = T * h * delta
    ring = Fraction(2 * (n - 1) * payload, n)
    count = fwd + bwd
    return {
        "reductions_fwd": fwd,
        "reductions_bwd": bwd,
        "payload_bytes": payload,
        "ring_bytes": ring,                # per rank per reduction
        "page2_bytes": 2 * payload,        # 2·δ·b·S·H per reduction
        "total_payload": count * payload,
        "total_ring": count * ring,
        "total_page2": count * 2 * payload,
    }


def mlp_flops(T, h, f, act):
    per_gemm = 2 * T * h * f
    gemms = 2 if act == "gelu" else 3
    return gemms * per_gemm, 2 * gemms * per_gemm


def attn_flops(b, s, h, n_q, n_kv, d, causal=True):
    T = b * s
    proj = 2 * T * h * (n_q + 2 * n_kv) * d + 2 * T * n_q * d * h
    pairs = s * (s + 1) // 2 if causal else s * s
    core = 4 * b * n_q * d * pairs
    fwd = proj + core
    return fwd, 2 * fwd


def layer_flops(b, s, h, f, n_q, n_kv, d, act="swiglu", causal=True):
    af, ab = attn_flops(b, s, h, n_q, n_kv, d, causal)
    mf, mb = mlp_flops(b * s, h, f, act)
    return af + mf, ab + mb
