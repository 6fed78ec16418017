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

Megatron-SP ([Troverld] §III.III): the all-reduce at a block's end becomes a
reduce-scatter to (b, s/N, H), the token-wise work (norm, dropout) runs on
s/N positions per rank, and an all-gather back to (b, s, H) opens the next
block.  In a ring each of the two moves (n−1)/n of the payload per rank, so
together they move what the all-reduce did.

Saved activations ([hjcheng-TP] MLP and Attention, the 激活值 lists for the
single card and for TP): MLP X (BS, d_model), H and A (BS, d_ff / N), the
dropout mask (BS, d_model); attention X, Q, K, V, the score matrix
S (B, h, S, S) and AV, all but X divided by N under TP.  See
``act_memory`` for the readings (GQA, SwiGLU, flash, the layer's norms, SP).

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

DTYPE_BYTES = {"f32": 4, "bf16": 2, "fp8": 1}   # fp8: [Grasp-TP] §6 buffers
_REDUCTIONS = {"mlp": (1, 1), "attn": (1, 1), "layer": (2, 2)}


def comm_report(scope, T, h, n, dtype):
    """Exact TP communication figures for one microbatch of one scope,
    with the Megatron-SP split of each all-reduce position."""
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
        # Megatron-SP: one reduce-scatter and one all-gather per position
        "sp_rs_bytes": Fraction((n - 1) * payload, n),
        "sp_ag_bytes": Fraction((n - 1) * payload, n),
        "sp_reduce_scatters": count,
        "sp_all_gathers": count,
        "sp_total": count * 2 * Fraction((n - 1) * payload, n),
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


def act_memory(b, s, h, h_ffn, n_q, n_kv, d, n, dtype="bf16", act="swiglu",
               dropout=False, seq_parallel=False):
    """Saved activations of one rank: element counts by tensor and bytes by
    block.

    Readings of the pages' lists: GQA keeps K and V at n_kv heads; SwiGLU
    saves G and U where GeLU saves H; the flash form keeps the log-sum-exp
    (b, heads, s) in fp32 instead of S; a pre-norm layer adds each RMSNorm's
    input (T, h) and rstd (T, fp32) and a dropout mask (1 byte per element)
    after each block's reduction; under Megatron-SP the token-wise tensors
    (norm inputs, rstd, masks) hold ⌈s/n⌉ positions per sequence per rank
    while the blocks' inputs stay whole.
    """
    if n_q % n or n_kv % n or h_ffn % n:
        raise ValueError("n must divide n_q, n_kv and h_ffn")
    delta = DTYPE_BYTES[dtype]
    T = b * s
    tok = b * (-(-s // n)) if seq_parallel else T   # ceil(s / n) per sequence
    q, k = n_q // n, n_kv // n
    e = {
        "mlp_x": T * h,
        "mlp_hidden": (1 if act == "gelu" else 2) * T * (h_ffn // n),
        "mlp_act": T * (h_ffn // n),
        "mlp_mask": tok * h if dropout else 0,
        "attn_x": T * h,
        "attn_q": T * q * d,
        "attn_kv": 2 * T * k * d,
        "attn_scores": b * q * s * s,
        "attn_lse": b * q * s,
        "attn_o": T * q * d,
        "norm_x": tok * h,
        "norm_rstd": tok,
    }
    mask_bytes = tok * h if dropout else 0           # 1 byte per element
    e["mlp_bytes"] = (e["mlp_x"] + e["mlp_hidden"] + e["mlp_act"]) * delta \
        + e["mlp_mask"]
    common = (e["attn_x"] + e["attn_q"] + e["attn_kv"] + e["attn_o"]) * delta \
        + mask_bytes
    e["attn_bytes_pages"] = common + e["attn_scores"] * delta
    e["attn_bytes_flash"] = common + e["attn_lse"] * 4
    e["layer_bytes_flash"] = (2 * (e["norm_x"] * delta + e["norm_rstd"] * 4)
                              + e["attn_bytes_flash"] + e["mlp_bytes"])
    return e
