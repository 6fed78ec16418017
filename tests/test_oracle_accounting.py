"""Pins of the accounting oracle: the pages' closed forms and loop counts."""

from fractions import Fraction

import pytest

import oracle


@pytest.mark.parametrize("T,h", [(64, 128), (4096, 1024), (8192, 4096),
                                 (1, 8), (3 * 7, 40)])
def test_mlp_flops_page_closed_forms(T, h):
    # hjcheng "TP" 单卡forward: 16·BS·d², 单卡backward: 32·BS·d² (d_ff = 4d)
    fwd, bwd = oracle.mlp_flops(T, h, 4 * h, "gelu")
    assert fwd == 16 * T * h * h
    assert bwd == 32 * T * h * h
    # TP forward: each rank does 1/n of it
    for n in (2, 4, 8):
        assert fwd % n == 0 and fwd // n == 16 * T * h * h // n


@pytest.mark.parametrize("b,s,h,nh", [(2, 2048, 4096, 32), (1, 64, 128, 2),
                                      (3, 5, 24, 3)])
def test_attn_flops_page_closed_forms(b, s, h, nh):
    # hjcheng "TP" Attention table: 8·BS·d² + 4·B·S²·d forward (MHA, full
    # mask), backward twice that
    fwd, bwd = oracle.attn_flops(b, s, h, nh, nh, h // nh, causal=False)
    assert fwd == 8 * b * s * h * h + 4 * b * s * s * h
    assert bwd == 2 * fwd


def test_flops_equal_loop_counts():
    # count the multiply-adds of the definitions with explicit loops
    T, h, f = 3, 5, 7
    macs = sum(1 for _t in range(T) for _j in range(f) for _k in range(h))
    macs += sum(1 for _t in range(T) for _i in range(h) for _j in range(f))
    assert oracle.mlp_flops(T, h, f, "gelu")[0] == 2 * macs
    b, s, nq, nkv, d, hh = 2, 6, 4, 2, 3, 10
    proj = b * s * hh * (nq + 2 * nkv) * d + b * s * nq * d * hh
    core = 0
    for _bi in range(b):
        for _j in range(nq):
            for q in range(s):
                for k in range(s):
                    if k <= q:
                        core += 2 * d          # one q·k dot and one p·v axpy
    fwd, bwd = oracle.attn_flops(b, s, hh, nq, nkv, d, causal=True)
    assert fwd == 2 * (proj + core) and bwd == 2 * fwd


@pytest.mark.parametrize("dtype,delta", [("f32", 4), ("bf16", 2)])
@pytest.mark.parametrize("n", [1, 2, 4, 8])
def test_comm_closed_forms(dtype, delta, n):
    b, s, h = 2, 4096, 4096
    T = b * s
    for scope, count in (("mlp", 2), ("attn", 2), ("layer", 4)):
        r = oracle.comm_report(scope, T, h, n, dtype)
        assert r["reductions_fwd"] + r["reductions_bwd"] == count
        # Grasp-TP §5: payload T·h·δ; ring 2(n−1)/n of it per rank
        assert r["payload_bytes"] == T * h * delta
        assert r["ring_bytes"] == Fraction(2 * (n - 1), n) * T * h * delta
        assert r["total_payload"] == count * T * h * delta
        # Troverld §II.II: 2δbSH per all-reduce, 4δbSH per block, 8δbSH/layer
        assert r["page2_bytes"] == 2 * delta * b * s * h
    assert oracle.comm_report("layer", T, h, n, dtype)["total_page2"] == \
        8 * delta * b * s * h
    assert oracle.comm_report("mlp", T, h, n, dtype)["total_page2"] == \
        4 * delta * b * s * h
    # Grasp-TP §5 per layer per rank: 8(n−1)/n·b·s·h·δ
    assert oracle.comm_report("layer", T, h, n, dtype)["total_ring"] == \
        Fraction(8 * (n - 1), n) * b * s * h * delta



# ---- saved activations: the pages' lists ([hjcheng-TP] MLP and Attention)
@pytest.mark.parametrize("b,s,dm,N", [(2, 16, 64, 1), (1, 128, 256, 4),
                                      (3, 40, 96, 8)])
def test_act_memory_page_lists(b, s, dm, N):
    BS = b * s
    # MLP, d_ff = 4 d_model, GeLU, with the dropout mask: single card
    # X + H + A + mask = BS·d + 2·BS·4d + BS·d; TP divides H and A by N
    r = oracle.act_memory(b, s, dm, 4 * dm, 8, 8, dm // 8, N, act="gelu",
                          dropout=True)
    mlp = r["mlp_x"] + r["mlp_hidden"] + r["mlp_act"] + r["mlp_mask"]
    assert mlp == 2 * BS * dm + 8 * BS * dm // N
    if N == 1:
        assert mlp == 10 * BS * dm
    # attention, MHA with h heads of d_model / h: single card
    # X + Q, K, V + S + AV = 5·BS·d + B·h·S²; TP divides all but X by N
    h_heads = 8
    r = oracle.act_memory(b, s, dm, 4 * dm, h_heads, h_heads, dm // h_heads,
                          N)
    attn = (r["attn_x"] + r["attn_q"] + r["attn_kv"] + r["attn_scores"]
            + r["attn_o"])
    assert attn == BS * dm + (4 * BS * dm + b * h_heads * s * s) // N
    with pytest.raises(ValueError):
        oracle.act_memory(b, s, dm, 4 * dm, 6, 6, 16, 4)   # n ∤ n_q


def test_act_memory_sequence_parallel():
    # SP with n = 1 is TP; otherwise the token-wise tensors shrink to ⌈s/n⌉
    # positions per sequence and nothing else changes
    base = dict(b=2, s=37, h=96, h_ffn=384, n_q=6, n_kv=3, d=16, dropout=True)
    assert oracle.act_memory(n=1, seq_parallel=True, **base) == \
        oracle.act_memory(n=1, **base)
    tp_ = oracle.act_memory(n=3, **base)
    sp = oracle.act_memory(n=3, seq_parallel=True, **base)
    for k in ("norm_x", "norm_rstd", "mlp_mask"):
        assert sp[k] * 37 == tp_[k] * 13          # ⌈37/3⌉ = 13 of 37
    for k in ("mlp_x", "mlp_hidden", "mlp_act", "attn_x", "attn_q",
              "attn_kv", "attn_scores", "attn_lse", "attn_o"):
        assert sp[k] == tp_[k]
    assert sp["layer_bytes_flash"] < tp_["layer_bytes_flash"]


@pytest.mark.parametrize("n", [1, 2, 3, 8])
def test_sp_split_moves_what_the_all_reduce_moved(n):
    # reduce-scatter + all-gather == one ring all-reduce, per position
    for scope in ("mlp", "attn", "layer"):
        r = oracle.comm_report(scope, 1000, 77, n, "bf16")
        assert r["sp_rs_bytes"] + r["sp_ag_bytes"] == r["ring_bytes"]
        assert r["sp_total"] == r["total_ring"]
        assert r["sp_reduce_scatters"] == r["reductions_fwd"] + \
            r["reductions_bwd"]
