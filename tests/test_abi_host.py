"""Host-side checks of the C ABI: it builds, loads, exports every declared
symbol, its accountant is bit-exact against the oracle, and invalid calls are
rejected before any launch (no GPU needed)."""

import ctypes
import os
import re
from fractions import Fraction

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tp.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tp_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(tp):
    names = declared_functions()
    assert len(names) >= 18
    L = tp.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(tp.SIGNATURES), "binding and header disagree"


WORKLOADS = [  # scope, T, h, n, dtype
    ("mlp", 64, 128, 2, "f32"), ("mlp", 4096, 1024, 4, "bf16"),
    ("mlp", 8192, 4096, 8, "bf16"), ("attn", 4096, 4096, 4, "bf16"),
    ("layer", 8192, 8192, 8, "bf16"), ("layer", 3, 40, 5, "f32"),
    ("mlp", 1, 8, 1, "bf16"), ("layer", 8192, 8192, 8, "fp8"),
    ("attn", 7, 9, 2, "fp8"),
]


@pytest.mark.parametrize("scope,T,h,n,dt", WORKLOADS)
def test_comm_bytes_bit_exact(tp, scope, T, h, n, dt):
    r = tp.comm_bytes({"mlp": 0, "attn": 1, "layer": 2}[scope], T, h, n,
                      {"f32": tp.F32, "bf16": tp.BF16, "fp8": tp.FP8}[dt])
    o = oracle.comm_report(scope, T, h, n, dt)
    assert r["reductions_fwd"] == o["reductions_fwd"]
    assert r["reductions_bwd"] == o["reductions_bwd"]
    assert r["payload_bytes"] == o["payload_bytes"]
    assert Fraction(r["ring_bytes_num"], r["ring_bytes_den"]) == o["ring_bytes"]
    assert r["page2_bytes"] == o["page2_bytes"]
    assert r["total_payload"] == o["total_payload"]
    assert Fraction(r["total_ring_num"], r["ring_bytes_den"]) == o["total_ring"]
    assert r["total_page2"] == o["total_page2"]
    sp = Fraction(r["sp_rs_bytes_num"], r["sp_bytes_den"])
    assert sp == o["sp_rs_bytes"]
    assert Fraction(r["sp_ag_bytes_num"], r["sp_bytes_den"]) == o["sp_ag_bytes"]
    assert r["sp_reduce_scatters"] == o["sp_reduce_scatters"]
    assert r["sp_all_gathers"] == o["sp_all_gathers"]
    assert Fraction(r["sp_total_num"], r["sp_bytes_den"]) == o["sp_total"]


def test_comm_bytes_named_workloads(tp):
    # 2 reductions per MLP, 4 per layer, each T·h·δ
    r = tp.comm_bytes(tp.SCOPE_MLP, 8192, 4096, 8, tp.BF16)
    assert r["total_payload"] == 2 * 67_108_864
    r = tp.comm_bytes(tp.SCOPE_LAYER, 8192, 8192, 8, tp.BF16)
    assert r["total_payload"] == 4 * 134_217_728
    assert r["total_page2"] == 1_073_741_824
    assert r["total_ring_num"] // r["ring_bytes_den"] == 939_524_096


@pytest.mark.parametrize("T,h,f,act", [(64, 128, 512, "gelu"),
                                       (4096, 1024, 4096, "gelu"),
                                       (8192, 4096, 11008, "swiglu"),
                                       (8192, 8192, 28672, "swiglu"),
                                       (7, 24, 40, "gelu")])
def test_mlp_flops_bit_exact(tp, T, h, f, act):
    d = tp.mlp_desc(T, h, f, 1, act=tp.GELU if act == "gelu" else tp.SWIGLU)
    assert tp.mlp_flops(d) == oracle.mlp_flops(T, h, f, act)


@pytest.mark.parametrize("b,s,h,nq,nkv,d,causal", [
    (2, 2048, 4096, 32, 8, 128, True), (1, 8192, 8192, 64, 8, 128, True),
    (2, 2048, 4096, 32, 8, 128, False), (3, 5, 24, 3, 1, 8, True)])
def test_attn_flops_bit_exact(tp, b, s, h, nq, nkv, d, causal):
    desc = tp.attn_desc(b, s, h, nq, nkv, d, 1, causal=causal)
    assert tp.attn_flops(desc) == oracle.attn_flops(b, s, h, nq, nkv, d,
                                                    causal)


def test_named_flop_totals(tp):
    a = tp.attn_flops(tp.attn_desc(1, 8192, 8192, 64, 8, 128, 8))
    m = tp.mlp_flops(tp.mlp_desc(8192, 8192, 28672, 8, act=tp.SWIGLU))
    assert sum(a) + sum(m) == 45_355_257_298_944
    assert sum(tp.mlp_flops(tp.mlp_desc(8192, 4096, 11008, 8,
                                        act=tp.SWIGLU))) == 6_648_609_374_208


FAKE = ctypes.c_void_p(0x100000)   # an aligned address never dereferenced


def _fwd(tp, desc, ws_bytes=1 << 40):
    L = tp.lib()
    return L.tp_mlp_fwd(ctypes.byref(desc), FAKE, FAKE, None, FAKE, None, None,
                        FAKE, FAKE, ws_bytes, None)


def test_mlp_rejects_before_launch(tp):
    L = tp.lib()
    assert L.tp_mlp_fwd(None, FAKE, FAKE, None, FAKE, None, None, FAKE, FAKE,
                        1, None) == 1                       # NULL desc
    assert _fwd(tp, tp.mlp_desc(64, 128, 500, 4)) == 2      # n ∤ h_ffn
    assert _fwd(tp, tp.mlp_desc(64, 124, 512, 2)) == 2      # h % 8
    assert _fwd(tp, tp.mlp_desc(64, 128, 512, 2, dtype=7)) == 3
    assert _fwd(tp, tp.mlp_desc(64, 128, 512, 2, dropout_p=1.0)) == 8
    assert _fwd(tp, tp.mlp_desc(0, 128, 512, 2)) == 2       # no tokens
    d = tp.mlp_desc(64, 128, 512, 2)
    assert _fwd(tp, d, ws_bytes=16) == 4                    # ws too small
    assert tp.mlp_workspace_bytes(d) >= 2 * 64 * 512 * 2
    mis = ctypes.c_void_p(0x100004)
    assert L.tp_mlp_fwd(ctypes.byref(d), mis, FAKE, None, FAKE, None, None,
                        FAKE, FAKE, 1 << 40, None) == 8     # misaligned
    assert L.tp_mlp_fwd(ctypes.byref(d), None, FAKE, None, FAKE, None, None,
                        FAKE, FAKE, 1 << 40, None) == 1


def test_attn_rejects_before_launch(tp):
    L = tp.lib()

    def call(desc, ws_bytes=1 << 40):
        return L.tp_attn_fwd(ctypes.byref(desc), FAKE, FAKE, FAKE, FAKE, FAKE,
                             None, None, FAKE, FAKE, ws_bytes, None)

    assert call(tp.attn_desc(1, 64, 512, 6, 4, 128, 2)) == 2   # n_kv ∤ n_q
    assert call(tp.attn_desc(1, 64, 512, 8, 2, 128, 4)) == 2   # n ∤ n_kv
    assert call(tp.attn_desc(1, 64, 512, 8, 2, 64, 2)) == 5    # d != 128
    assert call(tp.attn_desc(1, 64, 512, 8, 2, 128, 2, dtype=tp.F32)) == 5
    assert call(tp.attn_desc(1, 64, 512, 8, 2, 128, 2), ws_bytes=1) == 4
    assert tp.attn_workspace_bytes(tp.attn_desc(1, 64, 512, 8, 2, 128, 2)) > 0
    assert call(tp.attn_desc(0, 64, 512, 8, 2, 128, 2)) == 2   # no batch
    assert call(tp.attn_desc(1, 0, 512, 8, 2, 128, 2)) == 2    # no tokens
    # FP8 mode: E4M3 rows of X need h % 16 == 0
    assert call(tp.attn_desc(1, 64, 264, 2, 1, 128, 1, dtype=tp.FP8)) == 2


def test_attn_fp8_workspace_adds_the_e4m3_copies(tp):
    # X, Wq, Wk, Wv, O, Wo in E4M3 (one byte each) plus 6 scales and 6 amax
    # words, each region on a 256-byte boundary
    b, s, h, nq, nkv, d, n = 2, 200, 512, 8, 2, 128, 2
    T, qd, kd = b * s, nq * d, nkv * d
    base = tp.attn_workspace_bytes(tp.attn_desc(b, s, h, nq, nkv, d, n))
    f8 = tp.attn_workspace_bytes(tp.attn_desc(b, s, h, nq, nkv, d, n,
                                              dtype=tp.FP8))
    up = lambda x: (x + 255) // 256 * 256
    extra = sum(up(x) for x in (T * h, qd * h, kd * h, kd * h, T * qd,
                                h * qd, 24))
    assert f8 - up(base) == extra + 24      # the amax words end it


def test_status_strings(tp):
    L = tp.lib()
    for code in range(10):
        assert L.tp_status_string(code) != b"unknown status"


ACT_CONFIGS = [  # b, s, h, h_ffn, n_q, n_kv, d, n, dtype, act
    (1, 64, 128, 512, 2, 2, 64, 2, "f32", "gelu"),
    (4, 1024, 1024, 4096, 8, 8, 128, 4, "bf16", "gelu"),
    (2, 4096, 4096, 11008, 32, 8, 128, 8, "bf16", "swiglu"),
    (2, 2048, 4096, 11008, 32, 8, 128, 4, "bf16", "swiglu"),
    (1, 8192, 8192, 28672, 64, 8, 128, 8, "bf16", "swiglu"),
    (3, 37, 96, 384, 6, 3, 16, 3, "f32", "swiglu"),   # s not a multiple of n
]


@pytest.mark.parametrize("cfg", ACT_CONFIGS)
@pytest.mark.parametrize("dropout", [False, True])
@pytest.mark.parametrize("sp", [False, True])
def test_act_memory_bit_exact(tp, cfg, dropout, sp):
    b, s, h, f, nq, nkv, d, n, dt, act = cfg
    r = tp.act_memory(b, s, h, f, nq, nkv, d, n,
                      dtype={"f32": tp.F32, "bf16": tp.BF16}[dt],
                      act={"gelu": tp.GELU, "swiglu": tp.SWIGLU}[act],
                      dropout=dropout, seq_parallel=sp)
    o = oracle.act_memory(b, s, h, f, nq, nkv, d, n, dtype=dt, act=act,
                          dropout=dropout, seq_parallel=sp)
    assert r == o


def test_act_memory_matches_this_librarys_workspaces(tp):
    # the flash attention and MLP figures (all n ranks, without the block
    # input x and the masks) are what the library's fused-mode workspaces
    # hold, up to the 256-byte alignment of each region
    b, s, h, f, nq, nkv, d, n = 1, 8192, 8192, 28672, 64, 8, 128, 8
    r = tp.act_memory(b, s, h, f, nq, nkv, d, n)
    attn = n * ((r["attn_q"] + r["attn_kv"] + r["attn_o"]) * 2
                + r["attn_lse"] * 4)
    ws = tp.attn_workspace_bytes(tp.attn_desc(b, s, h, nq, nkv, d, n))
    assert 0 <= ws - attn < 5 * 256
    mlp = n * (r["mlp_hidden"] + r["mlp_act"]) * 2
    ws = tp.mlp_workspace_bytes(tp.mlp_desc(b * s, h, f, n, act=tp.SWIGLU))
    assert 0 <= ws - mlp < 3 * 256


def test_act_memory_rejects(tp):
    with pytest.raises(tp.TPError) as e:
        tp.act_memory(1, 64, 128, 512, 3, 3, 64, 2)     # n ∤ n_q
    assert e.value.code == 2
    with pytest.raises(tp.TPError) as e:
        tp.act_memory(1, 64, 128, 512, 2, 2, 64, 2, dtype=7)
    assert e.value.code == 3


@pytest.mark.parametrize("causal,tiles", [(True, 3), (False, 4)])
def test_ds_budget_sets_the_tile_scratch(tp, causal, tiles):
    # b=2, n_kv=2: four (batch, kv head) pairs, each with its group of 4 q
    # heads × (causal 3 | full 4) tiles of 128×128 fp16 (s=200: 2 blocks)
    d = tp.attn_desc(2, 200, 512, 8, 2, 128, 2, causal=causal)
    pair = 4 * tiles * 128 * 128 * 2
    prev = tp.attn_set_ds_budget(0)
    try:
        whole = tp.attn_bwd_scratch_bytes(d)
        assert tp.attn_set_ds_budget(1) == 8 << 30
        one = tp.attn_bwd_scratch_bytes(d)
        tp.attn_set_ds_budget(2 * pair)
        two = tp.attn_bwd_scratch_bytes(d)
    finally:
        tp.attn_set_ds_budget(prev)
    assert whole - one == 3 * pair
    assert whole - two == 2 * pair


def test_layer_workspaces_are_the_blocks_plus_the_norm_buffers(tp):
    b, s, h, f, nq, nkv, d, n = 2, 96, 512, 1024, 4, 2, 128, 2
    T = b * s
    up = lambda x: (x + 255) // 256 * 256
    for dt in (tp.BF16, tp.FP8):
        ld = tp.layer_desc(b, s, h, f, nq, nkv, d, n, dt)
        aw = tp.attn_workspace_bytes(tp.attn_desc(b, s, h, nq, nkv, d, n, dt))
        mw = tp.mlp_workspace_bytes(tp.mlp_desc(T, h, f, n, dt, tp.SWIGLU))
        assert aw > 0 and mw > 0
        # xn1, x1, xn2 (bf16), rstd1, rstd2 (fp32), attention ws, MLP ws;
        # bf16 mode: then the fp16 copies of xn1 and of [Wq; Wk; Wv]
        base = 3 * up(T * h * 2) + 2 * up(T * 4) + up(aw)
        qd, kd = nq * d, nkv * d
        if dt == tp.BF16:
            assert tp.layer_workspace_bytes(ld) == (
                base + up(mw) + up(T * h * 2) + (qd + 2 * kd) * h * 2)
        else:
            assert tp.layer_workspace_bytes(ld) == base + mw
        ab = tp.attn_bwd_scratch_bytes(tp.attn_desc(b, s, h, nq, nkv, d, n, dt))
        mb = tp.mlp_bwd_scratch_bytes(tp.mlp_desc(T, h, f, n, dt, tp.SWIGLU))
        nb = tp.rmsnorm_bwd_scratch_bytes(T, h)
        assert tp.layer_bwd_scratch_bytes(ld) == (
            2 * up(T * h * 2) + up(nb) + max(ab, mb))


def test_layer_rejects_before_launch(tp):
    L = tp.lib()

    def call(desc, ws_bytes=1 << 40):
        return L.tp_layer_fwd(ctypes.byref(desc), FAKE, FAKE, FAKE, FAKE, FAKE,
                              FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws_bytes,
                              None)

    ok = tp.layer_desc(1, 64, 512, 1024, 4, 2, 128, 2)
    assert call(ok, ws_bytes=16) == 4                          # ws too small
    assert call(tp.layer_desc(1, 64, 512, 1024, 4, 2, 128, 2,
                              dtype=tp.F32)) == 5
    assert call(tp.layer_desc(1, 64, 512, 1024, 4, 2, 128, 2, eps=0.0)) == 8
    assert call(tp.layer_desc(1, 64, 512, 1024, 6, 4, 128, 2)) == 2  # GQA
    assert call(tp.layer_desc(1, 64, 512, 1000, 4, 2, 128, 16)) == 2
    assert call(tp.layer_desc(0, 64, 512, 1024, 4, 2, 128, 2)) == 2
    assert L.tp_layer_fwd(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                          FAKE, FAKE, FAKE, FAKE, 1, None) == 1
    assert tp.layer_workspace_bytes(tp.layer_desc(1, 64, 512, 1024, 6, 4, 128,
                                                  2)) == 0


def test_ds_budget_is_read_once_per_backward_call(tp):
    # the dS tile region and the backward's passes come from one read of the
    # budget inside the call: scratch sized under a small budget is rejected
    # (before any launch) once the budget has grown, instead of being
    # written past its dS region by passes sized for the larger budget
    L = tp.lib()
    d = tp.attn_desc(2, 200, 512, 8, 2, 128, 2)
    prev = tp.attn_set_ds_budget(1)            # one (batch, kv head) pair
    try:
        one = tp.attn_bwd_scratch_bytes(d)
        tp.attn_set_ds_budget(0)               # default: all four pairs
        assert tp.attn_bwd_scratch_bytes(d) > one
        n0 = tp.launch_count()
        rc = L.tp_attn_bwd(ctypes.byref(d), *([FAKE] * 7), None,
                           *([FAKE] * 5), None, FAKE, one, None)
        assert rc == 4                          # TP_ERR_WORKSPACE
        assert tp.launch_count() == n0
    finally:
        tp.attn_set_ds_budget(prev)
