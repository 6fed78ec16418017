"""GPU parity of the FP8 path: E4M3 codes and scales bit-exact against the
oracle's quantization of the same bf16 values, the E4M3 GEMM, the MLP, the
attention block and the whole layer with their forward projections in FP8
mode against the oracle, and the bf16 backward that follows them."""

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8
from megatron_tensor_transformer_gate_gb300 import inputs as I
from megatron_tensor_transformer_gate_gb300.blocks import (TPAttention,
                                                          TPLayer, TPMLP)
from _parity import FP8_LAYER_FRO, check, check_fro

pytestmark = pytest.mark.gpu


def gpu_quantize(tp, x):
    q = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    s = torch.empty(1, dtype=torch.float32, device="cuda")
    w = torch.empty(1, dtype=torch.int32, device="cuda")
    tp.quantize_fp8(x, q, s, w)
    return q, s


def seeded(shape, seed, scale=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(
        torch.bfloat16)


@pytest.mark.parametrize("shape,scale", [((1, 8), 1.0), ((37, 24), 3.0),
                                         ((1000, 1024), 0.02),
                                         ((4096, 4096), 1e-3)])
def test_quantize_codes_and_scale_bit_exact(tp, shape, scale):
    x = seeded(shape, 7, scale)
    q, s = gpu_quantize(tp, x)
    tp.device_status()
    xf = I.to_f64(x).astype(np.float32)
    qo, so, _ = ofp8.quantize(xf)
    assert s.item() == float(so)
    qg = q.cpu().numpy()
    bad = np.argwhere(qg != qo)
    assert len(bad) == 0, "codes differ at %d elements, e.g. %s" % (
        len(bad), [(hex(qg[tuple(i)]), hex(qo[tuple(i)]), float(xf[tuple(i)]))
                   for i in bad[:8]])


def test_quantize_all_zero_tensor(tp):
    x = torch.zeros((16, 32), dtype=torch.bfloat16, device="cuda")
    q, s = gpu_quantize(tp, x)
    assert s.item() == 1.0 and int(q.max()) == 0


@pytest.mark.parametrize("M,N,K", [(8, 16, 16), (256, 256, 128),
                                   (300, 520, 208), (1000, 1000, 1024),
                                   (513, 384, 4096), (2500, 2000, 256)])
def test_gemm_fp8_parity(tp, M, N, K):
    A, Bm = seeded((M, K), 11), seeded((N, K), 12, 0.05)
    qa, sa = gpu_quantize(tp, A)
    qb, sb = gpu_quantize(tp, Bm)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    tp.gemm_fp8(qa, sa, qb, sb, C)
    tp.device_status()
    qao, sao, _ = ofp8.quantize(I.to_f64(A).astype(np.float32))
    qbo, sbo, _ = ofp8.quantize(I.to_f64(Bm).astype(np.float32))
    check(C, ofp8.gemm(qao, sao, qbo, sbo), f"fp8 gemm {M}x{N}x{K}")


def run_mlp(tp, cfg, mode, seed):
    T = cfg["b"] * cfg["s"]
    x = I.mlp_inputs(cfg, seed, "cpu")
    act = tp.GELU if cfg["act"] == "gelu" else tp.SWIGLU
    p = cfg.get("p", 0.0)
    m = TPMLP(T, cfg["h"], cfg["h_ffn"], cfg["n"], dtype=tp.FP8, act=act,
              mode=mode, dropout_p=p, seed=seed)
    d = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    if cfg.get("residual") == "X":
        d["R"] = d["X"]
    out = m.forward(d["X"], d["W1"], d["W2"], b1=d["b1"], b2=d["b2"],
                    R=d["R"])
    dres = d["dOut"] if cfg.get("residual") == "X" else None
    g = m.backward(d["dOut"], d["X"], d["W1"], d["W2"], dres=dres,
                   want_db2=x["b2"] is not None)
    tp.device_status()
    f = {k: I.to_f64(v) for k, v in x.items()}
    if cfg.get("residual") == "X":
        f["R"] = f["X"]
    kw = dict(act=cfg["act"], p=p, seed=seed)
    fo = ofp8.mlp_forward(f["X"], f["W1"], f["W2"], b1=f["b1"], b2=f["b2"],
                          R=f["R"], **kw)
    go = oracle.mlp_backward(f["dOut"], f["X"], f["W1"], f["W2"], fo,
                             dres=f["dOut"] if dres is not None else None,
                             **kw)
    check(out, fo["Out"], "Out")
    for k in ("dX", "dW1", "dW2"):
        check(g[k], go[k], k)
    if "db2" in g:
        check(g["db2"], go["db2"], "db2")


@pytest.mark.parametrize("mode", [0, 1])
def test_fp8_swiglu_mlp_workload_widths(tp, mode):
    # the SwiGLU MLP workload's widths (h 4096, h_ffn 11008, n 8) at T = 512
    cfg = I.workload("mlp_swiglu_bf16", b=1, s=512)
    run_mlp(tp, cfg, mode, 20260003)


@pytest.mark.parametrize("mode", [0, 1])
def test_fp8_gelu_bias_dropout_residual_ragged(tp, mode):
    # GeLU with b2, dropout and R = X at ragged sizes (T 300, h 272, f 1088)
    cfg = I.workload("mlp_gelu_bf16", b=3, s=100, h=272, h_ffn=1088, n=4)
    run_mlp(tp, cfg, mode, 9)


def test_fp8_mode_rejects_unaligned_widths(tp):
    # E4M3 rows must be multiples of 16 bytes: h = 264 is not
    desc = tp.mlp_desc(64, 264, 1056, 4, tp.FP8, tp.GELU)
    assert tp.mlp_workspace_bytes(desc) == 0
    X = torch.zeros((64, 264), dtype=torch.bfloat16, device="cuda")
    W1 = torch.zeros((1056, 264), dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros((264, 1056), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.mlp_fwd(desc, X, W1, W2, torch.empty_like(X), ws)
    assert e.value.code == 2


def run_attn(tp, cfg, mode, seed):
    b, s, h = cfg["b"], cfg["s"], cfg["h"]
    nq, nkv, d, n = cfg["n_q"], cfg["n_kv"], cfg["d"], cfg["n"]
    causal = cfg.get("causal", True)
    x = I.attn_inputs(cfg, seed, "cpu")
    dv = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    a = TPAttention(b, s, h, nq, nkv, d, n, causal=causal, mode=mode,
                    dtype=tp.FP8)
    out = a.forward(dv["X"], dv["Wq"], dv["Wk"], dv["Wv"], dv["Wo"],
                    bo=dv["bo"], R=dv["R"])
    g = a.backward(dv["dOut"], dv["X"], dv["Wq"], dv["Wk"], dv["Wv"],
                   dv["Wo"], want_dbo=x["bo"] is not None)
    tp.device_status()
    f = {k: I.to_f64(v) for k, v in x.items()}
    kw = dict(b=b, s=s, n_q=nq, n_kv=nkv, d=d, causal=causal)
    fo = ofp8.attention_forward(f["X"], f["Wq"], f["Wk"], f["Wv"], f["Wo"],
                                bo=f["bo"], R=f["R"], **kw)
    go = oracle.attention_backward(f["dOut"], f["X"], f["Wq"], f["Wk"],
                                   f["Wv"], f["Wo"], fo, **kw)
    # Out comes from O re-quantized to E4M3: the GPU's O (fp16 probabilities,
    # flash accumulation) and the oracle's differ in the last bf16 bits, which
    # moves some O elements across an E4M3 rounding boundary (a 2^-4 step);
    # those flips stay inside the Frobenius bound but not the row-wise one
    check_fro(out, fo["Out"], "Out")
    for k in ("dX", "dWq", "dWk", "dWv", "dWo"):
        check(g[k], go[k], k)
    if "dbo" in g:
        check(g["dbo"], go["dbo"], "dbo")


@pytest.mark.parametrize("mode", [0, 1])
def test_fp8_attention_workload(tp, mode):
    # the attention workload (b 2, s 2048, h 4096, 32 q / 8 kv heads, n 4)
    run_attn(tp, I.workload("attn_gqa_bf16"), mode, 20260004)


@pytest.mark.parametrize("causal", [True, False])
def test_fp8_attention_ragged_bias_residual(tp, causal):
    cfg = I.workload("attn_gqa_bf16", b=2, s=200, h=512, n_q=8, n_kv=2, n=2,
                     causal=causal, bo=True, residual="random",
                     w_std="fan_in")
    run_attn(tp, cfg, 1, 35)


def test_fp8_layer(tp):
    # the pre-norm layer with both blocks' forward projections on E4M3
    cfg = I.workload("layer_fp8", b=2, s=256, h=1024, h_ffn=2048, n_q=8,
                     n_kv=2, d=128, n=2)
    x = I.layer_inputs(cfg, 36, "cpu")
    names = ("g1", "Wq", "Wk", "Wv", "Wo", "g2", "W1", "W2")
    P = {k: x[k].cuda() for k in names}
    L = TPLayer(cfg["b"], cfg["s"], cfg["h"], cfg["h_ffn"], cfg["n_q"],
                cfg["n_kv"], cfg["d"], cfg["n"], dtype=tp.FP8)
    X = x["X"].cuda()
    out = L.forward(X, P)
    g = L.backward(x["dOut"].cuda(), X, P)
    tp.device_status()
    f = {k: I.to_f64(v) for k, v in x.items()}
    shp = dict(b=cfg["b"], s=cfg["s"], n_q=cfg["n_q"], n_kv=cfg["n_kv"],
               d=cfg["d"], eps=cfg["eps"])
    fo = oracle.layer_forward(f["X"], f, fp8=True, **shp)
    go = oracle.layer_backward(f["dOut"], f["X"], f, fo, **shp)
    # two quantized blocks' E4M3 code flips carried through the layer: the
    # FP8 layer's Frobenius bound
    check_fro(out, fo["Out"], "Out", FP8_LAYER_FRO)
    for k in ("dX", "dWq", "dWk", "dWv", "dWo", "dW1", "dW2", "dg1", "dg2"):
        check_fro(g[k], go[k], k, FP8_LAYER_FRO)


def test_fp8_attention_rejects_unaligned_width(tp):
    # h = 264: E4M3 rows of X are not a multiple of 16 bytes
    desc = tp.attn_desc(1, 64, 264, 2, 1, 128, 1, tp.FP8)
    assert tp.attn_workspace_bytes(desc) == 0
