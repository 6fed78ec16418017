"""GPU parity of the FP8 path: E4M3 codes and scales bit-exact against the
oracle's quantization of the same bf16 values, the E4M3 GEMM and the MLP
forward in FP8 mode against the oracle, and the bf16 backward that follows
it."""

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8
from megatron_tensor_transformer_gate_gb300 import inputs as I
from megatron_tensor_transformer_gate_gb300.blocks import TPMLP
from _parity import check

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
