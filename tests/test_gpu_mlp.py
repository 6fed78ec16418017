"""GPU parity of the TP MLP (forward + backward) against the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from megatron_tensor_transformer_gate_gb300 import inputs as I
from megatron_tensor_transformer_gate_gb300.blocks import TPMLP
from _parity import check, check_fro, f64

pytestmark = pytest.mark.gpu


def run_case(tp, cfg, mode, seed, check_full=True):
    T = cfg["b"] * cfg["s"]
    x = I.mlp_inputs(cfg, seed, "cpu")
    dt = tp.F32 if cfg["dtype"] == "f32" else tp.BF16
    act = tp.GELU if cfg["act"] == "gelu" else tp.SWIGLU
    p = cfg.get("p", 0.0)
    dseed = seed
    m = TPMLP(T, cfg["h"], cfg["h_ffn"], cfg["n"], dtype=dt, act=act,
              mode=mode, dropout_p=p, seed=dseed)
    d = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    if x["R"] is not None and cfg.get("residual") == "X":
        d["R"] = d["X"]
    out = m.forward(d["X"], d["W1"], d["W2"], b1=d["b1"], b2=d["b2"],
                    R=d["R"])
    dres = d["dOut"] if cfg.get("residual") == "X" else None
    g = m.backward(d["dOut"], d["X"], d["W1"], d["W2"], dres=dres,
                   want_db1=x["b1"] is not None, want_db2=x["b2"] is not None)
    tp.device_status()
    X = I.to_f64(x["X"])
    W1, W2 = I.to_f64(x["W1"]), I.to_f64(x["W2"])
    kw = dict(act=cfg["act"], p=p, seed=dseed)
    fo = oracle.mlp_forward(X, W1, W2, b1=I.to_f64(x["b1"]),
                            b2=I.to_f64(x["b2"]), R=I.to_f64(x["R"]), **kw)
    go = oracle.mlp_backward(I.to_f64(x["dOut"]), X, W1, W2, fo,
                             dres=I.to_f64(x["dOut"]) if dres is not None
                             else None, **kw)
    dts = cfg["dtype"]
    res = {"Out": check(out, fo["Out"], "Out", dts)}
    for k in ("dX", "dW1", "dW2"):
        res[k] = check(g[k], go[k], k, dts)
    if "db1" in g:
        res["db1"] = check(g["db1"], go["db1"], "db1", dts)
    if "db2" in g:
        res["db2"] = check(g["db2"], go["db2"], "db2", dts)
    return res, out, fo


@pytest.mark.parametrize("mode", [0, 1])
def test_fp32_gelu_workload(tp, mode):
    run_case(tp, I.workload("mlp_gelu_f32"), mode, 20260001)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_bf16_ragged(tp, mode, act):
    # T and the shard width are not tile multiples; several tiles each way
    cfg = I.workload("mlp_gelu_bf16", b=3, s=111, h=520, h_ffn=1056, n=4,
                     act=act, b1=(act == "gelu"), b2=True, residual="random",
                     p=0.1 if act == "gelu" else 0.0, w_std="fan_in")
    run_case(tp, cfg, mode, 7)


@pytest.mark.parametrize("mode", [0, 1])
def test_fp32_ragged_swiglu(tp, mode):
    cfg = I.workload("mlp_gelu_f32", b=1, s=77, h=72, h_ffn=96, n=3,
                     act="swiglu", b2=True, residual="random", p=0.2)
    run_case(tp, cfg, mode, 8)


@pytest.mark.parametrize("mode", [0, 1])
def test_bf16_gelu_bias_dropout_workload(tp, mode):
    run_case(tp, I.workload("mlp_gelu_bf16"), mode, 20260002)


def test_dropout_mask_bit_exact(tp):
    # no residual: a dropped element must be exactly 0.  A kept element is
    # (Z + b2)/(1 − p); it can only be 0 through an exact cancellation, which
    # the materialised mode's bf16 shard partials make possible for values
    # that are tiny anyway — so a kept zero must be tiny in the oracle too.
    cfg = I.workload("mlp_gelu_bf16", b=2, s=128, h=256, h_ffn=512, n=2,
                     residual=None, p=0.3)
    keep = oracle.dropout_keep(99, 256, 256, 0.3)
    for mode in (0, 1):
        res, out, fo = run_case(tp, cfg, mode, 99)
        zero = (out == 0).cpu().numpy()
        assert not (~zero & ~keep).any(), f"mode {mode}: dropped but nonzero"
        o = fo["Out"]
        rms = np.sqrt((o * o).mean(axis=1, keepdims=True))
        suspicious = zero & keep & (np.abs(o) > 1e-2 * rms)
        assert not suspicious.any(), \
            f"mode {mode}: {int(suspicious.sum())} kept elements zeroed"
        if mode == 0:
            assert not (zero & keep).any()


@pytest.mark.parametrize("mode", [0, 1])
def test_bf16_swiglu_reduced_T(tp, mode):
    # the SwiGLU workload's widths (h 4096, h_ffn 11008, n 8) at T = 512
    cfg = I.workload("mlp_swiglu_bf16", b=1, s=512)
    run_case(tp, cfg, mode, 20260003)


def test_bf16_swiglu_full_size_sampled(tp):
    # full SwiGLU workload in the fused launch configuration; sampled rows of
    # Out / dX and sampled hidden units of dW1 / dW2 against the oracle
    cfg = I.workload("mlp_swiglu_bf16")
    T, h, f, n = 8192, 4096, 11008, 8
    x = I.mlp_inputs(cfg, 20260003, "cuda")
    m = TPMLP(T, h, f, n, act=tp.SWIGLU)
    out = m.forward(x["X"], x["W1"], x["W2"])
    g = m.backward(x["dOut"], x["X"], x["W1"], x["W2"])
    tp.device_status()
    rows = np.array([0, 1, 127, 128, 4095, 5000, 8191])
    cols = np.array([0, 1375, 1376, 5000, 11007])
    X, W1, W2 = (I.to_f64(x[k]) for k in ("X", "W1", "W2"))
    dOut = I.to_f64(x["dOut"])
    s = oracle.sampled.mlp_rows(rows, X, W1, W2, dOut, act="swiglu")
    check(out[rows], s["Out"], "Out rows")
    check(g["dX"][rows], s["dX"], "dX rows")
    c = oracle.sampled.mlp_weight_cols(cols, X, W1, W2, dOut, act="swiglu")
    check(g["dW1"][cols], c["dW1_gate"], "dW1 gate rows")
    check(g["dW1"][f + cols], c["dW1_up"], "dW1 up rows")
    check(g["dW2"][:, cols], c["dW2"], "dW2 cols")


def test_fused_and_materialised_agree(tp):
    cfg = I.workload("mlp_gelu_bf16", b=1, s=256, h=512, h_ffn=1024, n=4,
                     residual="random", p=0.1)
    a, oa, _ = run_case(tp, cfg, 0, 5)
    b, ob, _ = run_case(tp, cfg, 1, 5)
    # same inputs: the two reduction modes differ only by rounding order
    assert np.abs(f64(oa) - f64(ob)).max() <= 0.05 * np.abs(f64(oa)).max()


def test_bf16_swiglu_layer_widths(tp):
    # the MLP block of the layer workload (h 8192, h_ffn 28672, n 8, weights
    # std 0.02, residual) at T = 512 on its own seeded inputs, both bounds
    cfg = I.workload("mlp_swiglu_bf16", b=1, s=512, h=8192, h_ffn=28672,
                     n=8, w_std=0.02, residual="X")
    run_case(tp, cfg, 0, 20260005)


def test_overlapped_reduction_equals_materialised(tp):
    # TP_REDUCE_OVERLAP sums the same partials band by band on a second
    # stream: bit-identical to the materialised mode, bias, dropout (the mask
    # draw index must follow the band's rows) and residual included
    cfg = I.workload("mlp_gelu_bf16")           # T 4096: four bands
    T = cfg["b"] * cfg["s"]
    x = I.mlp_inputs(cfg, 20260002, "cuda")
    res = {}
    for mode in (tp.MATERIALISED, tp.OVERLAP):
        m = TPMLP(T, cfg["h"], cfg["h_ffn"], cfg["n"], act=tp.GELU, mode=mode,
                  dropout_p=cfg["p"], seed=20260002)
        out = m.forward(x["X"], x["W1"], x["W2"], b2=x["b2"], R=x["X"])
        g = m.backward(x["dOut"], x["X"], x["W1"], x["W2"], dres=x["dOut"],
                       want_db2=True)
        tp.device_status()
        res[mode] = [out.clone()] + [g[k].clone() for k in ("dX", "dW1",
                                                             "dW2", "db2")]
    for a, b in zip(res[tp.MATERIALISED], res[tp.OVERLAP]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_partial_last_wave_in_the_mlp(tp, act):
    # T 2560 × h_ffn 2048: the first projection (GeLU: 80 pair tiles;
    # SwiGLU: 160) and the gradient GEMM with the activation backward in
    # its epilogue (80) end in a partly filled wave
    cfg = I.workload("mlp_gelu_bf16", b=1, s=2560, h=512, h_ffn=2048, n=2,
                     act=act, b1=(act == "gelu"), p=0.0, w_std="fan_in")
    run_case(tp, cfg, 0, 9)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_single_token(tp, act):
    # T = 1: one row through every GEMM (a 256-row pair tile with 255 rows
    # past the end), bias, dropout and residual.  Each weight gradient is
    # then one outer product, row j scaled by the hidden unit's dH[0, j],
    # which cancels to near 0 where the activation's derivative does; the
    # row-wise bound does not apply to such rows, so the weight gradients
    # are held to the Frobenius bound (Out, dX and the bias gradients to
    # both)
    cfg = I.workload("mlp_gelu_bf16", b=1, s=1, h=256, h_ffn=512, n=2,
                     act=act, b1=(act == "gelu"), b2=True, residual="X",
                     p=0.1 if act == "gelu" else 0.0, w_std="fan_in")
    T = 1
    x = I.mlp_inputs(cfg, 41, "cpu")
    a = tp.GELU if act == "gelu" else tp.SWIGLU
    m = TPMLP(T, cfg["h"], cfg["h_ffn"], cfg["n"], act=a, mode=1,
              dropout_p=cfg["p"], seed=41)
    d = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    out = m.forward(d["X"], d["W1"], d["W2"], b1=d["b1"], b2=d["b2"],
                    R=d["X"])
    g = m.backward(d["dOut"], d["X"], d["W1"], d["W2"], dres=d["dOut"],
                   want_db1=x["b1"] is not None, want_db2=True)
    tp.device_status()
    X, W1, W2 = I.to_f64(x["X"]), I.to_f64(x["W1"]), I.to_f64(x["W2"])
    kw = dict(act=act, p=cfg["p"], seed=41)
    fo = oracle.mlp_forward(X, W1, W2, b1=I.to_f64(x["b1"]),
                            b2=I.to_f64(x["b2"]), R=X, **kw)
    go = oracle.mlp_backward(I.to_f64(x["dOut"]), X, W1, W2, fo,
                             dres=I.to_f64(x["dOut"]), **kw)
    check(out, fo["Out"], "Out")
    check(g["dX"], go["dX"], "dX")
    for k in ("db1", "db2"):
        if k in g:
            check(g[k], go[k], k)
    for k in ("dW1", "dW2"):
        check_fro(g[k], go[k], k)
