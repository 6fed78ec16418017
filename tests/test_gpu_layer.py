"""GPU parity of the full pre-norm layer, the TP-degree sweep, and rerun
determinism."""

import numpy as np
import pytest
import torch

import oracle
from megatron_tensor_transformer_gate_gb300 import binding as B
from megatron_tensor_transformer_gate_gb300 import inputs as I
from megatron_tensor_transformer_gate_gb300.blocks import TPLayer, TPMLP
from _parity import check, check_fro, f64

pytestmark = pytest.mark.gpu

GRADS = ("dX", "dWq", "dWk", "dWv", "dWo", "dW1", "dW2", "dg1", "dg2")


def run_layer(tp, cfg, seed, mode=B.FUSED):
    x = I.layer_inputs(cfg, seed, "cpu")
    P = {k: x[k].cuda() for k in ("g1", "Wq", "Wk", "Wv", "Wo", "g2", "W1",
                                  "W2")}
    X, dOut = x["X"].cuda(), x["dOut"].cuda()
    layer = TPLayer(cfg["b"], cfg["s"], cfg["h"], cfg["h_ffn"], cfg["n_q"],
                    cfg["n_kv"], cfg["d"], cfg["n"], eps=cfg["eps"], mode=mode)
    out = layer.forward(X, P)
    g = layer.backward(dOut, X, P)
    tp.device_status()
    return x, out, g, layer


def test_layer_workload_widths_reduced_sequence(tp):
    # the layer workload's widths (h 8192, 64 q / 8 kv heads, h_ffn 28672,
    # n 8) at s = 512 tokens, fully checked against the fp64 oracle
    cfg = I.workload("layer_bf16", s=512)
    x, out, g, layer = run_layer(tp, cfg, 20260005)
    Pf = {k: I.to_f64(v) for k, v in x.items()}
    shp = dict(b=1, s=512, n_q=64, n_kv=8, d=128, eps=cfg["eps"])
    fo = oracle.layer_forward(Pf["X"], Pf, **shp)
    go = oracle.layer_backward(Pf["dOut"], Pf["X"], Pf, fo, **shp)
    failures = []

    def expect(fn, *args):
        try:
            fn(*args)
        except AssertionError as e:
            failures.append(str(e))

    # end to end: every output and gradient within the Frobenius bound
    expect(check_fro, out, fo["Out"], "Out")
    for k in GRADS:
        expect(check_fro, g[k], go[k], k)
    # block by block: each block's oracle fed the bf16 tensors that block
    # consumed (its input activation; for backward, also what its forward
    # saved), with both bounds
    kw = dict(b=1, s=512, n_q=64, n_kv=8, d=128)
    xn1, x1, xn2 = f64(layer.xn1), f64(layer.x1), f64(layer.xn2)
    at = oracle.attention_forward(xn1, Pf["Wq"], Pf["Wk"], Pf["Wv"], Pf["Wo"],
                                  R=Pf["X"], **kw)
    expect(check, layer.x1, at["Out"], "attention block output")
    ml = oracle.mlp_forward(xn2, Pf["W1"], Pf["W2"], act="swiglu", R=x1)
    expect(check, out, ml["Out"], "MLP block output")
    ms = {k: f64(v) for k, v in layer.mlp.saved().items()}
    mb = oracle.mlp_backward(Pf["dOut"], xn2, Pf["W1"], Pf["W2"], ms,
                             act="swiglu")
    expect(check, g["dW1"], mb["dW1"], "MLP block dW1")
    expect(check, g["dW2"], mb["dW2"], "MLP block dW2")
    asv = {k: f64(v) for k, v in layer.attn.saved().items()}
    ab = oracle.attention_backward(f64(layer.dx1), xn1, Pf["Wq"], Pf["Wk"],
                                   Pf["Wv"], Pf["Wo"], asv, **kw)
    for k in ("dWq", "dWk", "dWv", "dWo"):
        expect(check, g[k], ab[k], "attention block " + k)
    assert not failures, "; ".join(failures)


@pytest.mark.parametrize("mode", [B.FUSED, B.MATERIALISED])
def test_layer_ragged_small(tp, mode):
    cfg = I.workload("layer_bf16", b=2, s=150, h=512, h_ffn=1408, n_q=8,
                     n_kv=4, n=4)
    x, out, g, layer = run_layer(tp, cfg, 7, mode)
    Pf = {k: I.to_f64(v) for k, v in x.items()}
    shp = dict(b=2, s=150, n_q=8, n_kv=4, d=128, eps=cfg["eps"])
    fo = oracle.layer_forward(Pf["X"], Pf, **shp)
    go = oracle.layer_backward(Pf["dOut"], Pf["X"], Pf, fo, **shp)
    check(out, fo["Out"], "Out")
    for k in GRADS:
        check(g[k], go[k], k)


@pytest.mark.parametrize("act", [B.GELU, B.SWIGLU])
def test_tp_degree_sweep_same_result(tp, act):
    # the shards change only how the reduction is cut: every n gives the
    # oracle's (n-independent) result, and materialised sums in shard order
    cfg = I.workload("mlp_swiglu_bf16", b=1, s=256, h=512, h_ffn=2048,
                     act="swiglu" if act == B.SWIGLU else "gelu")
    x = I.mlp_inputs(cfg, 11, "cuda")
    X, W1, W2, dOut = x["X"], x["W1"], x["W2"], x["dOut"]
    xf = {k: I.to_f64(v) for k, v in x.items() if v is not None}
    fo = oracle.mlp_forward(xf["X"], xf["W1"], xf["W2"], act=cfg["act"])
    go = oracle.mlp_backward(xf["dOut"], xf["X"], xf["W1"], xf["W2"], fo,
                             act=cfg["act"])
    outs = []
    for n in (1, 2, 4, 8):
        for mode in (B.FUSED, B.MATERIALISED):
            m = TPMLP(256, 512, 2048, n, act=act, mode=mode)
            out = m.forward(X, W1, W2)
            g = m.backward(dOut, X, W1, W2)
            tp.device_status()
            check(out, fo["Out"], f"Out n={n} mode={mode}")
            check(g["dX"], go["dX"], f"dX n={n} mode={mode}")
            outs.append(out.clone())
    # fused mode does not depend on n at all (one accumulation over K)
    assert torch.equal(outs[0], outs[2]) and torch.equal(outs[0], outs[6])


def test_reruns_are_bit_identical(tp):
    cfg = I.workload("layer_bf16", b=1, s=256, h=1024, h_ffn=2816, n_q=8,
                     n_kv=2, n=2)
    _, out1, g1, _ = run_layer(tp, cfg, 3)
    _, out2, g2, _ = run_layer(tp, cfg, 3)
    assert torch.equal(out1, out2)
    for k in GRADS:
        assert torch.equal(g1[k], g2[k]), k
