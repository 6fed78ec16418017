"""Oracle for one pre-norm Transformer layer: RMSNorm → attention → residual →
RMSNorm → MLP → residual, forward and backward (fp64).

Test infrastructure: see the package docstring.

    x1  = x  + Attn(RMSNorm₁(x))
    out = x1 + MLP(RMSNorm₂(x1))

The four tensor-parallel reductions of the layer ([Grasp-TP] §5, [adu-TP]
张量并行的通信开销) sit at the attention output (forward), the MLP output
(forward), the MLP input gradient (backward) and the attention input gradient
(backward); the residual gradients bypass them.

Pins: composition of pinned parts, and central finite differences on a tiny
layer (tests/test_oracle_layer.py).
"""

from .attention import attention_forward, attention_backward
from .mlp import mlp_forward, mlp_backward
from .norm import rmsnorm_forward, rmsnorm_backward


def layer_forward(x, P, *, b, s, n_q, n_kv, d, eps=1e-5, act="swiglu",
                  causal=True, fp8=False):
    """``P`` holds g1, Wq, Wk, Wv, Wo, g2, W1, W2 (unsharded, fp64-convertible).
    fp8=True: both blocks' forward projections on E4M3 operands
    (``oracle.fp8.attention_forward`` and ``oracle.fp8.mlp_forward``), each
    block quantizing its input as stored (the RMSNorm outputs rounded to
    bf16); the backward then follows the saved values of that forward."""
    attn_f, mlp_f = attention_forward, mlp_forward
    stored = lambda n: n
    if fp8:
        # a block quantizes its input as stored: the norm outputs in bf16
        from . import fp8 as f8
        attn_f, mlp_f = f8.attention_forward, f8.mlp_forward
        stored = lambda n: dict(n, y=f8.round_bf16(n["y"]))
    n1 = stored(rmsnorm_forward(x, P["g1"], eps))
    at = attn_f(n1["y"], P["Wq"], P["Wk"], P["Wv"], P["Wo"], b=b, s=s,
                n_q=n_q, n_kv=n_kv, d=d, causal=causal, R=x)
    x1 = at["Out"]
    n2 = stored(rmsnorm_forward(x1, P["g2"], eps))
    ml = mlp_f(n2["y"], P["W1"], P["W2"], act=act, R=x1)
    return {"Out": ml["Out"], "x1": x1, "n1": n1, "n2": n2, "attn": at,
            "mlp": ml}


def layer_backward(dout, x, P, saved, *, b, s, n_q, n_kv, d, eps=1e-5,
                   act="swiglu", causal=True):
    ml = mlp_backward(dout, saved["n2"]["y"], P["W1"], P["W2"], saved["mlp"],
                      act=act)
    nb2 = rmsnorm_backward(ml["dX"], saved["x1"], P["g2"], eps, dres=dout)
    dx1 = nb2["dx"]
    at = attention_backward(dx1, saved["n1"]["y"], P["Wq"], P["Wk"], P["Wv"],
                            P["Wo"], saved["attn"], b=b, s=s, n_q=n_q,
                            n_kv=n_kv, d=d, causal=causal)
    nb1 = rmsnorm_backward(at["dX"], x, P["g1"], eps, dres=dx1)
    return {"dX": nb1["dx"], "dg1": nb1["dgamma"], "dg2": nb2["dgamma"],
            "dWq": at["dWq"], "dWk": at["dWk"], "dWv": at["dWv"],
            "dWo": at["dWo"], "dW1": ml["dW1"], "dW2": ml["dW2"],
            "dx1": dx1}
