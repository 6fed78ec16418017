"""The pre-norm layer of the oracle with the library's stored roundings put
back in, one switch per stored tensor (fp64 arithmetic otherwise).

Test infrastructure built on ``oracle/`` only: it attributes the composed
layer's error against the exact oracle to the 16-bit tensors the CUDA path
stores between its kernels.  Each name below is one stored tensor; its
format is "exact" (kept in fp64), "bf16", "fp16" or "f32":

  forward   xn1_qkv  the first RMSNorm output as the Q, K, V projections read it
            xn1_bwd  the first RMSNorm output as the weight gradients read it
            qkv      Q, K, V                     P  the probabilities in P·V
            O        the attention output        x1 the residual stream
            xn2      the second RMSNorm output   GU the SwiGLU gate and up
            A        the SwiGLU output           out the layer output
  backward  dH       [dG | dU]                   dxn2 the MLP input gradient
            dx1      the residual gradient       dO the attention-core dO
            dS       the score gradient          dQKV dQ, dK, dV
            dxn1     the attention input gradient
            dX       the layer input gradient    dW every weight gradient

``PLAN`` is what the library stores for the bf16 layer (the Q, K, V
projections read fp16 copies of the first norm's output); ``EXACT`` keeps
everything in fp64, so ``dict(EXACT, out="bf16", dX="bf16", dW="bf16")`` is
the rounding of the results alone.
"""

import math

import numpy as np
import torch

import oracle
from oracle.primitives import silu, silu_grad


def _through(v, dt):
    """v rounded to fp32 (as an fp32 accumulator holds it), then to dt
    (nearest even), returned as float64."""
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return t.to(dt).to(torch.float64).numpy()


def bf16(v):
    return _through(v, torch.bfloat16)


FORMATS = {"exact": lambda v: v, "bf16": bf16,
           "fp16": lambda v: _through(v, torch.float16),
           "f32": lambda v: _through(v, torch.float32)}

NAMES = ("xn1_qkv", "xn1_bwd", "qkv", "P", "O", "x1", "xn2", "GU", "A", "out",
         "dH", "dxn2", "dx1", "dO", "dS", "dQKV", "dxn1", "dX", "dW")
EXACT = {k: "exact" for k in NAMES}
PLAN = dict(EXACT, xn1_qkv="fp16", xn1_bwd="bf16", qkv="fp16", P="fp16",
            O="bf16", x1="bf16", xn2="bf16", GU="bf16", A="bf16", out="bf16",
            dH="bf16", dxn2="bf16", dx1="bf16", dO="fp16", dS="fp16",
            dQKV="bf16", dxn1="bf16", dX="bf16", dW="bf16")


def layer(x, P, dout, plan, *, b, s, n_q, n_kv, d, eps):
    """Out and every gradient of the causal pre-norm SwiGLU layer (the
    definitions of ``oracle.layer_forward`` / ``layer_backward``) with the
    tensors named in ``plan`` rounded where the library stores them; only
    Out, O and x1 when dout is None."""
    r = lambda k, v: FORMATS[plan[k]](v)
    T = b * s
    n1 = oracle.rmsnorm_forward(x, P["g1"], eps)
    xq = r("xn1_qkv", n1["y"])
    Q, K, V = (r("qkv", xq @ P[w].T) for w in ("Wq", "Wk", "Wv"))
    scale, group = 1.0 / math.sqrt(d), n_q // n_kv
    Qh, Kh, Vh = (M.reshape(b, s, -1, d) for M in (Q, K, V))
    O = np.zeros((b, s, n_q, d))
    probs = {}
    keep = np.tril(np.ones((s, s), dtype=bool))
    for bi in range(b):
        for j in range(n_q):
            S = np.where(keep, Qh[bi, :, j] @ Kh[bi, :, j // group].T * scale,
                         -np.inf)
            E = np.exp(S - S.max(axis=1, keepdims=True))
            probs[bi, j] = E / E.sum(axis=1, keepdims=True)
            O[bi, :, j] = r("P", probs[bi, j]) @ Vh[bi, :, j // group]
    O = r("O", O.reshape(T, n_q * d))
    x1 = r("x1", x + O @ P["Wo"].T)
    n2 = oracle.rmsnorm_forward(x1, P["g2"], eps)
    xn2 = r("xn2", n2["y"])
    f = P["W1"].shape[0] // 2
    G, U = xn2 @ P["W1"][:f].T, xn2 @ P["W1"][f:].T
    A = r("A", silu(G) * U)
    G, U = r("GU", G), r("GU", U)
    out = r("out", x1 + A @ P["W2"].T)
    if dout is None:
        return {"Out": out, "O": O, "x1": x1}
    # backward
    dA = dout @ P["W2"]
    dH = np.concatenate([r("dH", dA * U * silu_grad(G)),
                         r("dH", dA * silu(G))], axis=1)
    g = {"dW2": r("dW", dout.T @ A), "dW1": r("dW", dH.T @ xn2)}
    dxn2 = r("dxn2", dH @ P["W1"])
    nb2 = oracle.rmsnorm_backward(dxn2, x1, P["g2"], eps, dres=dout)
    dx1 = r("dx1", nb2["dx"])
    g["dg2"] = r("dW", nb2["dgamma"])
    g["dWo"] = r("dW", dx1.T @ O)
    dO = r("dO", dx1 @ P["Wo"])
    D = (dO * O).reshape(b, s, n_q, d).sum(axis=-1)   # from the stored O
    dOh = dO.reshape(b, s, n_q, d)
    dQ, dK, dV = np.zeros_like(Qh), np.zeros_like(Kh), np.zeros_like(Vh)
    for bi in range(b):
        for j in range(n_q):
            kv, Pm, go = j // group, probs[bi, j], dOh[bi, :, j]
            dV[bi, :, kv] += r("P", Pm).T @ go
            dS = r("dS", Pm * (go @ Vh[bi, :, kv].T - D[bi, :, j][:, None]))
            dQ[bi, :, j] = dS @ Kh[bi, :, kv] * scale
            dK[bi, :, kv] += dS.T @ Qh[bi, :, j] * scale
    dQ, dK, dV = (r("dQKV", M.reshape(T, -1)) for M in (dQ, dK, dV))
    xb = r("xn1_bwd", n1["y"])
    g.update(dWq=r("dW", dQ.T @ xb), dWk=r("dW", dK.T @ xb),
             dWv=r("dW", dV.T @ xb))
    dxn1 = r("dxn1", dQ @ P["Wq"] + dK @ P["Wk"] + dV @ P["Wv"])
    nb1 = oracle.rmsnorm_backward(dxn1, x, P["g1"], eps, dres=dx1)
    g["dX"] = r("dX", nb1["dx"])
    g["dg1"] = r("dW", nb1["dgamma"])
    g["Out"] = out
    g["O"] = O
    return g
