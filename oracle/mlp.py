"""Oracle for the Megatron MLP block (GeLU or SwiGLU), forward and backward.

Test infrastructure: see the package docstring.

Layout conventions (shared with the product only as a *convention*, not as
code): activations are [T, h] row-major with T = b·s tokens; weights are
stored [out_features, in_features] as ``Linear.weight`` is ([Grasp-TP] §1
notes this storage transposition), so the first projection is X·W1ᵀ.  For
SwiGLU, W1 is [2·f, h]: rows [0, f) are the gate projection, rows [f, 2f) the
up projection.

What is computed (unsharded, [hjcheng-TP] MLP 单卡forward / 单卡backward,
[Grasp-TP] §3):

    GeLU:    H = X·W1ᵀ (+ b1),  A = GeLU(H)
    SwiGLU:  G = X·Wgᵀ, U = X·Wuᵀ,  A = SiLU(G) ⊙ U       ([Grasp-TP] §3)
    Z = A·W2ᵀ;  Y = Z (+ b2, once, after the sum: [Grasp-TP] §3 bias note)
    Out = R + mask ⊙ Y / (1 − p)                           ([Troverld] §I.III)

Backward by the chain rule, with dZ = dOut ⊙ mask / (1 − p) as printed in
[hjcheng-TP] 单卡backward, dW2 = dZᵀ·A, dA = dZ·W2, then through the
activation to dH (or dG, dU), dW1 = dHᵀ·X, and dX = dH·W1 (+ dres, the
gradient of a residual that is the block's own input).

Pins (tests/test_oracle_mlp.py): the sharded sum equals the unsharded result
([hjcheng-TP] TP backward: Z = Σ_i Z^i; [adu-TP] Z = Y1B1 + Y2B2); GeLU of the
column shards equals the column shards of GeLU ([Grasp-TP] §2, [adu-TP] 列切分);
row-first sharding breaks under GeLU ([adu-TP] 行切分); a per-shard bias is off
by (n − 1)·b ([Grasp-TP] §3); hand-worked tiny cases; central finite
differences of every gradient.
"""

import numpy as np

from .primitives import gelu, gelu_grad, silu, silu_grad, dropout_keep


def _dropout_scale(p):
    return 1.0 / (1.0 - p)


def _activation(X, W1, b1, act):
    """First projection + activation on whatever rows of W1 are passed in."""
    if act == "gelu":
        H = X @ W1.T
        if b1 is not None:
            H = H + b1
        return {"H": H, "A": gelu(H)}
    if act == "swiglu":
        f = W1.shape[0] // 2
        G = X @ W1[:f].T
        U = X @ W1[f:].T
        if b1 is not None:
            G = G + b1[:f]
            U = U + b1[f:]
        return {"G": G, "U": U, "A": silu(G) * U}
    raise ValueError("act must be 'gelu' or 'swiglu'")


def _output(Z, b2, R, p, seed):
    """Bias once after the reduction, then dropout, then the residual."""
    Y = Z if b2 is None else Z + b2
    if p > 0.0:
        keep = dropout_keep(seed, Y.shape[0], Y.shape[1], p)
        Y = np.where(keep, Y * _dropout_scale(p), 0.0)
    if R is not None:
        Y = Y + R
    return Y


def mlp_forward(X, W1, W2, *, act="gelu", b1=None, b2=None, R=None, p=0.0,
                seed=0):
    """Unsharded MLP forward.  Returns a dict with Out, Z and the saved H/G/U/A."""
    X = np.asarray(X, dtype=np.float64)
    saved = _activation(X, np.asarray(W1, np.float64), b1, act)
    Z = saved["A"] @ np.asarray(W2, np.float64).T
    out = dict(saved)
    out["Z"] = Z
    out["Out"] = _output(Z, b2, R, p, seed)
    return out


def _shard_rows(f, n, i):
    if f % n:
        raise ValueError("n must divide h_ffn")
    w = f // n
    return slice(i * w, (i + 1) * w)


def _w1_shard(W1, act, n, i):
    """Rows of W1 held by rank i (column-parallel: split along the output dim)."""
    if act == "gelu":
        return W1[_shard_rows(W1.shape[0], n, i)]
    f = W1.shape[0] // 2
    r = _shard_rows(f, n, i)
    return np.concatenate([W1[:f][r], W1[f:][r]], axis=0)


def _b1_shard(b1, act, n, i):
    if b1 is None:
        return None
    if act == "gelu":
        return b1[_shard_rows(b1.shape[0], n, i)]
    f = b1.shape[0] // 2
    r = _shard_rows(f, n, i)
    return np.concatenate([b1[:f][r], b1[f:][r]])


def mlp_forward_sharded(X, W1, W2, n, *, act="gelu", b1=None, b2=None, R=None,
                        p=0.0, seed=0, bias_per_shard=False):
    """The same block computed as n ranks would ([hjcheng-TP] TP forward).

    Rank i holds rows i of W1 (column-parallel) and the matching columns of W2
    (row-parallel), computes A_i = act(X·W1_iᵀ) locally and the partial
    Z^i = A_i·W2_iᵀ, and the g all-reduce sums the partials: Z = Σ_i Z^i.
    ``bias_per_shard=True`` reproduces the mistake [Grasp-TP] §3 warns of (each
    rank adding the full b2 before the reduction) for the pin that shows it.
    Returns Out, the partials and the per-shard activations.
    """
    X = np.asarray(X, np.float64)
    W1 = np.asarray(W1, np.float64)
    W2 = np.asarray(W2, np.float64)
    f = W1.shape[0] if act == "gelu" else W1.shape[0] // 2
    partials, acts = [], []
    for i in range(n):
        cols = _shard_rows(f, n, i)
        a = _activation(X, _w1_shard(W1, act, n, i), _b1_shard(b1, act, n, i),
                        act)
        Zi = a["A"] @ W2[:, cols].T
        if bias_per_shard and b2 is not None:
            Zi = Zi + b2
        partials.append(Zi)
        acts.append(a)
    Z = partials[0].copy()
    for Zi in partials[1:]:
        Z += Zi
    out_bias = None if bias_per_shard else b2
    return {"Out": _output(Z, out_bias, R, p, seed), "Z": Z,
            "partials": partials, "acts": acts}


def _grad_through_output(dOut, p, seed):
    if p > 0.0:
        keep = dropout_keep(seed, dOut.shape[0], dOut.shape[1], p)
        return np.where(keep, dOut * _dropout_scale(p), 0.0)
    return dOut


def _grad_through_activation(dA, saved, act):
    """dA → gradient of the first projection's output (dH, or [dG | dU])."""
    if act == "gelu":
        return dA * gelu_grad(saved["H"])
    G, U = saved["G"], saved["U"]
    dG = dA * U * silu_grad(G)
    dU = dA * silu(G)
    return np.concatenate([dG, dU], axis=1)


def mlp_backward(dOut, X, W1, W2, saved, *, act="gelu", p=0.0, seed=0,
                 dres=None):
    """Unsharded MLP backward.

    ``saved`` is the dict returned by ``mlp_forward``.  Returns dX, dW1, db1
    (the column sum of the first projection's output gradient), dW2, db2, and
    the intermediate dZ, dA, dH1 (dH, or [dG | dU] for SwiGLU).
    """
    dOut = np.asarray(dOut, np.float64)
    X = np.asarray(X, np.float64)
    W1 = np.asarray(W1, np.float64)
    W2 = np.asarray(W2, np.float64)
    dZ = _grad_through_output(dOut, p, seed)
    db2 = dZ.sum(axis=0)
    dW2 = dZ.T @ saved["A"]
    dA = dZ @ W2
    dH1 = _grad_through_activation(dA, saved, act)
    db1 = dH1.sum(axis=0)
    dW1 = dH1.T @ X
    dX = dH1 @ W1
    if dres is not None:
        dX = dX + dres
    return {"dX": dX, "dW1": dW1, "db1": db1, "dW2": dW2, "db2": db2,
            "dZ": dZ, "dA": dA, "dH1": dH1}


def mlp_backward_sharded(dOut, X, W1, W2, n, *, act="gelu", b1=None, p=0.0,
                         seed=0, dres=None):
    """Backward as n ranks compute it ([hjcheng-TP] TP backward, [adu-TP] f).

    Every rank sees the same dZ (the g reduction made Z replicated), computes
    its local dW1_i, dW2_i and a partial input gradient dX_i = dH_i·W1_i; the
    f all-reduce sums the partials.  Returns dX, the partials and the
    per-rank weight gradients re-assembled into full tensors.
    """
    dOut = np.asarray(dOut, np.float64)
    X = np.asarray(X, np.float64)
    W1 = np.asarray(W1, np.float64)
    W2 = np.asarray(W2, np.float64)
    f = W1.shape[0] if act == "gelu" else W1.shape[0] // 2
    dZ = _grad_through_output(dOut, p, seed)
    dW1 = np.zeros_like(W1)
    dW2 = np.zeros_like(W2)
    partials = []
    for i in range(n):
        cols = _shard_rows(f, n, i)
        W1i = _w1_shard(W1, act, n, i)
        a = _activation(X, W1i, _b1_shard(b1, act, n, i), act)
        dW2[:, cols] = dZ.T @ a["A"]
        dAi = dZ @ W2[:, cols]
        dHi = _grad_through_activation(dAi, a, act)
        dW1i = dHi.T @ X
        if act == "gelu":
            dW1[cols] = dW1i
        else:
            w = f // n
            dW1[:f][cols] = dW1i[:w]
            dW1[f:][cols] = dW1i[w:]
        partials.append(dHi @ W1i)
    dX = partials[0].copy()
    for P in partials[1:]:
        dX += P
    if dres is not None:
        dX = dX + dres
    return {"dX": dX, "partials": partials, "dW1": dW1, "dW2": dW2,
            "db2": dZ.sum(axis=0)}
