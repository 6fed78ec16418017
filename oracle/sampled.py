"""Row- and column-sampled oracle values for full-size checks (fp64).

Test infrastructure: see the package docstring.

At full size the unsharded oracle is affordable for the MLP but not cheap; a
token row of the MLP output depends only on that token's input row, and a
column of a weight gradient only on one column of the hidden activations, so
these helpers evaluate the same definitions as ``oracle.mlp`` on a subset:

* ``mlp_rows``: Out[t, :] and dX[t, :] for sampled tokens t;
* ``mlp_weight_cols``: dW1[j, :] for sampled hidden units j (and, for SwiGLU,
  both the gate row j and the up row f + j) and dW2[:, j];
* ``layer_sparse_upstream``: the whole pre-norm layer at full size for an
  upstream gradient that is zero outside a few token rows (forward rows
  sampled; every gradient, dense or as low-rank factors).

Each one restates the block's definition for its subset; pinned by agreeing
with the unsharded oracle on small shapes (tests/test_oracle_mlp.py).
"""

import numpy as np

from .primitives import gelu, gelu_grad, silu, silu_grad, dropout_keep


def _keep_rows(seed, rows, cols, p):
    return np.concatenate([dropout_keep(seed, 1, cols, p, row0=int(t))
                           for t in rows], axis=0)


def mlp_rows(rows, X, W1, W2, dOut, *, act="gelu", b1=None, b2=None, R=None,
             p=0.0, seed=0, dres=None):
    """Out and dX on the token rows ``rows`` (a 1-D integer array)."""
    rows = np.asarray(rows)
    W1 = np.asarray(W1, np.float64)
    W2 = np.asarray(W2, np.float64)
    x = np.asarray(X, np.float64)[rows]
    if act == "gelu":
        H = x @ W1.T
        if b1 is not None:
            H = H + b1
        A = gelu(H)
    else:
        f = W1.shape[0] // 2
        G = x @ W1[:f].T
        U = x @ W1[f:].T
        A = silu(G) * U
    Y = A @ W2.T
    if b2 is not None:
        Y = Y + b2
    scale = 1.0 / (1.0 - p)
    keep = _keep_rows(seed, rows, W2.shape[0], p) if p > 0 else None
    if keep is not None:
        Y = np.where(keep, Y * scale, 0.0)
    if R is not None:
        Y = Y + np.asarray(R, np.float64)[rows]
    dZ = np.asarray(dOut, np.float64)[rows]
    if keep is not None:
        dZ = np.where(keep, dZ * scale, 0.0)
    dA = dZ @ W2
    if act == "gelu":
        dH1 = dA * gelu_grad(H)
    else:
        dH1 = np.concatenate([dA * U * silu_grad(G), dA * silu(G)], axis=1)
    dX = dH1 @ W1
    if dres is not None:
        dX = dX + np.asarray(dres, np.float64)[rows]
    return {"Out": Y, "dX": dX}


def mlp_weight_cols(cols, X, W1, W2, dOut, *, act="gelu", b1=None, p=0.0,
                    seed=0):
    """dW1 rows and dW2 columns for the hidden units ``cols`` (1-D array).

    Returns dW1 [len(cols), h] (GeLU) or the gate and up rows
    ([len(cols), h] each, keys dW1_gate / dW1_up) for SwiGLU, and
    dW2 [h, len(cols)].
    """
    cols = np.asarray(cols)
    X = np.asarray(X, np.float64)
    W1 = np.asarray(W1, np.float64)
    W2 = np.asarray(W2, np.float64)
    dZ = np.asarray(dOut, np.float64)
    if p > 0:
        keep = dropout_keep(seed, dZ.shape[0], dZ.shape[1], p)
        dZ = np.where(keep, dZ / (1.0 - p), 0.0)
    dA = dZ @ W2[:, cols]
    if act == "gelu":
        H = X @ W1[cols].T
        if b1 is not None:
            H = H + b1[cols]
        dH = dA * gelu_grad(H)
        return {"dW1": dH.T @ X, "dW2": dZ.T @ gelu(H)}
    f = W1.shape[0] // 2
    G = X @ W1[cols].T
    U = X @ W1[f + cols].T
    dG = dA * U * silu_grad(G)
    dU = dA * silu(G)
    return {"dW1_gate": dG.T @ X, "dW1_up": dU.T @ X,
            "dW2": dZ.T @ (silu(G) * U)}


def layer_sparse_upstream(x, P, grad_rows, dOut_rows, out_rows, *, b, s, n_q,
                          n_kv, d, eps=1e-5):
    """The pre-norm SwiGLU layer at full size when the upstream gradient is
    zero except on a few token rows.

    Same definitions as ``oracle.layer`` (x1 = x + Attn(RMSNorm₁(x)),
    out = x1 + MLP(RMSNorm₂(x1)), causal GQA, reverse-mode chain), evaluated
    only where the values are needed:

    * forward: RMSNorm₁ and the K, V projections of every token (each query
      row attends to all earlier keys); queries, attention, out-projection,
      RMSNorm₂ and the MLP only for the rows in ``out_rows`` ∪ ``grad_rows``;
    * backward for dOut = 0 outside ``grad_rows`` (``dOut_rows`` holds those
      rows, in that order): the MLP, RMSNorm₂ and out-projection backward and
      dQ act on those rows only; dK, dV reach every earlier key; RMSNorm₁'s
      backward and dX cover every token.

    Returns Out on ``out_rows`` (dict row → vector), the full dX, dg1, dg2,
    dWk, dWv, and the rank-|grad_rows| weight gradients as factor pairs
    (dW = Lᵀ·R): ``dWq``, ``dWo``, ``dW1``, ``dW2``.

    Pinned by agreeing with ``oracle.layer_forward``/``layer_backward`` on
    small shapes with the same sparse upstream gradient
    (tests/test_oracle_norm_layer.py).
    """
    x = np.asarray(x, np.float64)
    g1, g2 = (np.asarray(P[k], np.float64) for k in ("g1", "g2"))
    Wq, Wk, Wv, Wo = (np.asarray(P[k], np.float64)
                      for k in ("Wq", "Wk", "Wv", "Wo"))
    W1, W2 = np.asarray(P["W1"], np.float64), np.asarray(P["W2"], np.float64)
    T, h = x.shape
    f = W1.shape[0] // 2
    group = n_q // n_kv
    scale = 1.0 / np.sqrt(d)
    grad_rows = [int(t) for t in grad_rows]
    rows = sorted(set(int(t) for t in out_rows) | set(grad_rows))

    # forward: RMSNorm₁, K, V of all tokens
    rstd1 = 1.0 / np.sqrt((x * x).mean(axis=1) + eps)
    y1 = x * rstd1[:, None] * g1
    K = y1 @ Wk.T
    V = y1 @ Wv.T
    fw = {}
    for t in rows:
        bi, pos = divmod(t, s)
        keys = slice(bi * s, bi * s + pos + 1)    # causal, same sequence
        q = y1[t] @ Wq.T
        O = np.zeros(n_q * d)
        probs = []
        for j in range(n_q):
            kv = j // group
            sc = (K[keys, kv * d:(kv + 1) * d] @ q[j * d:(j + 1) * d]) * scale
            e = np.exp(sc - sc.max())
            p = e / e.sum()
            probs.append(p)
            O[j * d:(j + 1) * d] = p @ V[keys, kv * d:(kv + 1) * d]
        x1 = x[t] + O @ Wo.T
        rstd2 = 1.0 / np.sqrt((x1 * x1).mean() + eps)
        y2 = x1 * rstd2 * g2
        G = y2 @ W1[:f].T
        U = y2 @ W1[f:].T
        A = silu(G) * U
        fw[t] = dict(q=q, O=O, probs=probs, keys=keys, x1=x1, rstd2=rstd2,
                     y2=y2, G=G, U=U, A=A, out=x1 + A @ W2.T)

    # backward
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    dx1_all = np.zeros_like(x)
    dy1 = np.zeros_like(x)
    dg2 = np.zeros(h)
    L1, R1, L2, R2, Lq, Rq, Lo, Ro = ([] for _ in range(8))
    for t, dout in zip(grad_rows, np.asarray(dOut_rows, np.float64)):
        c = fw[t]
        # MLP and RMSNorm₂ (row-local), residual
        dA = dout @ W2
        dG = dA * c["U"] * silu_grad(c["G"])
        dU = dA * silu(c["G"])
        dH = np.concatenate([dG, dU])
        dy2 = dH @ W1
        L1.append(dH); R1.append(c["y2"])
        L2.append(dout); R2.append(c["A"])
        gg = dy2 * g2
        dx1 = (c["rstd2"] * gg
               - c["x1"] * c["rstd2"] ** 3 * (gg @ c["x1"]) / h) + dout
        dg2 += dy2 * c["x1"] * c["rstd2"]
        dx1_all[t] = dx1
        # out-projection, then attention for this query row
        dO = dx1 @ Wo
        Lo.append(dx1); Ro.append(c["O"])
        dq = np.zeros(n_q * d)
        for j in range(n_q):
            kv = j // group
            ks = c["keys"]
            p = c["probs"][j]
            do = dO[j * d:(j + 1) * d]
            dp = V[ks, kv * d:(kv + 1) * d] @ do
            ds = p * (dp - do @ c["O"][j * d:(j + 1) * d])
            dq[j * d:(j + 1) * d] = (ds @ K[ks, kv * d:(kv + 1) * d]) * scale
            dK[ks, kv * d:(kv + 1) * d] += np.outer(ds, c["q"][j * d:(j + 1) * d]) * scale
            dV[ks, kv * d:(kv + 1) * d] += np.outer(p, do)
        Lq.append(dq); Rq.append(y1[t])
        dy1[t] += dq @ Wq
    dy1 += dK @ Wk + dV @ Wv
    # RMSNorm₁ backward over every token, plus the residual path
    gg = dy1 * g1
    dot = (gg * x).sum(axis=1)
    dX = rstd1[:, None] * gg - x * (rstd1 ** 3 * dot / h)[:, None] + dx1_all
    dg1 = (dy1 * x * rstd1[:, None]).sum(axis=0)
    pair = lambda L, R: (np.array(L), np.array(R))
    return {"Out": {t: fw[t]["out"] for t in out_rows}, "dX": dX,
            "dg1": dg1, "dg2": dg2, "dWk": dK.T @ y1, "dWv": dV.T @ y1,
            "dWq": pair(Lq, Rq), "dWo": pair(Lo, Ro), "dW1": pair(L1, R1),
            "dW2": pair(L2, R2)}
