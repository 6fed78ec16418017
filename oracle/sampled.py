"""Row- and column-sampled oracle values for full-size checks (fp64).

Test infrastructure: see the package docstring.

At full size the unsharded oracle is affordable for the MLP but not cheap; a
token row of the MLP output depends only on that token's input row, and a
column of a weight gradient only on one column of the hidden activations, so
these helpers evaluate the same definitions as ``oracle.mlp`` on a subset:

* ``mlp_rows``: Out[t, :] and dX[t, :] for sampled tokens t;
* ``mlp_weight_cols``: dW1[j, :] for sampled hidden units j (and, for SwiGLU,
  both the gate row j and the up row f + j) and dW2[:, j].

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
