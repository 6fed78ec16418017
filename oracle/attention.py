"""Oracle for the head-sharded causal GQA attention block, forward and backward.

Test infrastructure: see the package docstring.

What is computed (unsharded; [Grasp-TP] §4, [hjcheng-TP] Attention
单卡forward / 单卡backward, [Troverld] §I.III attention TP graph):

    Q = X·Wqᵀ  [T, n_q·d],  K = X·Wkᵀ, V = X·Wvᵀ  [T, n_kv·d]
    per batch element, query head j (kv head ⌊j·n_kv/n_q⌋):
        S = Q_j·K_kvᵀ / √d, masked so that key position ≤ query position,
        P = softmax over keys (max subtracted first), O_j = P·V_kv
    Z = O·Woᵀ (+ bo once after the head reduction);  Out = R + Z

Token t = batch·s + position.  Heads are contiguous d-wide column groups of Q,
K, V, O.  GQA: the q heads of one kv head are a contiguous group, so an
even split of both head counts keeps each group on one rank ([Grasp-TP] §4
GQA note, [Troverld] §I.III).

Backward is the textbook softmax backward on the full s×s matrix (no flash
tiling): dP = dO·Vᵀ, dS = P ⊙ (dP − rowsum(dP ⊙ P)), dQ = dS·K/√d,
dK = dSᵀ·Q/√d, dV = Pᵀ·dO, with dK and dV summed over each kv head's group;
then dWq = dQᵀ·X etc. and dX = dQ·Wq + dK·Wk + dV·Wv (+ dres).

Pins (tests/test_oracle_attention.py): s = 1 reduces to the V projection then
Wo; Q = 0 gives the causal prefix mean of V; position 0 sees only itself;
softmax rows sum to 1; future keys never change past outputs; the head-sharded
sum equals the unsharded result; n_kv = n_q is plain multi-head attention;
central finite differences of every gradient.
"""

import math

import numpy as np


def _heads(M, b, s, nh, d):
    return M.reshape(b, s, nh, d)


def _probs(Qh, Kh, scale, causal):
    """P = softmax(mask(Qh·Khᵀ·scale)) for one (batch, head); also returns LSE."""
    S = (Qh @ Kh.T) * scale
    if causal:
        S = np.where(np.tril(np.ones(S.shape, dtype=bool)), S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    l = E.sum(axis=1, keepdims=True)
    return E / l, (m + np.log(l))[:, 0]


def _check_heads(n_q, n_kv):
    if n_q % n_kv:
        raise ValueError("n_kv must divide n_q")


def attention_core(Q, K, V, *, b, s, n_q, n_kv, d, causal=True):
    """softmax(mask(Q·Kᵀ/√d))·V per (batch, q head) with kv head
    ⌊j·n_kv/n_q⌋; Q [T, n_q·d], K, V [T, n_kv·d].  Returns O [T, n_q·d] and
    LSE [b, n_q, s]."""
    _check_heads(n_q, n_kv)
    Qh, Kh, Vh = (_heads(Q, b, s, n_q, d), _heads(K, b, s, n_kv, d),
                  _heads(V, b, s, n_kv, d))
    group = n_q // n_kv
    scale = 1.0 / math.sqrt(d)
    O = np.zeros((b, s, n_q, d))
    LSE = np.zeros((b, n_q, s))
    for bi in range(b):
        for j in range(n_q):
            kv = j // group
            P, lse = _probs(Qh[bi, :, j], Kh[bi, :, kv], scale, causal)
            O[bi, :, j] = P @ Vh[bi, :, kv]
            LSE[bi, j] = lse
    return O.reshape(b * s, n_q * d), LSE


def attention_forward(X, Wq, Wk, Wv, Wo, *, b, s, n_q, n_kv, d, causal=True,
                      bo=None, R=None):
    """Unsharded attention forward.  Returns Out, Q, K, V, O, LSE."""
    _check_heads(n_q, n_kv)
    X = np.asarray(X, np.float64)
    Q = X @ np.asarray(Wq, np.float64).T
    K = X @ np.asarray(Wk, np.float64).T
    V = X @ np.asarray(Wv, np.float64).T
    Of, LSE = attention_core(Q, K, V, b=b, s=s, n_q=n_q, n_kv=n_kv, d=d,
                             causal=causal)
    Z = Of @ np.asarray(Wo, np.float64).T
    Out = Z if bo is None else Z + bo
    if R is not None:
        Out = Out + R
    return {"Out": Out, "Q": Q, "K": K, "V": V, "O": Of, "LSE": LSE, "Z": Z}


def attention_backward(dOut, X, Wq, Wk, Wv, Wo, saved, *, b, s, n_q, n_kv, d,
                       causal=True, dres=None):
    """Unsharded attention backward.  ``saved`` is ``attention_forward``'s dict.

    Returns dX, dWq, dWk, dWv, dWo, dbo and the intermediates dO, dQ, dK, dV.
    """
    dOut = np.asarray(dOut, np.float64)
    X = np.asarray(X, np.float64)
    Wq, Wk, Wv, Wo = (np.asarray(W, np.float64) for W in (Wq, Wk, Wv, Wo))
    dZ = dOut
    dbo = dZ.sum(axis=0)
    dWo = dZ.T @ saved["O"]
    dO = dZ @ Wo
    Qh = _heads(saved["Q"], b, s, n_q, d)
    Kh = _heads(saved["K"], b, s, n_kv, d)
    Vh = _heads(saved["V"], b, s, n_kv, d)
    dOh = _heads(dO, b, s, n_q, d)
    dQ = np.zeros_like(Qh)
    dK = np.zeros_like(Kh)
    dV = np.zeros_like(Vh)
    group = n_q // n_kv
    scale = 1.0 / math.sqrt(d)
    for bi in range(b):
        for j in range(n_q):
            kv = j // group
            P, _ = _probs(Qh[bi, :, j], Kh[bi, :, kv], scale, causal)
            g = dOh[bi, :, j]
            dV[bi, :, kv] += P.T @ g
            dP = g @ Vh[bi, :, kv].T
            dS = P * (dP - (dP * P).sum(axis=1, keepdims=True))
            dQ[bi, :, j] = (dS @ Kh[bi, :, kv]) * scale
            dK[bi, :, kv] += (dS.T @ Qh[bi, :, j]) * scale
    dQf = dQ.reshape(b * s, n_q * d)
    dKf = dK.reshape(b * s, n_kv * d)
    dVf = dV.reshape(b * s, n_kv * d)
    dX = dQf @ Wq + dKf @ Wk + dVf @ Wv
    if dres is not None:
        dX = dX + dres
    return {"dX": dX, "dWq": dQf.T @ X, "dWk": dKf.T @ X, "dWv": dVf.T @ X,
            "dWo": dWo, "dbo": dbo, "dO": dO, "dQ": dQf, "dK": dKf, "dV": dVf}


def _shard_heads(n_q, n_kv, n, i, d):
    if n_q % n or n_kv % n:
        raise ValueError("n must divide n_q and n_kv")
    qw, kw = (n_q // n) * d, (n_kv // n) * d
    return slice(i * qw, (i + 1) * qw), slice(i * kw, (i + 1) * kw)


def attention_forward_sharded(X, Wq, Wk, Wv, Wo, n, *, b, s, n_q, n_kv, d,
                              causal=True, bo=None, R=None):
    """The block as n ranks compute it ([Grasp-TP] §4, [Troverld] §I.III).

    Rank i owns q heads [i·n_q/n, (i+1)·n_q/n) and kv heads
    [i·n_kv/n, (i+1)·n_kv/n) (rows of Wq/Wk/Wv), runs attention on its local
    heads only (every reshape uses the local head count, [Grasp-TP] §3 reading
    note), and multiplies by its columns of Wo to get a full-shape partial.
    The g reduction sums the partials; bo is added once after it.
    """
    X = np.asarray(X, np.float64)
    partials = []
    for i in range(n):
        qs, ks = _shard_heads(n_q, n_kv, n, i, d)
        r = attention_forward(X, Wq[qs], Wk[ks], Wv[ks], Wo[:, qs], b=b, s=s,
                              n_q=n_q // n, n_kv=n_kv // n, d=d,
                              causal=causal)
        partials.append(r["Z"])
    Z = partials[0].copy()
    for P in partials[1:]:
        Z += P
    Out = Z if bo is None else Z + bo
    if R is not None:
        Out = Out + R
    return {"Out": Out, "Z": Z, "partials": partials}


def attention_backward_sharded(dOut, X, Wq, Wk, Wv, Wo, n, *, b, s, n_q, n_kv,
                               d, causal=True, dres=None):
    """Backward per rank; the f reduction sums the partial input gradients."""
    X = np.asarray(X, np.float64)
    partials = []
    grads = {"dWq": np.zeros_like(np.asarray(Wq, np.float64)),
             "dWk": np.zeros_like(np.asarray(Wk, np.float64)),
             "dWv": np.zeros_like(np.asarray(Wv, np.float64)),
             "dWo": np.zeros_like(np.asarray(Wo, np.float64))}
    for i in range(n):
        qs, ks = _shard_heads(n_q, n_kv, n, i, d)
        kw = dict(b=b, s=s, n_q=n_q // n, n_kv=n_kv // n, d=d, causal=causal)
        f = attention_forward(X, Wq[qs], Wk[ks], Wv[ks], Wo[:, qs], **kw)
        g = attention_backward(dOut, X, Wq[qs], Wk[ks], Wv[ks], Wo[:, qs], f,
                               **kw)
        partials.append(g["dX"])
        grads["dWq"][qs] = g["dWq"]
        grads["dWk"][ks] = g["dWk"]
        grads["dWv"][ks] = g["dWv"]
        grads["dWo"][:, qs] = g["dWo"]
    dX = partials[0].copy()
    for P in partials[1:]:
        dX += P
    if dres is not None:
        dX = dX + dres
    grads.update({"dX": dX, "partials": partials})
    return grads
