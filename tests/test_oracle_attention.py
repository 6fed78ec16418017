"""Pins of the attention oracle."""

import math

import numpy as np
import pytest

import oracle
from oracle.attention import _probs
from _fd import assert_grad
from _golden import load, matrix


def _rand_attn(b, s, h, nq, nkv, d, seed, wscale=0.5):
    r = np.random.default_rng(seed)
    return dict(X=r.standard_normal((b * s, h)),
                Wq=r.standard_normal((nq * d, h)) * wscale,
                Wk=r.standard_normal((nkv * d, h)) * wscale,
                Wv=r.standard_normal((nkv * d, h)) * wscale,
                Wo=r.standard_normal((h, nq * d)) * wscale,
                bo=r.standard_normal(h) * 0.1,
                dOut=r.standard_normal((b * s, h)))


def _fwd(m, **kw):
    return oracle.attention_forward(m["X"], m["Wq"], m["Wk"], m["Wv"],
                                    m["Wo"], **kw)


def test_hand_worked():
    g = load("attn_tiny.txt")
    m = {k: matrix(g[k]) for k in ("X", "Wq", "Wk", "Wv", "Wo")}
    for k in ("Wq", "Wk", "Wv"):
        m[k] = m[k].reshape(1, -1)
    m["Wo"] = m["Wo"].reshape(-1, 1)
    kw = dict(b=1, s=2, n_q=1, n_kv=1, d=1)
    c = _fwd(m, causal=True, **kw)
    np.testing.assert_allclose(c["Out"], matrix(g["Out_causal"]), atol=1e-14)
    np.testing.assert_allclose(c["LSE"][0, 0], matrix(g["LSE_causal"]),
                               atol=1e-14)
    f = _fwd(m, causal=False, **kw)
    np.testing.assert_allclose(f["Out"], matrix(g["Out_full"]), atol=1e-14)


def test_single_position_is_value_projection():
    # s = 1: softmax over one key is 1, so O_j = V_{kv(j)}
    b, h, nq, nkv, d = 3, 8, 4, 2, 2
    m = _rand_attn(b, 1, h, nq, nkv, d, 1)
    out = _fwd(m, b=b, s=1, n_q=nq, n_kv=nkv, d=d)
    V = (m["X"] @ m["Wv"].T).reshape(b, nkv, d)
    O = np.repeat(V, nq // nkv, axis=1).reshape(b, nq * d)
    np.testing.assert_allclose(out["Out"], O @ m["Wo"].T, atol=1e-13)


def test_zero_query_gives_causal_prefix_mean():
    b, s, h, nq, nkv, d = 2, 5, 8, 2, 1, 4
    m = _rand_attn(b, s, h, nq, nkv, d, 2)
    m["Wq"][:] = 0.0
    out = _fwd(m, b=b, s=s, n_q=nq, n_kv=nkv, d=d)
    V = (m["X"] @ m["Wv"].T).reshape(b, s, d)
    mean = np.cumsum(V, axis=1) / np.arange(1, s + 1)[None, :, None]
    O = out["O"].reshape(b, s, nq, d)
    for j in range(nq):
        np.testing.assert_allclose(O[:, :, j], mean, atol=1e-13)
    np.testing.assert_allclose(O[:, 0, 0], V[:, 0], atol=1e-14)


def test_softmax_rows_sum_to_one_and_mask():
    r = np.random.default_rng(3)
    Qh, Kh = r.standard_normal((6, 4)) * 3, r.standard_normal((6, 4)) * 3
    P, lse = _probs(Qh, Kh, 0.5, True)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-15)
    assert (np.triu(P, 1) == 0).all()
    S = Qh @ Kh.T * 0.5
    for q in range(6):
        assert abs(lse[q] - math.log(np.exp(S[q, :q + 1]).sum())) < 1e-12


def test_future_keys_do_not_change_past():
    b, s, h, nq, nkv, d = 1, 6, 8, 4, 2, 2
    m = _rand_attn(b, s, h, nq, nkv, d, 4)
    a = _fwd(m, b=b, s=s, n_q=nq, n_kv=nkv, d=d)
    m2 = dict(m)
    m2["X"] = m["X"].copy()
    m2["X"][4:] += 3.0
    c = _fwd(m2, b=b, s=s, n_q=nq, n_kv=nkv, d=d)
    np.testing.assert_allclose(c["Out"][:4], a["Out"][:4], rtol=0, atol=1e-14)
    assert np.abs(c["Out"][4:] - a["Out"][4:]).max() > 1e-3


def test_mqa_equals_mha_with_repeated_kv():
    b, s, h, nq, d = 2, 4, 8, 4, 2
    m = _rand_attn(b, s, h, nq, 1, d, 5)
    gqa = _fwd(m, b=b, s=s, n_q=nq, n_kv=1, d=d)
    mha = dict(m, Wk=np.tile(m["Wk"], (nq, 1)), Wv=np.tile(m["Wv"], (nq, 1)))
    ref = _fwd(mha, b=b, s=s, n_q=nq, n_kv=nq, d=d)
    np.testing.assert_allclose(gqa["Out"], ref["Out"], atol=1e-13)


@pytest.mark.parametrize("n", [1, 2, 4])
def test_head_sharded_sum_equals_unsharded(n):
    b, s, h, nq, nkv, d = 2, 5, 8, 8, 4, 2
    m = _rand_attn(b, s, h, nq, nkv, d, 6)
    kw = dict(b=b, s=s, n_q=nq, n_kv=nkv, d=d, bo=m["bo"], R=m["X"])
    full = _fwd(m, **kw)
    sh = oracle.attention_forward_sharded(m["X"], m["Wq"], m["Wk"], m["Wv"],
                                          m["Wo"], n, **kw)
    assert np.abs(sh["Out"] - full["Out"]).max() <= 1e-12 * np.abs(
        full["Out"]).max()
    kwb = dict(b=b, s=s, n_q=nq, n_kv=nkv, d=d)
    g = oracle.attention_backward(m["dOut"], m["X"], m["Wq"], m["Wk"],
                                  m["Wv"], m["Wo"], _fwd(m, **kwb), **kwb)
    gs = oracle.attention_backward_sharded(m["dOut"], m["X"], m["Wq"],
                                           m["Wk"], m["Wv"], m["Wo"], n,
                                           **kwb)
    for k in ("dX", "dWq", "dWk", "dWv", "dWo"):
        assert np.abs(gs[k] - g[k]).max() <= 1e-12 * np.abs(g[k]).max(), k


def test_shard_degree_must_divide_heads():
    m = _rand_attn(1, 2, 8, 4, 2, 2, 7)
    with pytest.raises(ValueError):
        oracle.attention_forward_sharded(m["X"], m["Wq"], m["Wk"], m["Wv"],
                                         m["Wo"], 4, b=1, s=2, n_q=4, n_kv=2,
                                         d=2)


@pytest.mark.parametrize("causal", [True, False])
def test_backward_finite_differences(causal):
    b, s, h, nq, nkv, d = 2, 3, 4, 4, 2, 2
    m = _rand_attn(b, s, h, nq, nkv, d, 8)
    kw = dict(b=b, s=s, n_q=nq, n_kv=nkv, d=d, causal=causal)
    dOut = m["dOut"]

    def loss():
        return float((_fwd(m, bo=m["bo"], **kw)["Out"] * dOut).sum())

    f = _fwd(m, bo=m["bo"], **kw)
    g = oracle.attention_backward(dOut, m["X"], m["Wq"], m["Wk"], m["Wv"],
                                  m["Wo"], f, **kw)
    for name, arr in (("dX", "X"), ("dWq", "Wq"), ("dWk", "Wk"),
                      ("dWv", "Wv"), ("dWo", "Wo"), ("dbo", "bo")):
        assert_grad(g[name], loss, m[arr])
