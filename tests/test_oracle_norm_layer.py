"""Pins of the RMSNorm and layer oracles."""

import numpy as np

import oracle
from _fd import assert_grad


def test_rmsnorm_unit_rms_and_scale_invariance():
    r = np.random.default_rng(1)
    x = r.standard_normal((5, 16)) * 3
    y = oracle.rmsnorm_forward(x, np.ones(16), eps=0.0)["y"]
    np.testing.assert_allclose(np.sqrt((y * y).mean(axis=1)), 1.0, atol=1e-14)
    y2 = oracle.rmsnorm_forward(x * np.array([[0.5], [2], [7], [1e3], [1e-3]]),
                                np.ones(16), eps=0.0)["y"]
    np.testing.assert_allclose(y2, y, atol=1e-13)
    # a row of equal entries c maps to sign(c)·γ when ε = 0
    g = r.standard_normal(16)
    y3 = oracle.rmsnorm_forward(np.full((1, 16), -4.0), g, eps=0.0)["y"]
    np.testing.assert_allclose(y3[0], -g, atol=1e-14)


def test_rmsnorm_backward_finite_differences():
    r = np.random.default_rng(2)
    x = r.standard_normal((4, 8))
    g = 1 + 0.1 * r.standard_normal(8)
    dy = r.standard_normal((4, 8))
    dres = r.standard_normal((4, 8))

    def loss():
        return float((oracle.rmsnorm_forward(x, g, 1e-5)["y"] * dy).sum())

    b = oracle.rmsnorm_backward(dy, x, g, 1e-5)
    assert_grad(b["dx"], loss, x)
    assert_grad(b["dgamma"], loss, g)
    b2 = oracle.rmsnorm_backward(dy, x, g, 1e-5, dres=dres)
    np.testing.assert_allclose(b2["dx"] - b["dx"], dres, atol=1e-14)


def _tiny_layer(seed):
    r = np.random.default_rng(seed)
    h, nq, nkv, d, f = 8, 4, 2, 2, 12
    P = dict(g1=1 + 0.1 * r.standard_normal(h),
             Wq=r.standard_normal((nq * d, h)) * 0.4,
             Wk=r.standard_normal((nkv * d, h)) * 0.4,
             Wv=r.standard_normal((nkv * d, h)) * 0.4,
             Wo=r.standard_normal((h, nq * d)) * 0.4,
             g2=1 + 0.1 * r.standard_normal(h),
             W1=r.standard_normal((2 * f, h)) * 0.4,
             W2=r.standard_normal((h, f)) * 0.4)
    return P, dict(b=2, s=3, n_q=nq, n_kv=nkv, d=d), h


def test_layer_is_the_composition():
    P, shp, h = _tiny_layer(3)
    x = np.random.default_rng(4).standard_normal((6, h))
    out = oracle.layer_forward(x, P, **shp)
    n1 = oracle.rmsnorm_forward(x, P["g1"])["y"]
    x1 = x + oracle.attention_forward(n1, P["Wq"], P["Wk"], P["Wv"], P["Wo"],
                                      **shp)["Out"]
    n2 = oracle.rmsnorm_forward(x1, P["g2"])["y"]
    ref = x1 + oracle.mlp_forward(n2, P["W1"], P["W2"], act="swiglu")["Out"]
    np.testing.assert_allclose(out["Out"], ref, atol=1e-13)


def test_layer_backward_finite_differences():
    P, shp, h = _tiny_layer(5)
    r = np.random.default_rng(6)
    x = r.standard_normal((6, h))
    dout = r.standard_normal((6, h))

    def loss():
        return float((oracle.layer_forward(x, P, **shp)["Out"] * dout).sum())

    sv = oracle.layer_forward(x, P, **shp)
    g = oracle.layer_backward(dout, x, P, sv, **shp)
    assert_grad(g["dX"], loss, x)
    for k in ("g1", "Wq", "Wk", "Wv", "Wo", "g2", "W1", "W2"):
        assert_grad(g["d" + k], loss, P[k], max_entries=24)


def test_sampled_layer_with_sparse_upstream_matches_dense_oracle():
    # oracle.sampled.layer_sparse_upstream restates the layer for the
    # full-size GPU check; on small shapes (two sequences, GQA groups of 2,
    # rows in both sequences, a row at a sequence start) it must equal the
    # dense layer oracle given the same sparse upstream gradient
    rng = np.random.default_rng(11)
    b, s, h, nq, nkv, d, f = 2, 24, 64, 4, 2, 16, 96
    T = b * s
    P = {"g1": 1 + 0.1 * rng.standard_normal(h),
         "g2": 1 + 0.1 * rng.standard_normal(h),
         "Wq": 0.2 * rng.standard_normal((nq * d, h)),
         "Wk": 0.2 * rng.standard_normal((nkv * d, h)),
         "Wv": 0.2 * rng.standard_normal((nkv * d, h)),
         "Wo": 0.2 * rng.standard_normal((h, nq * d)),
         "W1": 0.2 * rng.standard_normal((2 * f, h)),
         "W2": 0.2 * rng.standard_normal((h, f))}
    x = rng.standard_normal((T, h))
    rows = [47, 30, 24, 23, 5]
    dOut = np.zeros((T, h))
    dOut[rows] = rng.standard_normal((len(rows), h))
    kw = dict(b=b, s=s, n_q=nq, n_kv=nkv, d=d)
    fo = oracle.layer_forward(x, P, **kw)
    go = oracle.layer_backward(dOut, x, P, fo, **kw)
    sm = oracle.sampled.layer_sparse_upstream(x, P, rows, dOut[rows],
                                              [0, 23, 24, 40], **kw)

    def rel(a, ref):
        return np.abs(a - ref).max() / np.abs(ref).max()

    for t in (0, 23, 24, 40):
        assert rel(sm["Out"][t], fo["Out"][t]) < 1e-12
    for k in ("dX", "dg1", "dg2", "dWk", "dWv"):
        assert rel(sm[k], go[k]) < 1e-12, k
    for k in ("dWq", "dWo", "dW1", "dW2"):
        L, R = sm[k]
        assert rel(L.T @ R, go[k]) < 1e-12, k
