"""Pins of the oracle's elementwise primitives and dropout generator."""

import numpy as np
import pytest

import oracle
from _golden import load, matrix


def test_splitmix64_published_vector():
    g = load("splitmix64_seed1234567.txt")
    seed = int(g["seed"][0])
    expect = [int(v) for v in g["outputs"]]
    assert oracle.splitmix64_stream(seed, len(expect)) == expect


def test_splitmix64_vectorised_matches_stream():
    # the numpy finaliser on counter inputs reproduces the scalar stream
    seed = 1234567
    ref = oracle.splitmix64_stream(seed, 64)
    e = np.arange(64, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (e + np.uint64(1)) * np.uint64(0x9E3779B97F4A7C15)
    got = oracle.splitmix64_mix(z)
    assert [int(v) for v in got] == ref


def test_gelu_table_values():
    g = load("normal_cdf.txt")
    x = matrix(g["x"])
    phi = matrix(g["Phi"])
    np.testing.assert_allclose(oracle.gelu(x), x * phi, rtol=0, atol=2e-15)
    # odd symmetry of Φ: GeLU(-x) = -x·(1 - Φ(x))
    np.testing.assert_allclose(oracle.gelu(-x), -x * (1 - phi), rtol=0,
                               atol=2e-15)


def test_silu_table_value():
    g = load("normal_cdf.txt")
    s1 = float(g["sigmoid_1"][0])
    assert abs(oracle.silu(np.array([1.0]))[0] - s1) < 1e-15
    assert abs(oracle.silu(np.array([-1.0]))[0] + (1 - s1)) < 1e-15
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    # far tails: SiLU(x) → x for large x, → 0 for very negative x
    assert abs(oracle.silu(np.array([50.0]))[0] - 50.0) < 1e-12
    assert abs(oracle.silu(np.array([-50.0]))[0]) < 1e-18


@pytest.mark.parametrize("fn,grad", [(oracle.gelu, oracle.gelu_grad),
                                     (oracle.silu, oracle.silu_grad)])
def test_activation_grad_finite_difference(fn, grad):
    x = np.linspace(-6, 6, 241)
    eps = 1e-6
    fd = (fn(x + eps) - fn(x - eps)) / (2 * eps)
    np.testing.assert_allclose(grad(x), fd, rtol=0, atol=1e-8)


def test_dropout_threshold_and_fraction():
    assert oracle.dropout_threshold(0.0) == 0
    assert oracle.dropout_threshold(0.1) == 1677722       # round(0.1·2^24)
    assert oracle.dropout_threshold(0.5) == 1 << 23
    T, h, p = 2048, 2048, 0.1
    keep = oracle.dropout_keep(20260001, T, h, p)
    N = T * h
    q = 1 - oracle.dropout_threshold(p) / float(1 << 24)
    sigma = (N * q * (1 - q)) ** 0.5
    assert abs(keep.sum() - N * q) < 6 * sigma
    assert oracle.dropout_keep(5, 7, 9, 0.0).all()


def test_dropout_mask_is_the_stream():
    # element e = t·h + j uses draw e of the stream; top 24 bits vs threshold
    seed, rows, cols, p = 987654321, 3, 5, 0.3
    draws = oracle.splitmix64_stream(seed, rows * cols)
    thr = oracle.dropout_threshold(p)
    expect = np.array([(d >> 40) >= thr for d in draws]).reshape(rows, cols)
    assert (oracle.dropout_keep(seed, rows, cols, p) == expect).all()
    # a row offset selects the later draws
    more = oracle.splitmix64_stream(seed, 4 * cols)
    row3 = np.array([(d >> 40) >= thr for d in more[3 * cols:]])
    assert (oracle.dropout_keep(seed, 1, cols, p, row0=3)[0] == row3).all()
