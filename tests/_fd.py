"""Central finite differences of a scalar loss, for pinning oracle gradients."""

import numpy as np


def fd_grad(loss, arr, eps=1e-6, max_entries=None, rng=None):
    """d loss / d arr by central differences, entry by entry (in place edit).

    With ``max_entries`` only a random subset of entries is probed; the
    returned mask says which.
    """
    flat = arr.reshape(-1)
    idx = np.arange(flat.size)
    if max_entries is not None and flat.size > max_entries:
        rng = rng or np.random.default_rng(0)
        idx = rng.choice(flat.size, max_entries, replace=False)
    g = np.zeros(flat.size)
    probed = np.zeros(flat.size, dtype=bool)
    for i in idx:
        old = flat[i]
        flat[i] = old + eps
        lp = loss()
        flat[i] = old - eps
        lm = loss()
        flat[i] = old
        g[i] = (lp - lm) / (2 * eps)
        probed[i] = True
    return g.reshape(arr.shape), probed.reshape(arr.shape)


def assert_grad(analytic, loss, arr, rtol=1e-6, atol=1e-8, **kw):
    fd, probed = fd_grad(loss, arr, **kw)
    a = np.asarray(analytic)[probed]
    f = fd[probed]
    scale = max(np.abs(f).max(), 1e-30)
    err = np.abs(a - f).max()
    assert err <= atol + rtol * scale, f"max |analytic - fd| = {err:.3e} (scale {scale:.3e})"
