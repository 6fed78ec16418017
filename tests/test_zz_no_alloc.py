"""The RMSNorm backward entry point that allocates nothing.

Some callers cannot allocate device memory for scratch — code living under
another framework's memory pool, real-time loops that forbid cudaMalloc after
start-up, embeddings that pass the library only inputs and outputs.  For them
tp_rmsnorm_bwd_noalloc keeps its dγ partial sums in a fixed array inside the
library.  These checks call it through the C ABI and compare it with
tp_rmsnorm_bwd (which takes caller scratch) on two calls in a row, the second
with a different shape and data so that contents left in the shared array by
the first call cannot leak into the second.  This file is collected last.
"""

import pytest
import torch

from _parity import check

pytestmark = pytest.mark.gpu


def _case(T, h, seed, dtype=torch.bfloat16):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(T, h, generator=g, device="cuda").to(dtype)
    dy = torch.randn(T, h, generator=g, device="cuda").to(dtype)
    dres = torch.randn(T, h, generator=g, device="cuda").to(dtype)
    gamma = (1 + 0.02 * torch.randn(h, generator=g, device="cuda")).to(dtype)
    return x, dy, dres, gamma


def _reference(tp, x, dy, dres, gamma):
    T, h = x.shape
    y = torch.empty_like(x)
    rstd = torch.empty(T, dtype=torch.float32, device="cuda")
    tp.rmsnorm_fwd(x, gamma, y, rstd)
    dx = torch.empty_like(x)
    dg = torch.empty_like(gamma)
    scratch = torch.empty(tp.rmsnorm_bwd_scratch_bytes(T, h), dtype=torch.uint8,
                          device="cuda")
    tp.rmsnorm_bwd(dy, x, gamma, rstd, dx, dg, scratch, dres=dres)
    return rstd, dx, dg


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_scratch_entry_two_calls(tp, dtype):
    tol = "bf16" if dtype == torch.bfloat16 else "f32"
    for T, h, seed in ((1000, 8192, 1), (40, 520, 2)):
        x, dy, dres, gamma = _case(T, h, seed, dtype)
        rstd, dx_ref, dg_ref = _reference(tp, x, dy, dres, gamma)
        dx = torch.full_like(x, float("nan"))
        dg = torch.full_like(gamma, float("nan"))
        tp.rmsnorm_bwd_noalloc(dy, x, gamma, rstd, dx, dg, dres=dres)
        tp.device_status()
        check(dx, dx_ref, f"dx T={T} h={h}", tol)
        check(dg, dg_ref, f"dgamma T={T} h={h}", tol)


def test_noalloc_rejects_width_beyond_the_fixed_array(tp):
    T, h = 8, 8200
    x = torch.zeros(T, h, dtype=torch.bfloat16, device="cuda")
    gamma = torch.ones(h, dtype=torch.bfloat16, device="cuda")
    rstd = torch.ones(T, dtype=torch.float32, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.rmsnorm_bwd_noalloc(x, x, gamma, rstd, torch.empty_like(x),
                               torch.empty_like(gamma))
    assert e.value.code == 4
