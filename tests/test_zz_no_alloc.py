"""The RMSNorm backward entry point that allocates nothing.

Some callers cannot allocate device memory for scratch — code living under
another framework's memory pool, real-time loops that forbid cudaMalloc after
start-up, embeddings that pass the library only inputs and outputs.  For them
tp_rmsnorm_bwd_noalloc keeps its dγ partial sums in a fixed array inside the
library.  These checks call it through the C ABI on two calls in a row, the
second with a different shape and data so that contents left in the shared
array by the first call cannot leak into the second, and compare it with the
fp64 oracle (both error bounds) and with tp_rmsnorm_bwd, which takes caller
scratch and must give the same bits.  This file is collected last.
"""

import pytest
import torch

import oracle
from megatron_tensor_transformer_gate_gb300 import inputs as I
from _parity import check

pytestmark = pytest.mark.gpu


def _case(T, h, seed, dtype):
    x = I.normal((T, h), 1.0, seed + 1, "cuda", dtype)
    dy = I.normal((T, h), 1.0, seed + 2, "cuda", dtype)
    dres = I.normal((T, h), 1.0, seed + 3, "cuda", dtype)
    gamma = I.normal((h,), 0.02, seed + 4, "cuda", dtype, mean=1.0)
    return x, dy, dres, gamma


def _with_scratch(tp, x, dy, dres, gamma, rstd):
    T, h = x.shape
    dx = torch.empty_like(x)
    dg = torch.empty_like(gamma)
    scratch = torch.empty(tp.rmsnorm_bwd_scratch_bytes(T, h), dtype=torch.uint8,
                          device="cuda")
    tp.rmsnorm_bwd(dy, x, gamma, rstd, dx, dg, scratch, dres=dres)
    return dx, dg


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_oracle_and_scratch_entry_two_calls(tp, dtype):
    tol = "bf16" if dtype == torch.bfloat16 else "f32"
    eps = 1e-5
    for T, h, seed in ((1000, 8192, 20260100), (40, 520, 20260200)):
        x, dy, dres, gamma = _case(T, h, seed, dtype)
        y = torch.empty_like(x)
        rstd = torch.empty(T, dtype=torch.float32, device="cuda")
        tp.rmsnorm_fwd(x, gamma, y, rstd, eps)
        dx = torch.full_like(x, float("nan"))
        dg = torch.full_like(gamma, float("nan"))
        tp.rmsnorm_bwd_noalloc(dy, x, gamma, rstd, dx, dg, dres=dres)
        dx_s, dg_s = _with_scratch(tp, x, dy, dres, gamma, rstd)
        tp.device_status()
        # same kernels, same chunking: the same bits as the scratch entry
        assert torch.equal(dx, dx_s), f"dx T={T} h={h}"
        assert torch.equal(dg, dg_s), f"dgamma T={T} h={h}"
        o = oracle.rmsnorm_backward(I.to_f64(dy), I.to_f64(x),
                                    I.to_f64(gamma), eps, dres=I.to_f64(dres))
        check(dx, o["dx"], f"dx T={T} h={h}", tol)
        check(dg, o["dgamma"], f"dgamma T={T} h={h}", tol)


def test_noalloc_rejects_width_beyond_the_fixed_array(tp):
    T, h = 8, 8200
    x = torch.zeros(T, h, dtype=torch.bfloat16, device="cuda")
    gamma = torch.ones(h, dtype=torch.bfloat16, device="cuda")
    rstd = torch.ones(T, dtype=torch.float32, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.rmsnorm_bwd_noalloc(x, x, gamma, rstd, torch.empty_like(x),
                               torch.empty_like(gamma))
    assert e.value.code == 4
