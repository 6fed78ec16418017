"""The failure path of the bounded device waits, without a GPU fault: a
kernel's wait on a barrier that nothing completes gives up after its limit,
the host reads TP_ERR_DEVICE_TIMEOUT from the status word, and the context
keeps working."""

import time

import numpy as np
import pytest
import torch

from _parity import f64

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_reports_and_the_context_survives(tp):
    tp.device_status()                    # start from a clear status word
    t0 = time.perf_counter()
    tp.selftest_wait_timeout()
    with pytest.raises(tp.TPError) as e:
        tp.device_status()
    elapsed = time.perf_counter() - t0
    assert e.value.code == 7              # TP_ERR_DEVICE_TIMEOUT
    assert 0.5 < elapsed < 60.0, elapsed  # the ~2 s limit, not a hang
    tp.device_status()                    # the read cleared the word
    g = torch.Generator().manual_seed(3)
    A = torch.randn(256, 192, generator=g).to(torch.bfloat16)
    Bm = torch.randn(320, 192, generator=g).to(torch.bfloat16)
    C = torch.empty((256, 320), dtype=torch.bfloat16, device="cuda")
    tp.gemm(A.cuda(), Bm.cuda(), C)
    tp.device_status()
    ref = f64(A) @ f64(Bm).T
    assert np.abs(f64(C) - ref).max() <= 8e-3 * np.abs(ref).max()
