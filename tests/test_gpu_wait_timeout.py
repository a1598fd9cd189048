"""The bounded wait that every pipelined kernel uses: a barrier that never
completes makes the wait give up after its limit, the kernel records
SAR_ERR_TIMEOUT and returns, the host reads that status back, and the
context stays usable for the next kernels."""

import time

import pytest
import torch

import chunked_prefill_hybrid_sar_gb300 as sar
from chunked_prefill_hybrid_sar_gb300 import _lib
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _gemm_still_right():
    g = synth.generator(3)
    a = synth.normal(g, (96, 256), dtype=torch.float16)
    w = synth.normal(g, (128, 256), 0.05, dtype=torch.float16)
    c = torch.empty(96, 128, dtype=torch.float32, device=DEV)
    sar.gemm(a.to(DEV), w.to(DEV), c, epilogue=sar.SAR_EPI_F32)
    sar.op_sync_status()
    ref = a.double() @ w.double().T
    assert ((c.double().cpu() - ref).abs().max() / ref.abs().max()).item() < 1e-5


@pytest.mark.parametrize("arrivals", [0, 1])
def test_wait_that_never_completes_reports_timeout(arrivals):
    sar.op_sync_status()  # nothing pending
    t0 = time.perf_counter()
    sar.op_wait_check(1_000_000, arrivals)  # 1 ms limit
    with pytest.raises(sar.SarError) as e:
        sar.op_sync_status()
    elapsed = time.perf_counter() - t0
    assert e.value.code == _lib.SAR_ERR_TIMEOUT
    assert "site 50" in str(e.value)
    assert elapsed < 1.0, elapsed  # gave up after about its limit, not the 2 s default
    sar.op_sync_status()  # the record was cleared by the read
    _gemm_still_right()


def test_wait_that_completes_reports_nothing():
    sar.op_wait_check(1_000_000, 2)
    sar.op_sync_status()
    _gemm_still_right()


def test_wait_check_rejects_bad_arguments():
    for limit, arrivals in ((0, 1), (-5, 1), (1000, 3), (1000, -1)):
        with pytest.raises(sar.SarError) as e:
            sar.op_wait_check(limit, arrivals)
        assert e.value.code == _lib.SAR_ERR_INVALID_ARG
