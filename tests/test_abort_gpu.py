"""The product kernel's abort path, run out on the GPU without a fault.

gemm_selftest_withheld_load launches the real GEMM kernel with the first
unit's producer withholding one ring stage: it issues neither the
expected-bytes arrive nor the loads, so the stage never fills. Every address
stays valid and no copy is left in flight. The waits behind the stage
(the epilogue's accumulator wait, the matrix issuer's ring wait, the
producer's own wait for a slot the issuer never frees) each run out after a
short limit; the first to do so records the launch's timeout and its site in
the device status word, the other roles see it and stop, and the launch
returns. The test checks that status, that the launch came back in bounded
time, and that the next GEMM on the same context is bit-exact.
"""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

# wait sites (role << 8 | barrier kind) that a withheld stage can run out first
SITES = {0x001: "producer empty slot", 0x002: "producer drain", 0x103: "issuer accumulator empty",
         0x104: "issuer full slot", 0x206: "epilogue accumulator full"}


@pytest.fixture(scope="module")
def dtg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tiled_gemm_gb300 as mod
    torch.cuda.set_device(0)
    mod.gemm_last_device_status()
    return mod


def _exact(dtg, M, N, K, seed, options=None):
    A, B = workloads.make_operands(M, N, K, "f16", "k", ("int", -3, 3), seed)
    C = dtg.gemm(A.cuda(), B.cuda(), out_dtype=torch.float32, options=options)
    status = dtg.gemm_last_device_status()
    assert status == (dtg.GEMM_OK, 0), status
    C_ref, _ = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, "f16", "k")
    assert np.array_equal(C.cpu().numpy().astype(np.float64), C_ref)


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("withhold_kb", [0, 5])
def test_withheld_stage_times_out_and_returns(dtg, cta_group, withhold_kb):
    M, N, K = 1024, 768, 1024
    A, B = workloads.make_operands(M, N, K, "f16", "k", ("int", -3, 3), 30 + withhold_kb)
    Ad, Bd = A.cuda(), B.cuda()
    C = torch.zeros(M, N, dtype=torch.float32, device="cuda")
    assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dtg.gemm_selftest_withheld_load(Ad, Bd, C, cta_group=cta_group, withhold_kb=withhold_kb, timeout_ms=20)
    status, site = dtg.gemm_last_device_status()      # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert status == dtg.GEMM_ERR_TIMEOUT, dtg.gemm_status_string(status)
    assert site in SITES, hex(site)
    assert 0.015 < elapsed < 2.0, elapsed             # ran out near its 20 ms limit, then returned
    assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)   # reading cleared it
    # the same context: the same product without a withheld stage is exact, with
    # the same tile shape and with the default plan
    _exact(dtg, M, N, K, 30 + withhold_kb, options={"cta_group": cta_group, "stream_k": 1})
    _exact(dtg, 4096, 4096, 512, 7)


def test_withheld_stage_out_of_range_is_rejected(dtg):
    A, B = workloads.make_operands(256, 256, 256, "f16", "k", ("int", -3, 3), 1)
    C = torch.zeros(256, 256, dtype=torch.float32, device="cuda")
    with pytest.raises(dtg.GemmError):
        # 256 K in 128-deep stages: k-blocks 0 and 1 only
        dtg.gemm_selftest_withheld_load(A.cuda(), B.cuda(), C, cta_group=2, withhold_kb=2, timeout_ms=20)
    assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)
