"""Failure detection without a GPU fault: every in-kernel wait is bounded.

With the wait limit set to 1 ns, ordinary waits of the GEMM pipeline expire;
the kernel must record A4W4_ERR_TIMEOUT in the status word, drain its in-flight
copies and MMAs, free TMEM and return -- leaving the context usable, which
the follow-up call with the default limit checks."""

import numpy as np
import pytest
import torch

import mxfp4_a4w4_gemm_gb300 as a4w4
import workloads
from gpu_util import dev_bits, gemm_violations, host_bits
from oracle import gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mxfp4_a4w4_gemm_gb300 import build
    build.build()
    a4w4.lib()


@pytest.mark.parametrize("M,N,K", [(8, 7168, 4224), (300, 512, 4224), (1024, 5120, 1024)])
def test_expired_wait_is_reported_and_context_survives(M, N, K):
    A_bits, W_bits = workloads.dense_problem(M, N, K, "decode")
    Wq = torch.empty(a4w4.a4w4_weight_codes_bytes(N, K), dtype=torch.uint8, device="cuda")
    Ws = torch.empty(a4w4.a4w4_weight_scales_bytes(N, K), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_prepare_gemm_weight(dev_bits(W_bits), N, K, Wq, Ws)
    A = dev_bits(A_bits)
    ws_bytes = a4w4.a4w4_gemm_workspace_bytes(M, N, K)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_workspace_init(ws, ws_bytes)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert a4w4.a4w4_get_device_status() == 0
    a4w4.a4w4_set_wait_limit_ns(1)
    try:
        a4w4.a4w4_gemm(A, M, K, Wq, Ws, N, C, ws, ws_bytes)
        status = a4w4.a4w4_get_device_status()
    finally:
        a4w4.a4w4_set_wait_limit_ns(0)
    assert status == a4w4.A4W4_ERR_TIMEOUT
    assert a4w4.a4w4_get_device_status() == 0           # reading clears it
    # the context is intact: re-initialise the split-K counters and recompute
    a4w4.a4w4_workspace_init(ws, ws_bytes)
    a4w4.a4w4_gemm(A, M, K, Wq, Ws, N, C, ws, ws_bytes)
    assert a4w4.a4w4_get_device_status() == 0
    c = host_bits(C)
    rng = np.random.default_rng(1)
    ms, ns = rng.integers(0, M, 2000), rng.integers(0, N, 2000)
    ref, abs_sum, _ = gemm.gemm_a4w4_entries(A_bits, W_bits, ms, ns)
    assert gemm_violations(c[ms, ns], ref, abs_sum)[0].size == 0
