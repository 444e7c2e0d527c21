"""GPU parity: the A16WFP4 GEMM (BF16 activations, not quantised, x MXFP4
weights prepared by a4w4_prepare_gemm_weight) against the oracle's
gemm_a16w4, element by element, with |C - ref| <= 2^-8 |ref| + 2^-20 sum|a w|
(float64 ref before rounding); rows >= M never written."""

import numpy as np
import pytest
import torch

import mxfp4_a4w4_gemm_gb300 as a4w4
import workloads
from gpu_util import dev_bits, gemm_violations
from oracle import gemm

pytestmark = pytest.mark.gpu

GUARD_ROWS = 2
CANARY = 0x7FC1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mxfp4_a4w4_gemm_gb300 import build
    build.build()
    a4w4.lib()


def run(A_bits, W_bits, flags=0):
    M, K = A_bits.shape
    N = W_bits.shape[0]
    Wq = torch.empty(a4w4.a4w4_weight_codes_bytes(N, K), dtype=torch.uint8, device="cuda")
    Ws = torch.empty(a4w4.a4w4_weight_scales_bytes(N, K), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_prepare_gemm_weight(dev_bits(W_bits), N, K, Wq, Ws)
    C = torch.full((M + GUARD_ROWS, N), CANARY, dtype=torch.int16, device="cuda")
    a4w4.a4w4_gemm_a16w4(dev_bits(A_bits), M, K, Wq, Ws, N, C, flags)
    assert a4w4.a4w4_get_device_status() == 0
    out = C.cpu().numpy().view(np.uint16)
    assert np.all(out[M:] == CANARY), "rows >= M were written"
    return out[:M]


CASES = [(1, 7168, 4224, "decode"), (8, 1536, 7168, "decode"), (32, 7168, 768, "decode"),
         (16, 256, 256, "small"), (17, 512, 1024, "large"), (40, 256, 384, "large"), (100, 1536, 4224, "large"),
         (1, 256, 16384, "large"), (37, 1536, 4224, "stress"), (3, 2048, 2304, "decode"),
         (200, 512, 1024, "large"), (129, 256, 384, "stress")]


@pytest.mark.parametrize("M,N,K,family", CASES, ids=[f"{f}-{m}x{n}x{k}" for m, n, k, f in CASES])
def test_a16w4_every_output(M, N, K, family):
    A, W = workloads.dense_problem(M, N, K, family)
    c = run(A, W)
    ref, abs_sum, cref = gemm.gemm_a16w4(A, W)
    bad = gemm_violations(c, ref, abs_sum)
    assert bad[0].size == 0, (f"{bad[0].size} of {c.size} outside tolerance, first (m, n) "
                              f"{list(zip(bad[0][:5].tolist(), bad[1][:5].tolist()))}")
    assert np.mean(c == cref) > 0.9


def test_a16w4_is_not_a4w4():
    """On general activations the A16WFP4 result follows the unquantised
    activations (and differs from the A4W4 result of the same inputs)."""
    A, W = workloads.dense_problem(8, 512, 1024, "large")
    c = run(A, W)
    r16, s16, _ = gemm.gemm_a16w4(A, W)
    r4, _, _ = gemm.gemm_a4w4(A, W)
    assert gemm_violations(c, r16, s16)[0].size == 0
    assert np.mean(np.abs(r16 - r4) > gemm.tolerance(r16, s16)) > 0.5


def test_a16w4_weight_prefetch_back_to_back():
    M, N, K = 8, 1536, 4224
    problems = [workloads.dense_problem(M, N, K, "decode", seed=200 + j) for j in range(3)]
    outs = [run(A, W, flags=a4w4.A4W4_GEMM_WEIGHT_PREFETCH) for A, W in problems]
    for (A, W), c in zip(problems, outs):
        ref, abs_sum, _ = gemm.gemm_a16w4(A, W)
        assert gemm_violations(c, ref, abs_sum)[0].size == 0


@pytest.mark.parametrize("M,N,K", [(5, 256, 1024), (20, 512, 2304)])
def test_a16w4_wide_scale_range(M, N, K):
    """Weight blocks whose E8M0 scales span 2^-127 .. 2^124 (decoded weights
    down to BF16 subnormals and up near BF16's largest binade), each against
    activations of the reciprocal magnitude: every output within tolerance."""
    A, W = workloads.wide_scale_problem(M, N, K)
    c = run(A, W)
    ref, abs_sum, _ = gemm.gemm_a16w4(A, W)
    bad = gemm_violations(c, ref, abs_sum)
    assert bad[0].size == 0, (f"{bad[0].size} of {c.size} outside tolerance, first (m, n) "
                              f"{list(zip(bad[0][:5].tolist(), bad[1][:5].tolist()))}")


@pytest.mark.parametrize("M,N,K", [(1, 7168, 4224), (32, 1536, 7168)])
def test_a16w4_bitwise_deterministic(M, N, K):
    """Split-K partials are summed in cluster-rank order: repeated runs agree bit for bit."""
    A, W = workloads.dense_problem(M, N, K, "decode")
    c1 = run(A, W)
    c2 = run(A, W)
    assert np.array_equal(c1, c2)


@pytest.mark.parametrize("M,N,K", [(1, 7168, 4224), (32, 1536, 7168)])
def test_a16w4_expired_wait_is_reported_and_context_survives(M, N, K):
    """With a 1 ns wait limit the kernel's waits expire: it reports
    A4W4_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and returns; the
    next call with the default limit gives the same bits as a normal run."""
    A, W = workloads.dense_problem(M, N, K, "decode")
    want = run(A, W)
    Wq = torch.empty(a4w4.a4w4_weight_codes_bytes(N, K), dtype=torch.uint8, device="cuda")
    Ws = torch.empty(a4w4.a4w4_weight_scales_bytes(N, K), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_prepare_gemm_weight(dev_bits(W), N, K, Wq, Ws)
    C = torch.empty((M, N), dtype=torch.int16, device="cuda")
    assert a4w4.a4w4_get_device_status() == 0
    a4w4.a4w4_set_wait_limit_ns(1)
    try:
        a4w4.a4w4_gemm_a16w4(dev_bits(A), M, K, Wq, Ws, N, C, 0)
        status = a4w4.a4w4_get_device_status()
    finally:
        a4w4.a4w4_set_wait_limit_ns(0)
    assert status == a4w4.A4W4_ERR_TIMEOUT
    assert a4w4.a4w4_get_device_status() == 0
    a4w4.a4w4_gemm_a16w4(dev_bits(A), M, K, Wq, Ws, N, C, 0)
    assert a4w4.a4w4_get_device_status() == 0
    assert np.array_equal(C.cpu().numpy().view(np.uint16), want)
