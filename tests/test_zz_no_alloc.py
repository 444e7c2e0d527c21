"""a4w4_gemm_noalloc: the GEMM entry point that allocates nothing, for callers
that cannot allocate device memory where they call the GEMM (a framework
allocator owns all device memory, or cudaMalloc's implicit synchronisation is
not acceptable on that path).  Its split-K scratch is a fixed 16 MiB array in
the library.  Checked through the C ABI against a4w4_gemm (caller workspace)
within the tests' per-element tolerance, on two calls in a row.

This file is collected last on purpose; it passes alone in a fresh process
(the first call does the per-device set-up) and after the other tests."""

import numpy as np
import pytest
import torch

import mxfp4_a4w4_gemm_gb300 as a4w4
import workloads
from gpu_util import dev_bits, host_bits
from oracle import gemm, mxfp4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mxfp4_a4w4_gemm_gb300 import build
    build.build()
    a4w4.lib()


def prepared(N, K):
    W_bits = workloads.weight_bits(N, K)
    Wq = torch.empty(a4w4.a4w4_weight_codes_bytes(N, K), dtype=torch.uint8, device="cuda")
    Ws = torch.empty(a4w4.a4w4_weight_scales_bytes(N, K), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_prepare_gemm_weight(dev_bits(W_bits), N, K, Wq, Ws)
    return W_bits, Wq, Ws


@pytest.mark.parametrize("M,N,K", [(8, 1536, 7168), (1, 7168, 4224), (32, 7168, 768), (200, 512, 4224)])
def test_noalloc_matches_workspace_gemm_twice(M, N, K):
    A_bits = workloads.decode_activation_bits(M, K)
    W_bits, Wq, Ws = prepared(N, K)
    A = dev_bits(A_bits)
    ws_bytes = a4w4.a4w4_gemm_workspace_bytes(M, N, K)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_workspace_init(ws, ws_bytes)
    C_ws = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    a4w4.a4w4_gemm(A, M, K, Wq, Ws, N, C_ws, ws, ws_bytes)
    ref_bits = host_bits(C_ws)
    ref = mxfp4.bf16_bits_to_f64(ref_bits)
    _, abs_sum, _ = gemm.gemm_a4w4(A_bits, W_bits)
    tol = gemm.tolerance(ref, abs_sum)
    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        a4w4.a4w4_gemm_noalloc(A, M, K, Wq, Ws, N, C)
        assert a4w4.a4w4_get_device_status() == 0
        got = mxfp4.bf16_bits_to_f64(host_bits(C))
        bad = ~(np.abs(got - ref) <= tol)
        assert not bad.any(), f"call {call}: {int(bad.sum())} outputs differ from a4w4_gemm beyond tolerance"


def test_noalloc_refuses_plans_beyond_its_scratch():
    # M = 129..256 with N = 1536 splits K 12 ways over 12 tiles of 128x256 fp32
    # partials: 12 * 12 * 128 KiB = 18 MiB of scratch, more than 16 MiB.
    M, N, K = 200, 1536, 7168
    assert a4w4.a4w4_gemm_workspace_bytes(M, N, K) > 16 << 20
    _, Wq, Ws = prepared(N, K)
    A = dev_bits(workloads.activation_bits(M, K))
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(a4w4.A4W4Error) as e:
        a4w4.a4w4_gemm_noalloc(A, M, K, Wq, Ws, N, C)
    assert e.value.code == a4w4.A4W4_ERR_WORKSPACE
