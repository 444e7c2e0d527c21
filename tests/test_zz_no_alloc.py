"""a4w4_gemm_noalloc: the dense GEMM entry point that allocates nothing.

It is for callers that cannot allocate device memory where they call the GEMM:
code under a framework allocator that owns all device memory, or a path that
cannot afford cudaMalloc's implicit synchronisation.  Its scratch (the
activation tiles quantised once, for M > 64 with N >= 4096 and every M > 128)
is a fixed 16 MiB array in the library.

Each case calls it twice in a row through the C ABI and checks both outputs
against the oracle with the tests' per-element tolerance, and bit for bit
against a4w4_gemm with a caller workspace (same plan, same kernels, same
reduction order).  The shapes cover a plan without scratch and plans whose
scratch holds the activation tiles, up to the largest workload shape.

This file is collected last on purpose; it passes alone in a fresh process
(the first call does the per-device set-up) and after the other tests."""

import numpy as np
import pytest
import torch

import mxfp4_a4w4_gemm_gb300 as a4w4
import workloads
from gpu_util import dev_bits, gemm_violations, host_bits
from oracle import gemm

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mxfp4_a4w4_gemm_gb300 import build
    build.build()
    a4w4.lib()


def prepared(W_bits):
    N, K = W_bits.shape
    Wq = torch.empty(a4w4.a4w4_weight_codes_bytes(N, K), dtype=torch.uint8, device="cuda")
    Ws = torch.empty(a4w4.a4w4_weight_scales_bytes(N, K), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_prepare_gemm_weight(dev_bits(W_bits), N, K, Wq, Ws)
    return Wq, Ws


CASES = [
    (8, 1536, 7168, "decode"),      # decode kernel, cluster split-K: no scratch
    (200, 512, 4224, "large"),      # activation tiles, 4 tiles run as 8 column halves
    (128, 8448, 7168, "large"),     # activation tiles, one row tile (33 tiles as 66 halves)
    (513, 1536, 4224, "stress"),    # activation tiles, ragged M, scale-edge blocks
    (1024, 5120, 1536, "large"),    # activation tiles, no split-K
    (2048, 8448, 7168, "large"),    # the largest workload shape (7.4 MiB of tiles)
]


@pytest.mark.parametrize("M,N,K,family", CASES, ids=[f"{m}x{n}x{k}" for m, n, k, _ in CASES])
def test_noalloc_matches_oracle_and_workspace_gemm_twice(M, N, K, family):
    ws_bytes = a4w4.a4w4_gemm_workspace_bytes(M, N, K)
    assert ws_bytes <= SCRATCH_BYTES
    A_bits, W_bits = workloads.dense_problem(M, N, K, family)
    Wq, Ws = prepared(W_bits)
    A = dev_bits(A_bits)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_workspace_init(ws, ws_bytes)
    C_ws = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    a4w4.a4w4_gemm(A, M, K, Wq, Ws, N, C_ws, ws, ws_bytes)
    assert a4w4.a4w4_get_device_status() == 0
    want = host_bits(C_ws)
    ref, abs_sum, _ = gemm.gemm_a4w4(A_bits, W_bits)
    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        a4w4.a4w4_gemm_noalloc(A, M, K, Wq, Ws, N, C)
        assert a4w4.a4w4_get_device_status() == 0
        got = host_bits(C)
        bad = gemm_violations(got, ref, abs_sum)[0]
        assert bad.size == 0, f"call {call}: {bad.size} of {got.size} outputs outside the oracle tolerance"
        assert np.array_equal(got, want), (f"call {call}: {int(np.sum(got != want))} outputs differ from "
                                           "a4w4_gemm's bits")


def test_noalloc_refuses_plans_beyond_its_scratch():
    # 4608 rows at K = 7168: 36 activation tiles x 28 K tiles x 17 KB =
    # 17.5 MB of scratch, more than 16 MiB.
    M, N, K = 4608, 256, 7168
    assert a4w4.a4w4_gemm_workspace_bytes(M, N, K) > SCRATCH_BYTES
    Wq, Ws = prepared(workloads.weight_bits(N, K))
    A = dev_bits(workloads.activation_bits(M, K))
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(a4w4.A4W4Error) as e:
        a4w4.a4w4_gemm_noalloc(A, M, K, Wq, Ws, N, C)
    assert e.value.code == a4w4.A4W4_ERR_WORKSPACE
