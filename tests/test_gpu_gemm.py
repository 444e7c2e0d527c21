"""GPU parity: the dense A4W4 GEMM against the oracle, element by element,
with |C - ref| <= 2^-8 |ref| + 2^-20 sum|a w| (float64 ref, before rounding)."""

import numpy as np
import pytest
import torch

import mxfp4_a4w4_gemm_gb300 as a4w4
import workloads
from gpu_util import dev_bits, gemm_violations, host_bits
from oracle import gemm

pytestmark = pytest.mark.gpu

GUARD_ROWS = 3
CANARY = 0x7FC1        # a NaN pattern that the GEMM never writes


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mxfp4_a4w4_gemm_gb300 import build
    build.build()
    a4w4.lib()


class Prepared:
    def __init__(self, W_bits):
        self.N, self.K = W_bits.shape
        self.Wq = torch.empty(a4w4.a4w4_weight_codes_bytes(self.N, self.K), dtype=torch.uint8, device="cuda")
        self.Ws = torch.empty(a4w4.a4w4_weight_scales_bytes(self.N, self.K), dtype=torch.uint8, device="cuda")
        a4w4.a4w4_prepare_gemm_weight(dev_bits(W_bits), self.N, self.K, self.Wq, self.Ws)


def run_gemm(A_bits, prep, ws=None):
    M, K = A_bits.shape
    N = prep.N
    ws_bytes = a4w4.a4w4_gemm_workspace_bytes(M, N, K)
    if ws is None or ws.numel() < ws_bytes:
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
        a4w4.a4w4_workspace_init(ws, ws_bytes)
    C = torch.full((M + GUARD_ROWS, N), 0, dtype=torch.int16, device="cuda")
    C.fill_(CANARY - 0x10000 if CANARY >= 0x8000 else CANARY)
    a4w4.a4w4_gemm(dev_bits(A_bits), M, K, prep.Wq, prep.Ws, N, C, ws, ws_bytes)
    assert a4w4.a4w4_get_device_status() == 0
    out = C.cpu().numpy().view(np.uint16)
    assert np.all(out[M:] == CANARY), "rows >= M were written"
    return out[:M], ws


def check_full(A_bits, W_bits, prep=None):
    prep = prep or Prepared(W_bits)
    c, _ = run_gemm(A_bits, prep)
    ref, abs_sum, cref = gemm.gemm_a4w4(A_bits, W_bits)
    bad = gemm_violations(c, ref, abs_sum)
    assert bad[0].size == 0, (f"{bad[0].size} of {c.size} outside tolerance; first (m, n): "
                              f"{list(zip(bad[0][:5].tolist(), bad[1][:5].tolist()))}")
    return c, cref


def test_small_workload_full():
    (M, N, K), = workloads.SMALL
    A, W = workloads.dense_problem(M, N, K, "small")
    c, cref = check_full(A, W)
    assert np.mean(c == cref) > 0.95       # most outputs round to the same BF16


@pytest.mark.parametrize("M", [1, 2, 15, 16, 17, 31, 33, 64, 65, 100, 128, 129, 255, 300])
def test_ragged_m_spans_tiles(M):
    N, K = 512, 768
    A, W = workloads.dense_problem(M, N, K, "decode", seed=M)
    check_full(A, W)


@pytest.mark.parametrize("M,N,K", [(8, 256, 128), (8, 256, 384), (200, 768, 4224), (40, 1536, 4224),
                                   (3, 2048, 2304), (130, 256, 256),
                                   # K ranges longer than a CTA's operand rings (several fill/drain rounds)
                                   (1, 256, 16384), (1, 256, 20480), (9, 256, 17408), (24, 512, 12288),
                                   (50, 256, 10368),
                                   # decode kernel with 16 K splits filling the grid (uneven K ranges)
                                   (16, 1536, 7168), (17, 1536, 4224), (32, 512, 7168),
                                   # large-M tiles without split-K: one K tile; K range longer than the ring
                                   (256, 512, 256), (1024, 5120, 1536),
                                   # persistent large-M walk: two tiles per CTA and a ragged last row
                                   # tile; a last partial wave run as 128-column halves after a full tile;
                                   # K = 128, one K tile half of which is padding; the switch from the
                                   # whole-tile ring (4 stages of one K tile) to the half-unit ring (3
                                   # stages of two K tiles) after 5 K tiles, the last half stage single
                                   (1100, 8192, 512), (1200, 4096, 512), (1100, 8192, 128),
                                   (1200, 4096, 1280)])
def test_k_tails_and_shapes(M, N, K):
    A, W = workloads.dense_problem(M, N, K, "large", seed=K)
    check_full(A, W)


def test_stress_blocks_small():
    A = workloads.stress_activation_bits(37, 4224)
    W = workloads.weight_bits(256, 4224)
    check_full(A, W)


def test_deterministic_and_workspace_reuse():
    A, W = workloads.dense_problem(8, 1536, 7168, "decode")
    prep = Prepared(W)
    c1, ws = run_gemm(A, prep)
    c2, _ = run_gemm(A, prep, ws)
    c3, _ = run_gemm(A, prep, ws)
    assert np.array_equal(c1, c2) and np.array_equal(c2, c3)


ALL_SHAPES = ([("decode", s) for s in workloads.DECODE_SWEEP] + [("large", s) for s in workloads.LARGE_M_SWEEP]
              + [("stress", s) for s in workloads.TAIL_STRESS])


@pytest.mark.parametrize("family,shape", ALL_SHAPES, ids=[f"{f}-{m}x{n}x{k}" for f, (m, n, k) in ALL_SHAPES])
def test_full_size_every_output(family, shape):
    """Every workload shape at full size, in the launch configuration the bench
    times (same plan, workspace-backed), every output checked against the
    oracle (2048 x 8448 x 7168: 17.3 M outputs, ~2.5e11 float64 multiply-adds)."""
    M, N, K = shape
    A, W = workloads.dense_problem(M, N, K, family)
    c, _ = run_gemm(A, Prepared(W))
    ref, abs_sum, cref = gemm.gemm_a4w4(A, W)
    bad = gemm_violations(c, ref, abs_sum)
    assert bad[0].size == 0, (f"{bad[0].size} of {c.size} outputs outside tolerance, first (m, n) "
                              f"{list(zip(bad[0][:5].tolist(), bad[1][:5].tolist()))}")
    assert np.all((c & 0x7F80) != 0x7F80), "NaN or Inf in the output"
    print(f"{M}x{N}x{K}: {c.size} outputs within tolerance, {np.mean(c == cref):.4%} equal to the rounded oracle")


def test_argument_errors():
    prep = Prepared(workloads.weight_bits(256, 256))
    A = dev_bits(workloads.activation_bits(4, 256))
    C = torch.empty((4, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(a4w4.A4W4Error) as e:
        a4w4.a4w4_gemm(A, 4, 256, prep.Wq, prep.Ws, 300, C)
    assert e.value.code == a4w4.A4W4_ERR_ARG
    ws_bytes = a4w4.a4w4_gemm_workspace_bytes(4, 256, 256)
    if ws_bytes:
        with pytest.raises(a4w4.A4W4Error) as e:
            a4w4.a4w4_gemm(A, 4, 256, prep.Wq, prep.Ws, 256, C, None, 0)
        assert e.value.code == a4w4.A4W4_ERR_WORKSPACE


@pytest.mark.parametrize("M", [65, 100, 128])
def test_mid_m_normal_orientation(M):
    """64 < M <= 128 with N >= 4096: tokens on the MMA's 128-row side, weights
    on N = 256, split-K reduced inside a cluster."""
    N, K = 4096, 1792
    A, W = workloads.dense_problem(M, N, K, "decode", seed=M + 1)
    check_full(A, W)


@pytest.mark.parametrize("M,N,K", [(1, 1536, 7168), (8, 7168, 768), (32, 1536, 4224), (512, 512, 1024)])
def test_weight_prefetch_back_to_back(M, N, K):
    """With weight prefetch on, each GEMM may stream its (unchanged) weights
    before the previous kernel on the stream has finished: results of several
    calls issued back to back, each on other weights and activations, match
    the oracle."""
    problems = [workloads.dense_problem(M, N, K, "decode", seed=100 + j) for j in range(3)]
    preps = [Prepared(W) for _, W in problems]
    torch.cuda.synchronize()
    outs = []
    ws_bytes = a4w4.a4w4_gemm_workspace_bytes(M, N, K)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_workspace_init(ws, ws_bytes)
    for (A, _), prep in zip(problems, preps):
        C = torch.empty((M, N), dtype=torch.int16, device="cuda")
        a4w4.a4w4_gemm_ex(dev_bits(A), M, K, prep.Wq, prep.Ws, N, C, ws, ws_bytes,
                          flags=a4w4.A4W4_GEMM_WEIGHT_PREFETCH)
        outs.append(C)
    assert a4w4.a4w4_get_device_status() == 0
    for (A, W), C in zip(problems, outs):
        ref, abs_sum, _ = gemm.gemm_a4w4(A, W)
        c = C.cpu().numpy().view(np.uint16)
        bad = gemm_violations(c, ref, abs_sum)
        assert bad[0].size == 0, f"{bad[0].size} of {c.size} outside tolerance"


@pytest.mark.parametrize("M,N,K,family", [
    (1, 7168, 4224, "decode"),    # decode kernel: st.async split-K slices summed in rank order
    (32, 7168, 4224, "decode"),   # swap-AB: cluster push, owner sums in split order
    (200, 1536, 7168, "large"),   # quantise-once tiles, persistent walk of column halves (no split-K)
    (2048, 8448, 7168, "large"),  # persistent walk: 3 whole tiles per CTA, the last wave as halves
], ids=lambda v: str(v))
def test_bitwise_deterministic_per_plan(M, N, K, family):
    """Every split-K reduction sums in a fixed order, and the persistent walk
    has none: three runs give the same bits."""
    A, W = workloads.dense_problem(M, N, K, family)
    prep = Prepared(W)
    c1, ws = run_gemm(A, prep)
    c2, _ = run_gemm(A, prep, ws)
    c3, _ = run_gemm(A, prep)
    assert np.array_equal(c1, c2) and np.array_equal(c2, c3)
