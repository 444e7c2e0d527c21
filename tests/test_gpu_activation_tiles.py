"""GPU parity: the MXFP4 activation operand tiles that the GEMM kernels build
from BF16 inputs -- inline in the producer warps of the decode and swap-AB
kernels, gathered and quantised per tile in the MoE GEMM1, or by the
quantise-once pre-pass of the large-M plans -- bit-exact against the oracle's
quantiser.

The product calls keep these tiles on chip; the test hooks of
include/a4w4_debug.h run the same plan and kernels and also store the tiles.
The dump is read back with the layout formulas of the headers (gpu_util), and
rows that do not exist (beyond M, padding slots of a routed block) and the K
padding must be zero."""

import numpy as np
import pytest
import torch

import mxfp4_a4w4_gemm_gb300 as a4w4
import workloads
from gpu_util import dev_bits, gemm_violations, host_bits, unshuffle_tiles
from oracle import gemm, mxfp4, moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mxfp4_a4w4_gemm_gb300 import build
    build.build()
    a4w4.lib()


def expected_tiles(A_bits, rows_total, KT):
    """Oracle quantisation of A padded with zero rows to rows_total and zero
    columns to KT * 256: (packed codes [rows_total, KT*128], scales [rows_total, KT*8])."""
    M, K = A_bits.shape
    pad = np.zeros((rows_total, KT * 256), dtype=np.uint16)
    pad[:M, :K] = A_bits
    return mxfp4.mxfp4_quant(pad)


def export_dense(A_bits, W_bits):
    M, K = A_bits.shape
    N = W_bits.shape[0]
    rows, x_tiles, KT = a4w4.a4w4_debug_gemm_activation_layout(M, N, K)
    Wq = torch.empty(a4w4.a4w4_weight_codes_bytes(N, K), dtype=torch.uint8, device="cuda")
    Ws = torch.empty(a4w4.a4w4_weight_scales_bytes(N, K), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_prepare_gemm_weight(dev_bits(W_bits), N, K, Wq, Ws)
    ws_bytes = a4w4.a4w4_gemm_workspace_bytes(M, N, K)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_workspace_init(ws, ws_bytes)
    atoms = x_tiles * KT
    dump = torch.full((atoms * (rows * 128 + 1024),), 0xA5, dtype=torch.uint8, device="cuda")
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    a4w4.a4w4_debug_gemm_export(dev_bits(A_bits), M, K, Wq, Ws, N, C, ws, ws_bytes, dump, dump.numel())
    assert a4w4.a4w4_get_device_status() == 0
    d = dump.cpu().numpy()
    codes, scales = unshuffle_tiles(d[:atoms * rows * 128], d[atoms * rows * 128:], rows, x_tiles, KT)
    return codes, scales, rows * x_tiles, KT, host_bits(C)


def assert_tiles_exact(A_bits, W_bits, check_output=True):
    codes, scales, rows_total, KT, c = export_dense(A_bits, W_bits)
    eq, es = expected_tiles(A_bits, rows_total, KT)
    bad_s = np.argwhere(scales != es)
    bad_q = np.argwhere(codes != eq)
    assert bad_s.size == 0, f"{len(bad_s)} scale bytes differ, first (row, block) {bad_s[:5].tolist()}"
    assert bad_q.size == 0, f"{len(bad_q)} code bytes differ, first (row, byte) {bad_q[:5].tolist()}"
    if check_output:      # the export changes nothing in the GEMM itself
        ref, abs_sum, _ = gemm.gemm_a4w4(A_bits, W_bits)
        assert gemm_violations(c, ref, abs_sum)[0].size == 0


# (M, N, K, input family): one or more shapes per producer path and plan
DENSE_CASES = [
    (1, 7168, 4224, "decode"),      # decode kernel, 16-token tile, K splits
    (8, 1536, 7168, "decode"),      # decode kernel, 16 K splits
    (16, 7168, 768, "decode"),      # decode kernel, one CTA holds K
    (32, 1536, 7168, "decode"),     # decode kernel, 32-token tile
    (32, 7168, 768, "decode"),      # decode kernel, two 16-token tiles (one CTA holds K)
    (24, 1536, 1024, "stress"),     # two 16-token tiles, the second ragged; 4-deep ring
    (32, 7168, 4224, "decode"),     # swap-AB, 32-token tile
    (1, 1536, 4224, "stress"),      # M tails on the scale-edge blocks
    (17, 1536, 4224, "stress"),
    (37, 1536, 4224, "stress"),     # swap-AB, 64-token tile
    (100, 1536, 4224, "stress"),    # swap-AB, 128-token tile
    (65, 7168, 4224, "stress"),     # quantise-once pre-pass, one tile, rows past M zero
    (513, 1536, 4224, "stress"),    # quantise-once pre-pass, ragged last tile
    (2047, 1536, 4224, "stress"),
]


@pytest.mark.parametrize("M,N,K,family", DENSE_CASES, ids=[f"{f}-{m}x{n}x{k}" for m, n, k, f in DENSE_CASES])
def test_dense_activation_tiles_bit_exact(M, N, K, family):
    A_bits, W_bits = workloads.dense_problem(M, N, K, family)
    assert_tiles_exact(A_bits, W_bits, check_output=M <= 1024)


def test_every_bf16_value_through_the_fused_quant():
    """All finite BF16 patterns in 32-blocks under several block maxima, as the
    rows of one decode-kernel GEMM (16 rows x 4096 K per launch)."""
    allbits = np.arange(0x10000, dtype=np.uint32)
    finite = allbits[(allbits & 0x7F80) != 0x7F80].astype(np.uint16)
    x = np.concatenate([finite, np.zeros((-finite.size) % 32, np.uint16)]).reshape(-1, 32)
    W_bits = workloads.weight_bits(256, 4096)
    for lead in (None, 0x3F80, 0x7F7F, 0x0080):
        y = x.copy()
        if lead is not None:
            y[:, 0] = lead
        flat = y.reshape(-1)
        flat = np.concatenate([flat, np.zeros((-flat.size) % (16 * 4096), np.uint16)]).reshape(-1, 16 * 4096)
        for chunk in flat:
            assert_tiles_exact(chunk.reshape(16, 4096), W_bits, check_output=False)


def test_moe_gathered_tiles_bit_exact():
    """MoE GEMM1: the tiles of the gathered token rows, quantised inline per
    tile (no workspace) and gathered from rows quantised once (workspace)."""
    T, n_exp, topk, Dm, inter = 37, 5, 3, 768, 128
    X = workloads.stress_activation_bits(T, Dm)
    ids = workloads.moe_topk_ids(T, n_exp, topk)
    W1 = np.stack([workloads.moe_expert_weight_bits(e, 2 * inter, Dm) for e in range(n_exp)])
    W1q = torch.empty(a4w4.a4w4_moe_w1_codes_bytes(n_exp, 2 * inter, Dm), dtype=torch.uint8, device="cuda")
    W1s = torch.empty(a4w4.a4w4_moe_w1_scales_bytes(n_exp, 2 * inter, Dm), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_moe_prepare_w1(dev_bits(W1), n_exp, 2 * inter, Dm, W1q, W1s)
    maxb = a4w4.a4w4_moe_max_blocks(T, topk, n_exp, 128)
    rows = torch.empty(maxb * 128, dtype=torch.int32, device="cuda")
    bexp = torch.empty(maxb, dtype=torch.int32, device="cuda")
    nb = torch.empty(1, dtype=torch.int32, device="cuda")
    swsb = a4w4.a4w4_moe_sort_workspace_bytes(T, topk, n_exp)
    sws = torch.empty(swsb, dtype=torch.uint8, device="cuda")
    a4w4.a4w4_moe_sort(torch.from_numpy(ids).cuda(), T, topk, n_exp, 128, rows, bexp, nb, sws, swsb)
    er, _, enb = moe.sort_routed_rows(ids, n_exp, 128)
    KT = Dm // 256
    eq_tok, es_tok = mxfp4.mxfp4_quant(X)
    for prequant in (False, True):
        ws, wsb = (None, 0)
        if prequant:
            wsb = a4w4.a4w4_moe_gemm1_workspace_bytes(T, Dm)
            ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        out_q = torch.empty((T * topk, inter // 2), dtype=torch.uint8, device="cuda")
        out_s = torch.empty((T * topk, inter // 32), dtype=torch.uint8, device="cuda")
        atoms = maxb * KT
        dump = torch.full((atoms * (16384 + 1024),), 0xA5, dtype=torch.uint8, device="cuda")
        a4w4.a4w4_debug_moe_gemm1_export(dev_bits(X), T, Dm, rows, bexp, nb, topk, W1q, W1s, n_exp, inter, out_q,
                                         out_s, ws, wsb, dump, dump.numel())
        assert a4w4.a4w4_get_device_status() == 0
        d = dump.cpu().numpy()
        codes, scales = unshuffle_tiles(d[:atoms * 16384], d[atoms * 16384:], 128, maxb, KT)
        eq = np.zeros_like(codes)
        es = np.zeros_like(scales)
        valid = er < T * topk
        eq[:enb * 128][valid] = eq_tok[er[valid] // topk]
        es[:enb * 128][valid] = es_tok[er[valid] // topk]
        assert np.array_equal(scales, es), f"prequant={prequant}: {int(np.sum(scales != es))} scale bytes differ"
        assert np.array_equal(codes, eq), f"prequant={prequant}: {int(np.sum(codes != eq))} code bytes differ"
