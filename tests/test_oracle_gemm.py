"""Pins for oracle.gemm (CPU only).

* exact brute force: an independent pure-Python quantiser (frexp scale,
  nearest-value rounding) and exact rational sums, on tiny non-square shapes
  and on the full 16 x 256 x 256 workload;
* lossless special case: on-grid inputs make quantisation the identity, so
  the GEMM must equal a plain float64 matmul of the inputs;
* the pages' printed accuracy band ("[gfx950][FlyDSL] Add direct dense A4W4
  MXFP4 GEMM", Kernel microbenchmark: relative L2 2.42%-4.15% against a BF16
  emulation), read as the squared L2 ratio of the quantised GEMM against the
  unquantised one on N(0,1) x N(0,0.02) data.
"""

import math
from fractions import Fraction

import numpy as np

import workloads
from oracle import gemm, mxfp4

GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bf16_value(bits):
    return float(np.array([int(bits) << 16], np.uint32).view(np.float32)[0])


def brute_quant_row(vals):
    """Independent quantiser: returns exact Fractions of the dequantised row."""
    out = []
    for b in range(0, len(vals), 32):
        blk = vals[b:b + 32]
        amax = max(abs(v) for v in blk)
        if amax == 0:
            e = -127
        else:
            m, ex = math.frexp(amax)
            e = max(-127, min(127, ex - 1 - 2))
        scale = Fraction(2) ** e
        for v in blk:
            y = Fraction(abs(v)) / scale
            i = min(range(8), key=lambda j: (abs(y - Fraction(GRID[j])), j % 2))
            q = Fraction(GRID[i]) * scale
            out.append(-q if math.copysign(1.0, v) < 0 else q)
    return out


def exact_bf16_bits(q):
    """RNE of an exact rational to BF16 by comparing the two float32-neighbour candidates."""
    f = float(q)
    base = int(np.array([np.float32(f)], np.float32).view(np.uint32)[0] >> 16)
    best = None
    for c in (base - 1, base, base + 1):
        if not 0 <= c < 0x10000 or (c & 0x7F80) == 0x7F80:
            continue
        d = abs(Fraction(bf16_value(c)) - q)
        key = (d, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def brute_force_gemm(A_bits, W_bits):
    a = [brute_quant_row([bf16_value(x) for x in row]) for row in A_bits]
    w = [brute_quant_row([bf16_value(x) for x in row]) for row in W_bits]
    return [[sum(x * y for x, y in zip(ar, wr)) for wr in w] for ar in a]


def test_exact_bruteforce_tiny_nonsquare():
    rng = np.random.default_rng(0)
    A = workloads.to_bf16_bits(rng.standard_normal((3, 64)).astype(np.float32))
    W = workloads.to_bf16_bits((rng.standard_normal((5, 64)) * 0.02).astype(np.float32))
    A[1, 32:] = 0                       # a zero block
    exact = brute_force_gemm(A, W)
    ref, abs_sum, c = gemm.gemm_a4w4(A, W)
    assert ref.shape == (3, 5)
    for m in range(3):
        for n in range(5):
            assert abs(Fraction(ref[m, n]) - exact[m][n]) <= Fraction(64) * Fraction(2) ** -53 * Fraction(abs_sum[m, n])
            assert c[m, n] == exact_bf16_bits(exact[m][n])


def test_exact_bruteforce_small_workload():
    """The full 16 x 256 x 256 workload, every entry, exact."""
    (M, N, K), = workloads.SMALL
    A, W = workloads.dense_problem(M, N, K, "small")
    exact = brute_force_gemm(A, W)
    ref, abs_sum, c = gemm.gemm_a4w4(A, W)
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(ref[m, n]) - exact[m][n]) <= Fraction(K) * Fraction(2) ** -53 * Fraction(abs_sum[m, n])
            assert c[m, n] == exact_bf16_bits(exact[m][n])


def test_lossless_special_case_equals_plain_matmul():
    rng = np.random.default_rng(4)
    mags = np.array(GRID)

    def on_grid(rows, K, e_lo, e_hi):
        v = mags[rng.integers(0, 8, (rows, K))] * np.where(rng.random((rows, K)) < 0.5, -1, 1)
        v[:, ::32] = 4.0                                  # every block's amax in [4, 8)
        e = rng.integers(e_lo, e_hi, (rows, K // 32))
        return np.ldexp(v, np.repeat(e, 32, axis=1))

    A = on_grid(7, 256, -4, 4)
    W = on_grid(9, 256, -10, -2)
    A_bits = mxfp4.round_to_bf16_bits(A)
    W_bits = mxfp4.round_to_bf16_bits(W)
    assert np.array_equal(mxfp4.bf16_bits_to_f64(A_bits), A)
    ref, abs_sum, _ = gemm.gemm_a4w4(A_bits, W_bits)
    assert np.array_equal(ref, A @ W.T)                     # exact: small dyadic sums
    assert np.array_equal(abs_sum, np.abs(A) @ np.abs(W).T)


def test_entries_agree_with_full_gemm():
    A, W = workloads.dense_problem(33, 256, 512, "decode")
    ref, abs_sum, c = gemm.gemm_a4w4(A, W)
    rng = np.random.default_rng(9)
    ms, ns = rng.integers(0, 33, 200), rng.integers(0, 256, 200)
    r2, a2, c2 = gemm.gemm_a4w4_entries(A, W, ms, ns)
    assert np.allclose(r2, ref[ms, ns], rtol=1e-12, atol=0)
    assert np.array_equal(c2, c[ms, ns])


def _squared_rel_l2(A_bits, W_bits):
    ref, _, _ = gemm.gemm_a4w4(A_bits, W_bits)
    plain = mxfp4.bf16_bits_to_f64(A_bits) @ mxfp4.bf16_bits_to_f64(W_bits).T
    return float(np.sum((ref - plain) ** 2) / np.sum(plain ** 2))


def test_error_band_of_the_pages():
    for (M, N, K), family in (((128, 1536, 4224), "large"), ((64, 1536, 7168), "decode"), ((64, 7168, 768), "large")):
        A, W = workloads.dense_problem(M, N, K, family)
        r = _squared_rel_l2(A, W)
        assert 0.0242 <= r <= 0.0415, (M, N, K, family, r)


def test_tolerance_formula():
    t = gemm.tolerance(np.array([-256.0, 0.0]), np.array([1024.0, 2.0 ** 20]))
    assert t[0] == 1.0 + 2.0 ** -10 and t[1] == 1.0


def test_a16w4_matches_exact_rational_brute_force():
    """A16WFP4: BF16 activations used exactly, MXFP4 weights (independent
    quantiser), exact rational sums, BF16 rounding."""
    rng = np.random.default_rng(11)
    M, N, K = 3, 5, 64
    A = workloads.to_bf16_bits((rng.standard_normal((M, K)) * 3).astype(np.float32))
    W = workloads.to_bf16_bits((rng.standard_normal((N, K)) * 0.1).astype(np.float32))
    ref, abs_sum, cbits = gemm.gemm_a16w4(A, W)
    for m in range(M):
        a = [Fraction(bf16_value(v)) for v in A[m]]
        for n in range(N):
            w = brute_quant_row([bf16_value(v) for v in W[n]])
            exact = sum(x * y for x, y in zip(a, w))
            assert abs(Fraction(ref[m, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)
            assert cbits[m, n] == exact_bf16_bits(exact)
            assert abs(Fraction(abs_sum[m, n]) - sum(abs(x * y) for x, y in zip(a, w))) <= abs_sum[m, n] * 2 ** -50


def test_a16w4_equals_a4w4_when_activations_are_on_the_grid():
    """If every 32-block of A is already MXFP4-representable at the scale the
    rule picks (quantisation is the identity), A16WFP4 and A4W4 agree; with
    general A they differ (the activation quantisation is not skipped in A4W4)."""
    rng = np.random.default_rng(12)
    M, N, K = 4, 8, 128
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    vals = grid[rng.integers(0, 8, (M, K))] * np.where(rng.random((M, K)) < 0.5, -1.0, 1.0)
    vals[:, ::32] = 6.0                       # block max 6 -> scale 2^0 keeps the grid values
    A = workloads.to_bf16_bits(vals.astype(np.float32))
    W = workloads.weight_bits(N, K)
    r16, _, c16 = gemm.gemm_a16w4(A, W)
    r4, _, c4 = gemm.gemm_a4w4(A, W)
    assert np.array_equal(r16, r4) and np.array_equal(c16, c4)
    A2 = workloads.activation_bits(M, K)
    assert not np.allclose(gemm.gemm_a16w4(A2, W)[0], gemm.gemm_a4w4(A2, W)[0], rtol=1e-3)
