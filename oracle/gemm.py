"""Dense A4W4 MXFP4 GEMM oracle (float64) -- TEST INFRASTRUCTURE ONLY.

"[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM", Summary and
Implementation: BF16 activations A [M, K] are quantised to MXFP4 along K,
weights W [N, K] are quantised once along K, the MXFP4 x MXFP4 products are
summed, and the output C [M, N] is BF16.  Rows m >= M do not exist (M-tail
masking); K is a multiple of 32 (the pages' scope asks K % 128 == 0).

Written out:

    a~ = decode(quant(A))   w~ = decode(quant(W))      (oracle.mxfp4)
    ref[m, n]  = sum_k a~[m, k] * w~[n, k]            float64
    abs[m, n]  = sum_k |a~[m, k] * w~[n, k]|          float64
    C[m, n]    = BF16_RNE(ref[m, n])

gemm_a16w4 is the A16WFP4 variant (BF16 activations unquantised, same
weights, same bound).

Every product a~ * w~ is exact in float64 (3 significant bits each, exponents
within range); the float64 sum (a library matmul) is within
K * 2**-53 * abs of the exact value, far below the acceptance bound

    |C_gpu - ref| <= 2**-8 * |ref| + 2**-20 * abs            (per element)

which covers the BF16 output rounding (half an ulp is at most 2**-8 * |ref|)
plus fp32 accumulation order on the GPU.  The bound is checked against the
unrounded ``ref``: checking against the rounded C would reject a legitimate
one-ulp disagreement next to a BF16 rounding midpoint.
"""

import numpy as np

from . import mxfp4

TOL_REL = 2.0 ** -8
TOL_ABS_SUM = 2.0 ** -20


def dequantized(bits):
    """BF16 bits [..., K] -> exact float64 values of their MXFP4 quantisation."""
    return mxfp4.quant_dequant(mxfp4.bf16_bits_to_f64(bits))


def gemm_a4w4(A_bits, W_bits):
    """Full oracle GEMM.  A_bits [M, K], W_bits [N, K] BF16 bit patterns.

    Returns (ref float64 [M, N], abs_sum float64 [M, N], C_bits uint16 [M, N]).
    """
    a = dequantized(A_bits)
    w = dequantized(W_bits)
    ref = a @ w.T
    abs_sum = np.abs(a) @ np.abs(w).T
    return ref, abs_sum, mxfp4.round_to_bf16_bits(ref)


def gemm_a4w4_entries(A_bits, W_bits, ms, ns):
    """Oracle values of selected output entries C[ms[i], ns[i]] only.

    Quantises just the rows of A and W that the sample touches, so any
    single entry of a large GEMM can be checked on its own.
    """
    ms = np.asarray(ms, dtype=np.int64)
    ns = np.asarray(ns, dtype=np.int64)
    um, im = np.unique(ms, return_inverse=True)
    un, inn = np.unique(ns, return_inverse=True)
    a = dequantized(np.asarray(A_bits)[um])
    w = dequantized(np.asarray(W_bits)[un])
    prod = a[im] * w[inn]
    ref = prod.sum(axis=1)
    abs_sum = np.abs(prod).sum(axis=1)
    return ref, abs_sum, mxfp4.round_to_bf16_bits(ref)


def gemm_a16w4(A_bits, W_bits):
    """A16WFP4 GEMM: BF16 activations against MXFP4 weights.

    "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM", Summary (the #4772
    bullet): BF16 activation x decoded MXFP4 weight, BF16 out.  The
    activations are used as they are (exact float64 values of the BF16
    inputs); only the weights are quantised (oracle.mxfp4), then

        ref[m, n] = sum_k a[m, k] * w~[n, k]       float64
        abs[m, n] = sum_k |a[m, k] * w~[n, k]|     float64
        C[m, n]   = BF16_RNE(ref[m, n])

    A product of a BF16 value (8 significant bits) and a decoded E2M1 value (2)
    is exact in float64.  Returns (ref, abs_sum, C_bits) like gemm_a4w4.
    """
    a = mxfp4.bf16_bits_to_f64(A_bits)
    w = dequantized(W_bits)
    ref = a @ w.T
    abs_sum = np.abs(a) @ np.abs(w).T
    return ref, abs_sum, mxfp4.round_to_bf16_bits(ref)


def tolerance(ref, abs_sum):
    """Per-element acceptance bound for a BF16 GEMM output against ``ref``."""
    return TOL_REL * np.abs(ref) + TOL_ABS_SUM * abs_sum
