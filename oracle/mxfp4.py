"""MXFP4 number format and block quantiser (float64, numpy) -- test oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What is computed, and where it comes from
-----------------------------------------
"[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM", Summary: both operands of
the A4W4 product are MXFP4 -- 4-bit E2M1 element codes sharing one 8-bit E8M0
power-of-two scale.  The pages never state how the scale is chosen; this file
uses the OCP Microscaling (MX) v1.0 rule, written out here:

  For every 32 consecutive elements x_0..x_31 along the reduction axis:
    amax = max_i |x_i|
    e    = floor(log2(amax)) - 2          (e = -127 when amax == 0)
    e    = clamp(e, -127, 127)            (E8M0 code = e + 127)
    y_i  = |x_i| * 2**-e                  (exact in float64)
    q_i  = nearest E2M1 magnitude to y_i; an exact midpoint goes to the
           magnitude whose mantissa bit is 0 ("ties to even"); y_i >= 6
           gives 6 (saturation; E2M1 has no infinity)
    code = sign_bit(x_i) << 3 | index(q_i)    (a negative x that rounds to
           zero keeps its sign: code 8)

E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit):
  index 0..7  ->  0, 0.5, 1, 1.5, 2, 3, 4, 6      (index = code & 7;
  the mantissa bit is index & 1, so "ties to even" = ties to the even index)

Packing (a reading, the pages are silent): element 2j sits in the low nibble
of byte j, element 2j+1 in the high nibble.  Plain scale layout: one E8M0 byte
per 32-block, row-major [rows, cols/32].

Float inputs are finite (NaN/Inf are outside the precondition).
"""

import numpy as np

# E2M1 magnitudes by 3-bit index (OCP MX v1.0, FP4 E2M1 element type).
E2M1_MAGNITUDE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E2M1_MAX = 6.0
BLOCK = 32
E8M0_BIAS = 127
E_MIN, E_MAX = -127, 127


def bf16_bits_to_f64(bits):
    """BF16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_to_bf16_bits(x):
    """Round float64 values to BF16 (round to nearest, ties to even).

    BF16 keeps 8 significant bits (7 stored) with float32's exponent range, so
    the rounding quantum of a normal value a is 2**(floor(log2 a) - 7) and of
    a subnormal one 2**-133.  Values that round to >= 2**128 become infinity.
    Returns uint16 bit patterns.
    """
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    _, ex = np.frexp(a)                      # a = m * 2**ex with m in [0.5, 1)
    qexp = np.maximum(ex - 8, -133)          # log2 of the rounding quantum
    r = np.rint(np.ldexp(a, -qexp))          # exact scaling, then RNE to integer
    v = np.ldexp(r, qexp)                    # the BF16 value (exact in float64)
    inf = v >= 2.0 ** 128
    v32 = np.where(inf, 0.0, v).astype(np.float32)   # exact: v is a BF16 value
    bits = (v32.view(np.uint32) >> 16).astype(np.uint32)
    bits = np.where(inf, 0x7F80, bits)
    bits = bits | (neg.astype(np.uint32) << 15)
    return bits.astype(np.uint16)


def e8m0_exponent(amax):
    """Shared exponent e of a block with absolute maximum ``amax`` (float64).

    e = floor(log2 amax) - 2, clamped to [-127, 127]; a zero block gets -127.
    floor(log2 a) is read from frexp (a = m * 2**ex, m in [0.5, 1) gives
    floor(log2 a) = ex - 1), never from a rounded log2.
    """
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(amax)
    e = np.where(amax > 0, ex - 1 - 2, E_MIN)
    return np.clip(e, E_MIN, E_MAX).astype(np.int64)


def e2m1_round_index(y):
    """Round non-negative float64 y to the index of the nearest E2M1 magnitude.

    An exact midpoint between neighbours i and i+1 goes to whichever of the
    two is even; y beyond the last midpoint (5.0) saturates to index 7 (6.0).
    """
    y = np.asarray(y, dtype=np.float64)
    idx = np.zeros(y.shape, dtype=np.int64)
    for i in range(7):
        mid = 0.5 * (E2M1_MAGNITUDE[i] + E2M1_MAGNITUDE[i + 1])
        up_on_tie = (i + 1) % 2 == 0
        idx += (y > mid) | ((y == mid) & up_on_tie)
    return idx


def quantize_blocks(x):
    """MXFP4-quantise float64 ``x`` [..., K] along its last axis (K % 32 == 0).

    Returns (codes uint8 [..., K] one 4-bit code per element,
             e8m0  uint8 [..., K/32]).
    """
    x = np.asarray(x, dtype=np.float64)
    K = x.shape[-1]
    assert K % BLOCK == 0, "the block axis must be a multiple of 32"
    blocks = x.reshape(x.shape[:-1] + (K // BLOCK, BLOCK))
    amax = np.abs(blocks).max(axis=-1)
    e = e8m0_exponent(amax)
    y = np.ldexp(np.abs(blocks), -e[..., None])
    idx = e2m1_round_index(y)
    sign = np.signbit(blocks).astype(np.int64)
    codes = (sign << 3) | idx
    return codes.reshape(x.shape).astype(np.uint8), (e + E8M0_BIAS).astype(np.uint8)


def decode(codes, e8m0):
    """Exact float64 values of unpacked E2M1 ``codes`` [..., K] with scales [..., K/32]."""
    codes = np.asarray(codes, dtype=np.int64)
    K = codes.shape[-1]
    mag = E2M1_MAGNITUDE[codes & 7]
    val = np.where((codes >> 3) & 1, -mag, mag)
    e = np.asarray(e8m0, dtype=np.int64) - E8M0_BIAS
    val = val.reshape(codes.shape[:-1] + (K // BLOCK, BLOCK))
    return np.ldexp(val, e[..., None]).reshape(codes.shape)


def pack_codes(codes):
    """Two 4-bit codes per byte: element 2j low nibble, element 2j+1 high nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_codes(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def mxfp4_quant(x_bits):
    """Standalone MXFP4 quantisation of a BF16 matrix [rows, cols] (cols % 32 == 0).

    "[gfx1250] Fuse A4W4 stage1 FP4 quantization", Summary (the standalone
    quant kept as the fallback) and the dense page's inline activation quant.
    Returns (packed codes uint8 [rows, cols/2], plain row-major E8M0 scales
    uint8 [rows, cols/32]).
    """
    codes, e8m0 = quantize_blocks(bf16_bits_to_f64(x_bits))
    return pack_codes(codes), e8m0


def quant_dequant(x):
    """Quantise float64 x [..., K] to MXFP4 and return the exact decoded values."""
    codes, e8m0 = quantize_blocks(x)
    return decode(codes, e8m0)
