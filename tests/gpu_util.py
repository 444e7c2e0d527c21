"""Helpers for the GPU parity tests (test code: no method arithmetic beyond
reading the library's documented byte layouts back)."""

import numpy as np
import torch

import workloads


def dev_bits(bits):
    """uint16 BF16 bit patterns (numpy) -> contiguous bfloat16 CUDA tensor."""
    return workloads.bits_to_torch(bits).cuda()


def host_bits(t):
    """bfloat16 CUDA tensor -> uint16 numpy bit patterns."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def unshuffle_tiles(codes, scales, rows, tiles, KT):
    """Read tiles of `rows` rows x 256 K in the swizzled operand layout of
    include/a4w4.h (codes: atom a = tile * KT + kt of rows * 128 bytes, byte b
    of row r at (r/8)*1024 + (r%8)*128 + ((b/16) ^ (r%8))*16 + b%16; scales:
    1024 bytes per atom, 32-block j of row r at (j/4)*512 + (r%32)*16 +
    (r/32)*4 + j%4) back into plain row-major packed codes [tiles*rows, KT*128]
    and E8M0 scales [tiles*rows, KT*8].

    Written from the header's formulas, independently of the CUDA code.
    """
    codes = np.asarray(codes, dtype=np.uint8)[:tiles * KT * rows * 128].reshape(tiles, KT, rows * 128)
    scales = np.asarray(scales, dtype=np.uint8)[:tiles * KT * 1024].reshape(tiles, KT, 1024)
    n = np.arange(tiles * rows)
    nt, r = n // rows, n % rows
    b = np.arange(128)
    out_c = np.empty((tiles * rows, KT * 128), dtype=np.uint8)
    off = (r[:, None] // 8) * 1024 + (r[:, None] % 8) * 128 + (((b[None, :] // 16) ^ (r[:, None] % 8)) * 16) + b[None, :] % 16
    for kt in range(KT):
        out_c[:, kt * 128:(kt + 1) * 128] = codes[nt[:, None], kt, off]
    out_s = np.empty((tiles * rows, KT * 8), dtype=np.uint8)
    j = np.arange(8)
    soff = (j[None, :] // 4) * 512 + (r[:, None] % 32) * 16 + (r[:, None] // 32) * 4 + j[None, :] % 4
    for kt in range(KT):
        out_s[:, kt * 8:(kt + 1) * 8] = scales[nt[:, None], kt, soff]
    return out_c, out_s


def shuffle_tiles(codes, scales, rows, tiles, KT):
    """Inverse of unshuffle_tiles: plain packed codes [tiles*rows, KT*128] and
    scales [tiles*rows, KT*8] -> (tile codes bytes, tile scale bytes) in the
    header's operand layout (scale-atom rows beyond `rows` stay zero)."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    out_c = np.zeros((tiles, KT, rows * 128), dtype=np.uint8)
    out_s = np.zeros((tiles, KT, 1024), dtype=np.uint8)
    n = np.arange(tiles * rows)
    nt, r = n // rows, n % rows
    b = np.arange(128)
    off = (r[:, None] // 8) * 1024 + (r[:, None] % 8) * 128 + (((b[None, :] // 16) ^ (r[:, None] % 8)) * 16) + b[None, :] % 16
    j = np.arange(8)
    soff = (j[None, :] // 4) * 512 + (r[:, None] % 32) * 16 + (r[:, None] // 32) * 4 + j[None, :] % 4
    for kt in range(KT):
        out_c[nt[:, None], kt, off] = codes[:, kt * 128:(kt + 1) * 128]
        out_s[nt[:, None], kt, soff] = scales[:, kt * 8:(kt + 1) * 8]
    return out_c.reshape(-1), out_s.reshape(-1)


def unshuffle_weight(wq, ws, N, K):
    """Preshuffled weights (include/a4w4.h) -> plain packed codes [N, KP/2] and
    E8M0 scales [N, KP/32] (KP = K rounded up to 256).  Atom (nt, kt) is
    number ((nt // 2) * KT + kt) * 2 + nt % 2; the atoms are put back in
    (nt, kt) order, then read with unshuffle_tiles."""
    KT = -(-K // 256)
    nt = np.arange(N // 128)[:, None]
    kt = np.arange(KT)[None, :]
    order = (((nt // 2) * KT + kt) * 2 + nt % 2).reshape(-1)       # atom number of (nt, kt), row-major
    wq = np.asarray(wq, dtype=np.uint8).reshape(-1, 16384)[order]
    ws = np.asarray(ws, dtype=np.uint8).reshape(-1, 1024)[order]
    return unshuffle_tiles(wq.reshape(-1), ws.reshape(-1), 128, N // 128, KT)


def gemm_violations(c_bits, ref, abs_sum):
    """Indices where a BF16 GEMM output breaks |C - ref| <= 2^-8|ref| + 2^-20 sum|a w|."""
    from oracle import gemm, mxfp4
    c = mxfp4.bf16_bits_to_f64(c_bits)
    err = np.abs(c - ref)
    return np.nonzero(~(err <= gemm.tolerance(ref, abs_sum)))
