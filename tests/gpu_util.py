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


def unshuffle_weight(wq, ws, N, K):
    """Read the preshuffled weight layout of include/a4w4.h back into plain
    row-major packed codes [N, K/2] and E8M0 scales [N, K/32].

    Written from the header's formulas, independently of the CUDA code.
    """
    KP = -(-K // 256) * 256
    KT = KP // 256
    wq = np.asarray(wq, dtype=np.uint8).reshape(N // 128, KT, 16384)
    ws = np.asarray(ws, dtype=np.uint8).reshape(N // 128, KT, 1024)
    n = np.arange(N)
    nt, r = n // 128, n % 128
    b = np.arange(128)
    codes = np.empty((N, KP // 2), dtype=np.uint8)
    for kt in range(KT):
        off = (r[:, None] // 8) * 1024 + (r[:, None] % 8) * 128 + (((b[None, :] // 16) ^ (r[:, None] % 8)) * 16) + b[None, :] % 16
        codes[:, kt * 128:(kt + 1) * 128] = wq[nt[:, None], kt, off]
    scales = np.empty((N, KP // 32), dtype=np.uint8)
    j = np.arange(8)
    for kt in range(KT):
        off = (j[None, :] // 4) * 512 + (r[:, None] % 32) * 16 + (r[:, None] // 32) * 4 + j[None, :] % 4
        scales[:, kt * 8:(kt + 1) * 8] = ws[nt[:, None], kt, off]
    return codes, scales


def gemm_violations(c_bits, ref, abs_sum):
    """Indices where a BF16 GEMM output breaks |C - ref| <= 2^-8|ref| + 2^-20 sum|a w|."""
    from oracle import gemm, mxfp4
    c = mxfp4.bf16_bits_to_f64(c_bits)
    err = np.abs(c - ref)
    return np.nonzero(~(err <= gemm.tolerance(ref, abs_sum)))
