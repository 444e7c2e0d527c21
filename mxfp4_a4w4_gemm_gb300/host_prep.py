"""Preparing MoE GEMM1 weights that live in host memory, a chunk of experts at
a time, so that the BF16 copy never has to fit on the GPU at once (E=896
experts of [1536, 3584] BF16 are 9.9 GB; their MXFP4 form is 2.6 GB).  Also
the dense per-expert layout (one preshuffled matrix of the stacked experts)
used by the SiLU GEMM1 weights and the GEMM2 down projection."""

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from ._native import (a4w4_moe_prepare_w1, a4w4_moe_w1_codes_bytes, a4w4_moe_w1_scales_bytes,
                      a4w4_prepare_gemm_weight, a4w4_weight_codes_bytes, a4w4_weight_scales_bytes)


def prepare_moe_w1_from_host(expert_bits, E, two_I, D, chunk=32, threads=8, device="cuda"):
    """expert_bits(e) -> numpy uint16 BF16 bit patterns [two_I, D] of expert e.

    Returns (W1q, W1s) uint8 CUDA tensors in the preshuffled MoE layout."""
    W1q = torch.empty(a4w4_moe_w1_codes_bytes(E, two_I, D), dtype=torch.uint8, device=device)
    W1s = torch.empty(a4w4_moe_w1_scales_bytes(E, two_I, D), dtype=torch.uint8, device=device)
    cb = a4w4_weight_codes_bytes(two_I, D)
    sb = a4w4_weight_scales_bytes(two_I, D)
    with ThreadPoolExecutor(threads) as ex:
        for e0 in range(0, E, chunk):
            es = list(range(e0, min(E, e0 + chunk)))
            host = np.stack(list(ex.map(expert_bits, es)))
            dev = torch.from_numpy(host.view(np.int16)).to(device)
            a4w4_moe_prepare_w1(dev, len(es), two_I, D, W1q.data_ptr() + e0 * cb, W1s.data_ptr() + e0 * sb)
            torch.cuda.current_stream().synchronize()
            del dev
    return W1q, W1s


def prepare_dense_experts_from_host(expert_bits, E, rows, K, chunk=32, threads=8, device="cuda"):
    """expert_bits(e) -> numpy uint16 BF16 bit patterns [rows, K] of expert e.

    Returns (Wq, Ws) uint8 CUDA tensors: the dense preshuffled layout of the
    stacked [E*rows, K] matrix (expert e at e * a4w4_weight_codes_bytes(rows, K)
    and e * a4w4_weight_scales_bytes(rows, K)).  rows % 256 == 0."""
    assert rows % 256 == 0
    cb = a4w4_weight_codes_bytes(rows, K)
    sb = a4w4_weight_scales_bytes(rows, K)
    Wq = torch.empty(E * cb, dtype=torch.uint8, device=device)
    Ws = torch.empty(E * sb, dtype=torch.uint8, device=device)
    with ThreadPoolExecutor(threads) as ex:
        for e0 in range(0, E, chunk):
            es = list(range(e0, min(E, e0 + chunk)))
            host = np.concatenate(list(ex.map(expert_bits, es)))
            dev = torch.from_numpy(host.view(np.int16)).to(device)
            a4w4_prepare_gemm_weight(dev, len(es) * rows, K, Wq.data_ptr() + e0 * cb, Ws.data_ptr() + e0 * sb)
            torch.cuda.current_stream().synchronize()
            del dev
    return Wq, Ws
