"""GPU parity: the standalone MXFP4 quant and the weight preshuffle, bit-exact
against the oracle (through the C ABI)."""

import json
import os

import numpy as np
import pytest
import torch

import mxfp4_a4w4_gemm_gb300 as a4w4
import workloads
from gpu_util import dev_bits, unshuffle_weight
from oracle import mxfp4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mxfp4_a4w4_gemm_gb300 import build
    build.build()
    a4w4.lib()


def gpu_quant(bits):
    rows, cols = bits.shape
    q = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    s = torch.empty((rows, cols // 32), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_mxfp4_quant(dev_bits(bits), rows, cols, q, s)
    assert a4w4.a4w4_get_device_status() == 0
    return q.cpu().numpy(), s.cpu().numpy()


def assert_quant_equal(bits):
    q, s = gpu_quant(bits)
    rq, rs = mxfp4.mxfp4_quant(bits)
    bad_s = np.argwhere(s != rs)
    bad_q = np.argwhere(q != rq)
    assert bad_s.size == 0, f"{len(bad_s)} scale mismatches, first {bad_s[:5].tolist()}"
    assert bad_q.size == 0, f"{len(bad_q)} code-byte mismatches, first {bad_q[:5].tolist()}"


def test_quant_worked_example():
    d = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "mxfp4_worked_example.json")))
    row = np.zeros(32 * len(d["blocks"]))
    for b, blk in enumerate(d["blocks"]):
        for i, h in enumerate(blk["x"]):
            row[32 * b + i] = float.fromhex(h)
    bits = mxfp4.round_to_bf16_bits(row)[None, :]
    q, s = gpu_quant(bits)
    assert q[0].tobytes().hex() == d["packed_hex"]
    assert list(s[0]) == d["scales"]


def test_quant_every_bf16_value():
    """All 65536 BF16 bit patterns that are finite, in 2048 blocks of 32, under
    several block maxima (the first element of each block sets the scale)."""
    allbits = np.arange(0x10000, dtype=np.uint32)
    finite = allbits[(allbits & 0x7F80) != 0x7F80].astype(np.uint16)
    pad = (-finite.size) % 32
    x = np.concatenate([finite, np.zeros(pad, np.uint16)]).reshape(-1, 32)
    assert_quant_equal(x)
    for lead in (0x3F80, 0x4100, 0x0080, 0x7F7F, 0x8001):     # 1, 8, min normal, max, -min subnormal
        y = x.copy()
        y[:, 0] = lead
        assert_quant_equal(y)


@pytest.mark.parametrize("family,shape", [
    ("decode", (32, 4224)), ("decode", (8, 7168)), ("decode", (1, 768)),
    ("large", (2048, 7168)), ("stress", (2047, 4224)), ("stress", (37, 4224)),
])
def test_quant_workloads(family, shape):
    M, K = shape
    if family == "decode":
        bits = workloads.decode_activation_bits(M, K)
    elif family == "stress":
        bits = workloads.stress_activation_bits(M, K)
    else:
        bits = workloads.activation_bits(M, K)
    assert_quant_equal(bits)


@pytest.mark.parametrize("N,K", [(256, 256), (1536, 4224), (512, 768), (256, 7168)])
def test_prepare_weight_bit_exact(N, K):
    W = workloads.weight_bits(N, K)
    Wq = torch.empty(a4w4.a4w4_weight_codes_bytes(N, K), dtype=torch.uint8, device="cuda")
    Ws = torch.empty(a4w4.a4w4_weight_scales_bytes(N, K), dtype=torch.uint8, device="cuda")
    Wq.fill_(0xAB)
    Ws.fill_(0xCD)
    a4w4.a4w4_prepare_gemm_weight(dev_bits(W), N, K, Wq, Ws)
    assert a4w4.a4w4_get_device_status() == 0
    codes, scales = unshuffle_weight(Wq.cpu().numpy(), Ws.cpu().numpy(), N, K)
    rq, rs = mxfp4.mxfp4_quant(W)
    assert np.array_equal(codes[:, :K // 2], rq)
    assert np.array_equal(scales[:, :K // 32], rs)
    assert np.all(codes[:, K // 2:] == 0) and np.all(scales[:, K // 32:] == 0)   # K padding


def test_moe_prepare_pairs_gate_and_up_rows():
    E, I, D = 3, 256, 512
    W1 = np.stack([workloads.moe_expert_weight_bits(e, 2 * I, D) for e in range(E)])
    W1q = torch.empty(a4w4.a4w4_moe_w1_codes_bytes(E, 2 * I, D), dtype=torch.uint8, device="cuda")
    W1s = torch.empty(a4w4.a4w4_moe_w1_scales_bytes(E, 2 * I, D), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_moe_prepare_w1(dev_bits(W1), E, 2 * I, D, W1q, W1s)
    assert a4w4.a4w4_get_device_status() == 0
    cb = a4w4.a4w4_weight_codes_bytes(2 * I, D)
    sb = a4w4.a4w4_weight_scales_bytes(2 * I, D)
    q = W1q.cpu().numpy()
    s = W1s.cpu().numpy()
    for e in range(E):
        codes, scales = unshuffle_weight(q[e * cb:(e + 1) * cb], s[e * sb:(e + 1) * sb], 2 * I, D)
        order = np.concatenate([np.concatenate([np.arange(128 * j, 128 * j + 128), I + np.arange(128 * j, 128 * j + 128)])
                                for j in range(I // 128)])
        rq, rs = mxfp4.mxfp4_quant(W1[e][order])
        assert np.array_equal(codes, rq) and np.array_equal(scales, rs)
