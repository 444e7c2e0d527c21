"""The C ABI library loads and exports every symbol include/a4w4.h declares
(CPU only: no kernel is launched), and the calls that need no GPU behave."""

import os
import re

import pytest

import mxfp4_a4w4_gemm_gb300 as a4w4
from mxfp4_a4w4_gemm_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return a4w4.lib()


def declared_functions(header="a4w4.h"):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(a4w4_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported_and_bound(L):
    names = declared_functions()
    assert len(names) >= 18
    for n in names:
        assert hasattr(L, n), n
        assert n in a4w4.SIGNATURES, n
    # every binding is declared: nothing is bound that the header does not promise
    assert sorted(a4w4.SIGNATURES) == names


def test_debug_hooks_are_exported_and_bound(L):
    names = declared_functions("a4w4_debug.h")
    assert names == sorted(a4w4.DEBUG_SIGNATURES)
    for n in names:
        assert hasattr(L, n), n


def test_size_functions():
    assert a4w4.a4w4_weight_codes_bytes(256, 256) == 256 * 256 // 2
    assert a4w4.a4w4_weight_codes_bytes(1536, 4224) == 1536 * 4352 // 2          # K padded to 256
    assert a4w4.a4w4_weight_scales_bytes(1536, 4224) == 1536 * 4352 // 32
    assert a4w4.a4w4_moe_w1_codes_bytes(896, 1536, 3584) == 896 * 1536 * 3584 // 2
    assert a4w4.a4w4_moe_max_blocks(4096, 16, 896, 128) == 512 + 896
    assert a4w4.a4w4_moe_max_blocks(1, 16, 896, 128) == 1 + 16
    # large M: activations quantised once into 128-row x 256-K tiles (16 KB codes + 1 KB scales each)
    assert a4w4.a4w4_gemm_workspace_bytes(2048, 8448, 7168) == 16 * 28 * (16384 + 1024)
    assert a4w4.a4w4_gemm_workspace_bytes(200, 1536, 7168) == 2 * 28 * (16384 + 1024)   # no split-K partials
    # small M: split-K partials reduce inside a thread-block cluster, no workspace
    assert a4w4.a4w4_gemm_workspace_bytes(1, 1536, 7168) == 0


def test_kernel_routing_of_the_workload_shapes():
    # planned for GB300's 152 SMs when no device is visible (as on the GPU)
    name = a4w4.a4w4_gemm_kernel_name
    for K in (4224, 7168, 768):
        N = 1536 if K == 7168 else 7168
        for M in (1, 8):
            assert name(M, N, K) == "a4w4_decode_kernel<16,3>"
    assert name(32, 7168, 4224) == "a4w4_gemm_kernel<swap,32>"      # 5 splits: swap-AB's clusters suffice
    assert name(32, 1536, 7168) == "a4w4_decode_kernel<32,4>"       # 16 splits fill the grid
    assert name(32, 7168, 768) == "a4w4_decode_kernel<16,3>"        # one CTA holds the K range: two 16-token tiles
    assert name(20, 1536, 1024) == "a4w4_decode_kernel<16,4>"
    assert name(1, 256, 16384 * 4) == "a4w4_decode_kernel<16,4>"    # a 3-deep ring would need > 16 splits
    assert name(37, 1536, 4224) == "a4w4_gemm_kernel<swap,64>"
    assert name(100, 1536, 4224) == "a4w4_gemm_kernel<swap,128>"     # N < 4096: swap-AB up to 128 tokens
    for M in (128, 512, 2048):                                         # quantise once, persistent tile walk
        assert name(M, 8448, 7168) == "a4w4_large_kernel<prequant,persistent>"
    assert name(513, 1536, 4224) == "a4w4_large_kernel<prequant,persistent>"
    assert name(65, 8448, 7168) == "a4w4_large_kernel<prequant,persistent>"   # N >= 4096: from 65 rows
    assert name(128, 1536, 4224) == "a4w4_gemm_kernel<swap,128>"             # N < 4096: swap-AB to 128
    with pytest.raises(a4w4.A4W4Error) as e:
        name(1, 300, 256)
    assert e.value.code == a4w4.A4W4_ERR_ARG


def test_argument_errors_need_no_device():
    with pytest.raises(a4w4.A4W4Error) as e:
        a4w4.a4w4_gemm(16, 1, 256, 16, 16, 300, 16, stream=0)        # N % 256 != 0
    assert e.value.code == a4w4.A4W4_ERR_ARG
    with pytest.raises(a4w4.A4W4Error) as e:
        a4w4.a4w4_gemm(16, 1, 200, 16, 16, 256, 16, stream=0)        # K % 128 != 0
    assert e.value.code == a4w4.A4W4_ERR_ARG
    with pytest.raises(a4w4.A4W4Error) as e:
        a4w4.a4w4_gemm(8, 1, 256, 16, 16, 256, 16, stream=0)         # misaligned A
    assert e.value.code == a4w4.A4W4_ERR_ARG
    with pytest.raises(a4w4.A4W4Error) as e:
        a4w4.a4w4_mxfp4_quant(16, 4, 48, 16, 16, stream=0)           # cols % 32 != 0
    assert e.value.code == a4w4.A4W4_ERR_ARG
    with pytest.raises(a4w4.A4W4Error) as e:
        a4w4.a4w4_moe_sort(16, 4, 2, 8, 48, 16, 16, 16, 16, 1 << 20, stream=0)   # block_m
    assert e.value.code == a4w4.A4W4_ERR_ARG


def test_gemm_ex_rejects_unknown_flags():
    with pytest.raises(a4w4.A4W4Error) as e:
        a4w4.a4w4_gemm_ex(16, 1, 256, 16, 16, 256, 16, flags=2, stream=0)
    assert e.value.code == a4w4.A4W4_ERR_ARG


def test_debug_activation_layout_follows_the_plan():
    assert a4w4.a4w4_debug_gemm_activation_layout(1, 7168, 4224) == (16, 1, 17)
    assert a4w4.a4w4_debug_gemm_activation_layout(32, 7168, 4224) == (32, 1, 17)
    assert a4w4.a4w4_debug_gemm_activation_layout(37, 1536, 4224) == (64, 1, 17)
    assert a4w4.a4w4_debug_gemm_activation_layout(2047, 1536, 4224) == (128, 16, 17)


def test_strerror():
    assert a4w4.a4w4_strerror(0) == "ok"
    for c in (-1, -2, -3, -4, -5):
        assert a4w4.a4w4_strerror(c) != "unknown error"
