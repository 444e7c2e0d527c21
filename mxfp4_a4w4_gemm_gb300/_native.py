"""ctypes binding of liba4w4.so: the C ABI of include/a4w4.h, name for name.

Argument marshalling only.  Tensors (torch) are passed by ``data_ptr()`` and
must be contiguous; an ``int`` is taken as a raw pointer; ``stream=None``
means torch's current CUDA stream.  A non-zero return code raises
``A4W4Error``.  There is no fallback: if the library is not built the first
call raises.
"""

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_lib", "liba4w4.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "a4w4.h")

_c_int, _c_size, _vp, _i32p = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p

# name -> (restype, argtypes), in the order of include/a4w4.h
SIGNATURES = {
    "a4w4_weight_codes_bytes": (_c_size, [_c_int, _c_int]),
    "a4w4_weight_scales_bytes": (_c_size, [_c_int, _c_int]),
    "a4w4_prepare_gemm_weight": (_c_int, [_vp, _c_int, _c_int, _vp, _vp, _vp]),
    "a4w4_gemm_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "a4w4_gemm_kernel_name": (_c_int, [_c_int, _c_int, _c_int, ctypes.c_char_p, _c_size]),
    "a4w4_workspace_init": (_c_int, [_vp, _c_size, _vp]),
    "a4w4_gemm": (_c_int, [_vp, _c_int, _c_int, _vp, _vp, _c_int, _vp, _vp, _c_size, _vp]),
    "a4w4_gemm_ex": (_c_int, [_vp, _c_int, _c_int, _vp, _vp, _c_int, _vp, _vp, _c_size, ctypes.c_uint, _vp]),
    "a4w4_gemm_a16w4": (_c_int, [_vp, _c_int, _c_int, _vp, _vp, _c_int, _vp, ctypes.c_uint, _vp]),
    "a4w4_mxfp4_quant": (_c_int, [_vp, _c_int, _c_int, _vp, _vp, _vp]),
    "a4w4_moe_w1_codes_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "a4w4_moe_w1_scales_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "a4w4_moe_prepare_w1": (_c_int, [_vp, _c_int, _c_int, _c_int, _vp, _vp, _vp]),
    "a4w4_moe_max_blocks": (_c_int, [_c_int, _c_int, _c_int, _c_int]),
    "a4w4_moe_sort_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "a4w4_moe_sort": (_c_int, [_i32p, _c_int, _c_int, _c_int, _c_int, _i32p, _i32p, _i32p, _vp, _c_size, _vp]),
    "a4w4_moe_sort_aux_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "a4w4_moe_sort_aux": (_c_int, [_i32p, _c_int, _c_int, _c_int, _c_int, _i32p, _i32p, _i32p, _i32p, _i32p, _vp,
                                   _c_size, _vp]),
    "a4w4_moe_gemm1_workspace_bytes": (_c_size, [_c_int, _c_int]),
    "a4w4_moe_gemm1": (_c_int, [_vp, _c_int, _c_int, _i32p, _i32p, _i32p, _c_int, _vp, _vp, _c_int, _c_int,
                                _vp, _vp, _vp, _c_size, _vp]),
    "a4w4_moe_tiles_codes_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "a4w4_moe_tiles_scales_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "a4w4_moe_gemm1_ex": (_c_int, [_vp, _c_int, _c_int, _i32p, _i32p, _i32p, _c_int, _vp, _vp, _c_int, _c_int,
                                   _c_int, _c_int, _vp, _vp, _vp, _c_size, _vp]),
    "a4w4_moe_gemm2_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "a4w4_moe_gemm2": (_c_int, [_vp, _vp, _c_int, _c_int, _i32p, _i32p, _i32p, _c_int, _vp, _vp, _vp, _c_int,
                                _c_int, _vp, _vp, _c_size, _vp]),
    "a4w4_gemm_noalloc": (_c_int, [_vp, _c_int, _c_int, _vp, _vp, _c_int, _vp, _vp]),
    "a4w4_get_device_status": (_c_int, [_vp]),
    "a4w4_strerror": (ctypes.c_char_p, [_c_int]),
    "a4w4_set_wait_limit_ns": (None, [ctypes.c_ulonglong]),
}

# test hooks of include/a4w4_debug.h (not the product API)
_ip = ctypes.POINTER(ctypes.c_int)
DEBUG_SIGNATURES = {
    "a4w4_debug_gemm_activation_layout": (_c_int, [_c_int, _c_int, _c_int, _ip, _ip, _ip]),
    "a4w4_debug_gemm_export": (_c_int, [_vp, _c_int, _c_int, _vp, _vp, _c_int, _vp, _vp, _c_size, _vp, _c_size, _vp]),
    "a4w4_debug_moe_gemm1_export": (_c_int, [_vp, _c_int, _c_int, _i32p, _i32p, _i32p, _c_int, _vp, _vp, _c_int,
                                             _c_int, _vp, _vp, _vp, _c_size, _vp, _c_size, _vp]),
}

A4W4_GEMM_WEIGHT_PREFETCH = 1
A4W4_MOE_ACT_SWIGLU, A4W4_MOE_ACT_SILU = 0, 1
A4W4_MOE_OUT_ROWS, A4W4_MOE_OUT_TILES = 0, 1

_lib = None


class A4W4Error(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn} failed: {code} ({a4w4_strerror(code)})")


def lib():
    """The loaded liba4w4.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(python -m mxfp4_a4w4_gemm_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in list(SIGNATURES.items()) + list(DEBUG_SIGNATURES.items()):
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_contiguous():
            raise ValueError("tensor arguments must be contiguous")
        return x.data_ptr()
    raise TypeError(f"expected a tensor, an int pointer or None, got {type(x)}")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn, rc):
    if rc != 0:
        raise A4W4Error(fn, rc)


def a4w4_strerror(code):
    return lib().a4w4_strerror(int(code)).decode()


def a4w4_weight_codes_bytes(N, K):
    return lib().a4w4_weight_codes_bytes(N, K)


def a4w4_weight_scales_bytes(N, K):
    return lib().a4w4_weight_scales_bytes(N, K)


def a4w4_prepare_gemm_weight(W, N, K, Wq, Ws, stream=None):
    _check("a4w4_prepare_gemm_weight",
           lib().a4w4_prepare_gemm_weight(_ptr(W), N, K, _ptr(Wq), _ptr(Ws), _stream(stream)))


def a4w4_gemm_workspace_bytes(M, N, K):
    return lib().a4w4_gemm_workspace_bytes(M, N, K)


def a4w4_gemm_kernel_name(M, N, K):
    buf = ctypes.create_string_buffer(96)
    _check("a4w4_gemm_kernel_name", lib().a4w4_gemm_kernel_name(M, N, K, buf, len(buf)))
    return buf.value.decode()


def a4w4_workspace_init(workspace, ws_bytes, stream=None):
    _check("a4w4_workspace_init", lib().a4w4_workspace_init(_ptr(workspace), ws_bytes, _stream(stream)))


def a4w4_gemm(A, M, K, Wq, Ws, N, C, workspace=None, ws_bytes=0, stream=None):
    _check("a4w4_gemm", lib().a4w4_gemm(_ptr(A), M, K, _ptr(Wq), _ptr(Ws), N, _ptr(C), _ptr(workspace),
                                         ws_bytes, _stream(stream)))


def a4w4_gemm_ex(A, M, K, Wq, Ws, N, C, workspace=None, ws_bytes=0, flags=0, stream=None):
    _check("a4w4_gemm_ex", lib().a4w4_gemm_ex(_ptr(A), M, K, _ptr(Wq), _ptr(Ws), N, _ptr(C), _ptr(workspace),
                                               ws_bytes, flags, _stream(stream)))


def a4w4_gemm_a16w4(A, M, K, Wq, Ws, N, C, flags=0, stream=None):
    _check("a4w4_gemm_a16w4", lib().a4w4_gemm_a16w4(_ptr(A), M, K, _ptr(Wq), _ptr(Ws), N, _ptr(C), flags,
                                                    _stream(stream)))


def a4w4_mxfp4_quant(X, rows, cols, q, scales, stream=None):
    _check("a4w4_mxfp4_quant", lib().a4w4_mxfp4_quant(_ptr(X), rows, cols, _ptr(q), _ptr(scales), _stream(stream)))


def a4w4_moe_w1_codes_bytes(E, two_I, D):
    return lib().a4w4_moe_w1_codes_bytes(E, two_I, D)


def a4w4_moe_w1_scales_bytes(E, two_I, D):
    return lib().a4w4_moe_w1_scales_bytes(E, two_I, D)


def a4w4_moe_prepare_w1(W1, E, two_I, D, W1q, W1s, stream=None):
    _check("a4w4_moe_prepare_w1",
           lib().a4w4_moe_prepare_w1(_ptr(W1), E, two_I, D, _ptr(W1q), _ptr(W1s), _stream(stream)))


def a4w4_moe_max_blocks(T, topk, E, block_m):
    return lib().a4w4_moe_max_blocks(T, topk, E, block_m)


def a4w4_moe_sort_workspace_bytes(T, topk, E):
    return lib().a4w4_moe_sort_workspace_bytes(T, topk, E)


def a4w4_moe_sort(topk_ids, T, topk, E, block_m, sorted_rows, block_expert, num_blocks, ws, ws_bytes, stream=None):
    _check("a4w4_moe_sort", lib().a4w4_moe_sort(_ptr(topk_ids), T, topk, E, block_m, _ptr(sorted_rows),
                                                _ptr(block_expert), _ptr(num_blocks), _ptr(ws), ws_bytes,
                                                _stream(stream)))


def a4w4_moe_sort_aux_workspace_bytes(T, topk, E):
    return lib().a4w4_moe_sort_aux_workspace_bytes(T, topk, E)


def a4w4_moe_sort_aux(topk_ids, T, topk, E, block_m, sorted_rows, block_expert, num_blocks, sorted_tokens, row_slot,
                      ws, ws_bytes, stream=None):
    _check("a4w4_moe_sort_aux", lib().a4w4_moe_sort_aux(_ptr(topk_ids), T, topk, E, block_m, _ptr(sorted_rows),
                                                        _ptr(block_expert), _ptr(num_blocks), _ptr(sorted_tokens),
                                                        _ptr(row_slot), _ptr(ws), ws_bytes, _stream(stream)))


def a4w4_moe_gemm1_workspace_bytes(T, D):
    return lib().a4w4_moe_gemm1_workspace_bytes(T, D)


def a4w4_moe_gemm1(X, T, D, sorted_rows, block_expert, num_blocks, topk, W1q, W1s, E, I, out_q, out_s,
                   ws=None, ws_bytes=0, stream=None):
    _check("a4w4_moe_gemm1", lib().a4w4_moe_gemm1(_ptr(X), T, D, _ptr(sorted_rows), _ptr(block_expert),
                                                  _ptr(num_blocks), topk, _ptr(W1q), _ptr(W1s), E, I,
                                                  _ptr(out_q), _ptr(out_s), _ptr(ws), ws_bytes, _stream(stream)))


def a4w4_moe_tiles_codes_bytes(T, topk, E, I):
    return lib().a4w4_moe_tiles_codes_bytes(T, topk, E, I)


def a4w4_moe_tiles_scales_bytes(T, topk, E, I):
    return lib().a4w4_moe_tiles_scales_bytes(T, topk, E, I)


def a4w4_moe_gemm1_ex(X, T, D, sorted_rows, block_expert, num_blocks, topk, W1q, W1s, E, I, activation, out_layout,
                      out_q, out_s, ws=None, ws_bytes=0, stream=None):
    _check("a4w4_moe_gemm1_ex", lib().a4w4_moe_gemm1_ex(_ptr(X), T, D, _ptr(sorted_rows), _ptr(block_expert),
                                                        _ptr(num_blocks), topk, _ptr(W1q), _ptr(W1s), E, I,
                                                        activation, out_layout, _ptr(out_q), _ptr(out_s), _ptr(ws),
                                                        ws_bytes, _stream(stream)))


def a4w4_moe_gemm2_workspace_bytes(T, topk, D):
    return lib().a4w4_moe_gemm2_workspace_bytes(T, topk, D)


def a4w4_moe_gemm2(A_q, A_s, T, I, sorted_rows, block_expert, num_blocks, topk, topk_weights, W2q, W2s, E, D, Y,
                   ws, ws_bytes, stream=None):
    _check("a4w4_moe_gemm2", lib().a4w4_moe_gemm2(_ptr(A_q), _ptr(A_s), T, I, _ptr(sorted_rows), _ptr(block_expert),
                                                  _ptr(num_blocks), topk, _ptr(topk_weights), _ptr(W2q), _ptr(W2s),
                                                  E, D, _ptr(Y), _ptr(ws), ws_bytes, _stream(stream)))


def a4w4_gemm_noalloc(A, M, K, Wq, Ws, N, C, stream=None):
    """a4w4_gemm without a workspace, for callers that cannot allocate device
    memory at the call site: the plan's scratch (activation tiles quantised
    once, split-K partials and counters; only for M > 64) comes from a fixed
    16 MiB array in the library (shapes that need more raise A4W4Error,
    A4W4_ERR_WORKSPACE).  Make the first call on a device before any CUDA
    graph capture; calls that may overlap on one GPU share the array and must
    be serialised."""
    _check("a4w4_gemm_noalloc", lib().a4w4_gemm_noalloc(_ptr(A), M, K, _ptr(Wq), _ptr(Ws), N, _ptr(C),
                                                         _stream(stream)))


def a4w4_get_device_status(stream=None):
    """Synchronises the stream; returns (and clears) the device status code."""
    return lib().a4w4_get_device_status(_stream(stream))


def a4w4_set_wait_limit_ns(ns):
    lib().a4w4_set_wait_limit_ns(int(ns))


# ---------------------------------------------------------------------------
# test hooks (include/a4w4_debug.h)

def a4w4_debug_gemm_activation_layout(M, N, K):
    """(tile_rows, x_tiles, k_tiles) of a4w4_gemm(M, N, K)'s activation tiles."""
    r, x, k = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check("a4w4_debug_gemm_activation_layout",
           lib().a4w4_debug_gemm_activation_layout(M, N, K, ctypes.byref(r), ctypes.byref(x), ctypes.byref(k)))
    return r.value, x.value, k.value


def a4w4_debug_gemm_export(A, M, K, Wq, Ws, N, C, workspace, ws_bytes, dump, dump_bytes, stream=None):
    _check("a4w4_debug_gemm_export",
           lib().a4w4_debug_gemm_export(_ptr(A), M, K, _ptr(Wq), _ptr(Ws), N, _ptr(C), _ptr(workspace), ws_bytes,
                                        _ptr(dump), dump_bytes, _stream(stream)))


def a4w4_debug_moe_gemm1_export(X, T, D, sorted_rows, block_expert, num_blocks, topk, W1q, W1s, E, I, out_q, out_s,
                                ws, ws_bytes, dump, dump_bytes, stream=None):
    _check("a4w4_debug_moe_gemm1_export",
           lib().a4w4_debug_moe_gemm1_export(_ptr(X), T, D, _ptr(sorted_rows), _ptr(block_expert), _ptr(num_blocks),
                                             topk, _ptr(W1q), _ptr(W1s), E, I, _ptr(out_q), _ptr(out_s), _ptr(ws),
                                             ws_bytes, _ptr(dump), dump_bytes, _stream(stream)))
