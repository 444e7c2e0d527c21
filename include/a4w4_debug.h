/*
 * a4w4_debug.h -- test hooks of liba4w4.so.  Not part of the product API
 * (a4w4.h); they exist so that tests can read back intermediate results that
 * the product calls keep on chip.
 *
 * Activation export.  "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM",
 * Summary: the BF16 activations are quantised to MXFP4 inline, inside the
 * GEMM, so the codes and scales never reach global memory.  These calls run
 * exactly the plan and kernels of the product call and, in addition, store
 * the MXFP4 activation operand tiles that the kernels build (in shared memory,
 * or in the workspace for the quantise-once plans) into `dump`, so that they
 * can be compared bit for bit with a reference quantiser.
 *
 * Dump layout: tiles of `tile_rows` activation rows x 256 K (KT = K rounded up
 * to 256, / 256; atom a = x_tile * KT + kt):
 *   codes  at dump + a * tile_rows * 128, in the swizzled layout of a4w4.h's
 *          Wq tiles restricted to rows 0..tile_rows-1: byte b of row r at
 *          (r/8)*1024 + (r%8)*128 + ((b/16) ^ (r%8))*16 + b%16;
 *   scales at dump + atoms * tile_rows * 128 + a * 1024, in the layout of
 *          a4w4.h's Ws tiles: (j/4)*512 + (r%32)*16 + (r/32)*4 + j%4.
 * Row r of tile x is activation row x * tile_rows + r (dense GEMM), or the
 * routed row listed in sorted slot x * 128 + r (MoE GEMM1).  Rows that do not
 * exist (beyond M, padding slots) are zero.  The dump is cleared on `stream`
 * first; its size must be at least atoms * (tile_rows * 128 + 1024) bytes.
 */
#ifndef A4W4_DEBUG_H_
#define A4W4_DEBUG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Activation tile geometry of a4w4_gemm(M, N, K)'s plan on the current device
 * (GB300's 152 SMs when none is visible): rows per tile, activation tiles, K
 * tiles.  Host-only.  A4W4_ERR_ARG for a shape a4w4_gemm rejects. */
int a4w4_debug_gemm_activation_layout(int M, int N, int K, int* tile_rows, int* x_tiles, int* k_tiles);

/* a4w4_gemm(...) plus the activation export described above. */
int a4w4_debug_gemm_export(const void* A_bf16, int M, int K, const void* Wq, const void* Ws, int N,
                           void* C_bf16, void* workspace, size_t ws_bytes, void* dump, size_t dump_bytes,
                           void* stream);

/* a4w4_moe_gemm1(...) plus the activation export (tile_rows = 128, one tile
 * per sorted block, x_tiles = a4w4_moe_max_blocks(T, topk, E, 128)); blocks
 * beyond the routing's block count stay zero. */
int a4w4_debug_moe_gemm1_export(const void* X_bf16, int T, int D, const int32_t* sorted_rows,
                                const int32_t* block_expert, const int32_t* num_blocks, int topk,
                                const void* W1q, const void* W1s, int E, int I, void* out_q, void* out_s,
                                void* ws, size_t ws_bytes, void* dump, size_t dump_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* A4W4_DEBUG_H_ */
