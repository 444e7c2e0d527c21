/*
 * a4w4.h -- C ABI of the GB300 (sm_103a) MXFP4 A4W4 GEMM library (liba4w4.so).
 *
 * What it computes
 *   "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM", Summary and
 *   Implementation: BF16 activations are quantised inline to MXFP4 (E2M1 codes,
 *   one E8M0 power-of-two scale per 32 consecutive K elements) and multiplied
 *   against MXFP4 weights that the caller quantised and preshuffled once, with
 *   fp32 accumulation and BF16 output.  "[gfx1250] Fuse A4W4 stage1 FP4
 *   quantization", Summary: the grouped-MoE GEMM1 variant applies SwiGLU and
 *   emits MXFP4 codes and E8M0 scales directly.
 *
 *   Quantisation rule (OCP MX v1.0; the pages do not state one): per 32-block,
 *   e = floor(log2(max|x|)) - 2 clamped to [-127, 127] (-127 for an all-zero
 *   block), E8M0 code = e + 127, element code = sign << 3 | E2M1 index of
 *   |x| / 2^e rounded to nearest, ties to even, saturating at 6.
 *
 * Conventions for every call
 *   - Pointers named *_bf16 / Wq / Ws / q / scales / out_* are DEVICE pointers
 *     to caller-owned memory, 16-byte aligned, contiguous, row-major.  The
 *     library allocates no device memory and keeps no pointer after a call.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     only enqueued; no call synchronises except a4w4_get_device_status().
 *   - Packed E2M1: element 2j in the low nibble of byte j, 2j+1 in the high one.
 *   - Return codes: A4W4_OK or a negative A4W4_ERR_* (a4w4_strerror names it).
 *     Argument errors are detected before anything is enqueued.
 *   - Every kernel bounds its waits; a wait that runs out records
 *     A4W4_ERR_TIMEOUT in a device status word and the kernel returns early.
 *
 * Thread safety: calls may be issued from several host threads; calls that run
 * concurrently on the GPU must not share output buffers or a workspace.
 */
#ifndef A4W4_H_
#define A4W4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  A4W4_OK = 0,
  A4W4_ERR_ARG = -1,        /* null/misaligned pointer, or a shape outside the contract */
  A4W4_ERR_DEVICE = -2,     /* current device is not compute capability 10.3 (GB300) */
  A4W4_ERR_WORKSPACE = -3,  /* workspace smaller than a4w4_*_workspace_bytes() */
  A4W4_ERR_LAUNCH = -4,     /* a CUDA launch or API call failed */
  A4W4_ERR_TIMEOUT = -5     /* a bounded in-kernel wait expired (read by get_device_status) */
};

/* ------------------------------------------------------------------------ */
/* Weights: quantise + preshuffle once.
 * "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM", Implementation ("one-time
 * packed E2M1 weight and E8M0 scale preshuffle") and Scope ("N divisible by 256;
 * K divisible by 128"; "preshuffled once by the caller").
 *
 * Preshuffled layout (GB300 tensor-core operand tiles; KP = K rounded up to a
 * multiple of 256, KT = KP / 256, row tiles of 128 rows, nt = n / 128,
 * kt = k / 256, r = n % 128, atom = ((nt / 2) * KT + kt) * 2 + nt % 2: the two
 * 128-row atoms of a 256-row tile and one K tile are adjacent, so a GEMM tile
 * fetches them with one bulk copy):
 *   Wq: atom-major tiles of 16384 bytes.  Byte b (0..127) of row r of a tile
 *       holds the codes of k = kt*256 + 2b (low nibble) and 2b+1 (high nibble)
 *       at offset  atom*16384 + (r/8)*1024 + (r%8)*128 + ((b/16) ^ (r%8))*16 + b%16
 *       (the 128-byte swizzle of the tensor core's K-major shared-memory tiles).
 *   Ws: tiles of 1024 bytes.  The E8M0 scale of 32-block j (0..7) of tile
 *       (nt, kt) for row r is at  atom*1024 + (j/4)*512 + (r%32)*16 + (r/32)*4 + j%4.
 *   Codes and scales for k >= K are zero.
 */
size_t a4w4_weight_codes_bytes(int N, int K);   /* N * KP / 2  */
size_t a4w4_weight_scales_bytes(int N, int K);  /* N * KP / 32 */

/* W_bf16 [N, K] -> Wq, Ws (sizes above).  N % 256 == 0, K % 128 == 0, N,K > 0. */
int a4w4_prepare_gemm_weight(const void* W_bf16, int N, int K, void* Wq, void* Ws,
                             void* stream);

/* ------------------------------------------------------------------------ */
/* Dense A4W4 GEMM:  C[M, N] (BF16) = MXFP4(A)[M, K] x MXFP4(W)[N, K]^T.
 * "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM", Summary, Implementation
 * (inline activation quant, BF16 direct output, M-tail masking), Scope.
 *   A_bf16 [M, K] row-major; Wq, Ws from a4w4_prepare_gemm_weight(N, K);
 *   C_bf16 [M, N] row-major, rows >= M are never touched.
 *   M >= 1, N % 256 == 0, K % 128 == 0.
 * Small M uses weights-as-rows tiles (swap-AB) with split-K over the SMs,
 * reduced inside thread-block clusters (no workspace).  Larger M (M > 128;
 * M > 64 when N >= 4096) quantises the activations once into tiles, held in
 * `workspace`, and runs whole 128 x 256 output tiles (no split-K).  The
 * workspace must hold at least a4w4_gemm_workspace_bytes(M, N, K) bytes
 * (a4w4_workspace_init may zero it; its contents are overwritten before they
 * are read).  When that size is 0 the workspace may be NULL.  Every reduction
 * order is fixed, so results are bitwise deterministic. */
size_t a4w4_gemm_workspace_bytes(int M, int N, int K);
int a4w4_workspace_init(void* workspace, size_t ws_bytes, void* stream);
/* Name of the kernel instantiation a4w4_gemm(M, N, K) launches on the current
 * device (planned for GB300's 152 SMs when no device is visible), e.g.
 * "a4w4_decode_kernel<16,3>" (tokens per CTA, weight ring depth) or
 * "a4w4_gemm_kernel<swap,32>" / "a4w4_large_kernel<prequant,persistent>";
 * the quantise-once plans also launch the activation pre-pass.  Host-only, no
 * device work.  Writes a NUL-terminated string of at most n bytes (truncated)
 * into buf.  Returns A4W4_OK, or A4W4_ERR_ARG for a shape a4w4_gemm rejects,
 * a NULL buf or n == 0. */
int a4w4_gemm_kernel_name(int M, int N, int K, char* buf, size_t n);
int a4w4_gemm(const void* A_bf16, int M, int K, const void* Wq, const void* Ws, int N,
              void* C_bf16, void* workspace, size_t ws_bytes, void* stream);

/* a4w4_gemm with per-call options; a4w4_gemm(...) is a4w4_gemm_ex(..., 0, stream).
 * Flags (unknown bits give A4W4_ERR_ARG):
 *   A4W4_GEMM_WEIGHT_PREFETCH -- the GEMM is launched with programmatic
 *     dependent launch like every GEMM here (it may start while the previous
 *     kernel on `stream` still runs, and waits for that kernel before it
 *     touches A, C or the workspace); with this flag it also starts streaming
 *     Wq/Ws before that wait, hiding the weight fetch behind the previous
 *     kernel.  Set it only when the kernel issued just before this call on
 *     the same stream does not write Wq or Ws (weights prepared earlier and
 *     left unchanged, as in inference).  The promise covers this call alone. */
enum { A4W4_GEMM_WEIGHT_PREFETCH = 1 };
int a4w4_gemm_ex(const void* A_bf16, int M, int K, const void* Wq, const void* Ws, int N,
                 void* C_bf16, void* workspace, size_t ws_bytes, unsigned int flags, void* stream);

/* ------------------------------------------------------------------------ */
/* A16WFP4 GEMM:  C[M, N] (BF16) = A[M, K] (BF16, not quantised) x MXFP4(W)^T.
 * "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM", Summary (the #4772
 * bullet: BF16 activation x decoded MXFP4 weight).  Same arguments, layouts
 * and shape contract as a4w4_gemm_ex with the same preshuffled Wq/Ws; no
 * workspace.  Each weight tile is decoded to BF16 on chip (exact for E8M0
 * scales from 2^-127 to 2^125, i.e. weight blocks whose largest magnitude is
 * below 2^127) and multiplied in BF16 with fp32 accumulation; split-K is
 * reduced inside thread-block clusters in a fixed order (deterministic).
 * flags: A4W4_GEMM_WEIGHT_PREFETCH as for a4w4_gemm_ex. */
int a4w4_gemm_a16w4(const void* A_bf16, int M, int K, const void* Wq, const void* Ws, int N,
                    void* C_bf16, unsigned int flags, void* stream);

/* ------------------------------------------------------------------------ */
/* Standalone MXFP4 quantisation (plain layout).
 * "[gfx1250] Fuse A4W4 stage1 FP4 quantization", Summary (the standalone quant
 * kept as the fallback path).
 *   X_bf16 [rows, cols] -> q [rows, cols/2] packed codes, scales [rows, cols/32]
 *   E8M0 bytes, both row-major.  rows >= 1, cols % 32 == 0. */
int a4w4_mxfp4_quant(const void* X_bf16, int rows, int cols, void* q, void* scales,
                     void* stream);

/* ------------------------------------------------------------------------ */
/* Grouped MoE GEMM1 (gate+up projection, SwiGLU, MXFP4 requant).
 * "[gfx1250] Fuse A4W4 stage1 FP4 quantization", Summary and Performance;
 * "[HIP] [CK] [FlyDSL] [Kernel] Extend MXFP4 GEMM1 replacement to A4W4", Summary
 * (auxiliary sort of routed rows into per-expert blocks).
 *
 * Expert weights W1_bf16 [E, 2I, D]: rows 0..I-1 are the gate projection,
 * rows I..2I-1 the up projection.  a4w4_moe_prepare_w1 writes, per expert, the
 * dense preshuffled layout above of the row-reordered matrix whose 256-row
 * tile j holds gate rows 128j..128j+127 followed by up rows 128j..128j+127
 * (so one accumulator tile holds matching gate/up columns).  Expert e starts
 * at e * a4w4_weight_codes_bytes(2I, D) in W1q and e * a4w4_weight_scales_bytes(2I, D)
 * in W1s.  I % 128 == 0, D % 128 == 0. */
size_t a4w4_moe_w1_codes_bytes(int E, int two_I, int D);
size_t a4w4_moe_w1_scales_bytes(int E, int two_I, int D);
int a4w4_moe_prepare_w1(const void* W1_bf16, int E, int two_I, int D, void* W1q, void* W1s,
                        void* stream);

/* Sort of routed rows.  Routed row r = t * topk + k sends token t to expert
 * topk_ids[t, k] (int32 [T, topk], values in [0, E)).  Output: for experts
 * e = 0..E-1 in order, the rows routed to e in increasing r, padded with the
 * sentinel T*topk to a multiple of block_m (16, 32, 64 or 128);
 * sorted_rows[b*block_m + i] lists block b, block_expert[b] is its expert,
 * *num_blocks the block count (all on the device, no host synchronisation).
 * Buffers: sorted_rows >= a4w4_moe_max_blocks(T, topk, E, block_m) * block_m
 * entries, block_expert >= a4w4_moe_max_blocks(...) entries, num_blocks 1 entry,
 * ws >= a4w4_moe_sort_workspace_bytes(T, topk, E). */
int a4w4_moe_max_blocks(int T, int topk, int E, int block_m);
size_t a4w4_moe_sort_workspace_bytes(int T, int topk, int E);
int a4w4_moe_sort(const int32_t* topk_ids, int T, int topk, int E, int block_m,
                  int32_t* sorted_rows, int32_t* block_expert, int32_t* num_blocks,
                  void* ws, size_t ws_bytes, void* stream);

/* The same sort, with the auxiliary gather/scatter arrays, in one launch for
 * up to 2048 routed rows and two beyond.
 * "[HIP] [CK] [FlyDSL] [Kernel] Extend MXFP4 GEMM1 replacement to A4W4",
 * Summary (the adaptive MoE auxiliary sort; its review names the aux arrays
 * the sort emits for A4W4).  sorted_rows, block_expert and num_blocks are
 * identical to a4w4_moe_sort's; in addition sorted_tokens[s] is the token
 * (r / topk) of sorted slot s, or T for a padding slot (same length as
 * sorted_rows), and row_slot[r] is the slot that holds routed row r (int32
 * [T*topk]).  Up to 2048 routed rows (a decode batch) one CTA does the whole
 * sort; beyond, up to one CTA per SM each counts a run of rows, the last to
 * finish scans the counts, and a second launch places the rows.  E <= 4096,
 * T*topk <= 32768 x the SM count.  ws >= a4w4_moe_sort_aux_workspace_bytes(T,
 * topk, E) bytes, 16-byte aligned, zeroed once with a4w4_workspace_init (it
 * ends with a ticket counter that the last counting CTA resets). */
size_t a4w4_moe_sort_aux_workspace_bytes(int T, int topk, int E);
int a4w4_moe_sort_aux(const int32_t* topk_ids, int T, int topk, int E, int block_m,
                      int32_t* sorted_rows, int32_t* block_expert, int32_t* num_blocks,
                      int32_t* sorted_tokens, int32_t* row_slot, void* ws, size_t ws_bytes,
                      void* stream);

/* GEMM1 over sorted rows (block_m must be 128).  For every routed row r listed
 * by the sort: g = MXFP4(X[t]) . MXFP4(W1[e, gate rows]), u = ... (up rows),
 * h = silu(g) * u in fp32 (silu(g) = g / (1 + exp(-g)); no clamp, no bias,
 * top-k weights not applied), and h is requantised with the rule above:
 * out_q [T*topk, I/2] packed codes and out_s [T*topk, I/32] E8M0 bytes, row r.
 * X_bf16 [T, D]; W1q/W1s from a4w4_moe_prepare_w1.
 * Activation quantisation: with ws == NULL and ws_bytes == 0 each GEMM tile
 * quantises its gathered rows inline (as on the source pages).  Given a
 * workspace of at least a4w4_moe_gemm1_workspace_bytes(T, D) bytes, the tokens
 * are quantised once into it (codes [T, D/2] then scales [T, D/32]) and the
 * tiles gather those rows: each token feeds topk rows times I/128 tiles, so
 * this is the faster choice once T reaches a few tokens.  Same results. */
size_t a4w4_moe_gemm1_workspace_bytes(int T, int D);
int a4w4_moe_gemm1(const void* X_bf16, int T, int D, const int32_t* sorted_rows,
                   const int32_t* block_expert, const int32_t* num_blocks, int topk,
                   const void* W1q, const void* W1s, int E, int I, void* out_q, void* out_s,
                   void* ws, size_t ws_bytes, void* stream);

/* GEMM1 with a choice of activation and output layout; a4w4_moe_gemm1(...) is
 * a4w4_moe_gemm1_ex(..., A4W4_MOE_ACT_SWIGLU, A4W4_MOE_OUT_ROWS, ...).
 * "[gfx1250] Fuse A4W4 stage1 FP4 quantization", Summary: the epilogue emits
 * packed MXFP4 payloads and preshuffled E8M0 scales after SiLU or SwiGLU.
 *   activation:
 *     A4W4_MOE_ACT_SWIGLU  W1 prepared by a4w4_moe_prepare_w1 from [E, 2I, D]
 *                          (gate rows then up rows); h = silu(gate) * up.
 *     A4W4_MOE_ACT_SILU    the ungated form: W1[e] is [I, D], prepared as one
 *                          dense matrix [E*I, D] by a4w4_prepare_gemm_weight
 *                          (expert e starts at e * a4w4_weight_codes_bytes(I, D)
 *                          in W1q, e * a4w4_weight_scales_bytes(I, D) in W1s);
 *                          h = silu(x . w).  I % 256 == 0.
 *   out_layout:
 *     A4W4_MOE_OUT_ROWS    out_q [T*topk, I/2], out_s [T*topk, I/32], row r =
 *                          routed row r (as a4w4_moe_gemm1).
 *     A4W4_MOE_OUT_TILES   the operand layout a4w4_moe_gemm2 reads: for sorted
 *                          block b (128 slots) and K tile kt (256 of the I
 *                          columns; KT = I/256), atom a = b*KT + kt holds the
 *                          codes of slot b*128 + r at out_q + a*16384 in the Wq
 *                          tile layout above (row r, byte b') and its E8M0 scales
 *                          at out_s + a*1024 in the Ws layout; padding slots
 *                          hold zeros.  Sizes a4w4_moe_tiles_codes_bytes /
 *                          _scales_bytes; tiles of blocks at or beyond
 *                          *num_blocks are not written.  I % 256 == 0. */
enum { A4W4_MOE_ACT_SWIGLU = 0, A4W4_MOE_ACT_SILU = 1 };
enum { A4W4_MOE_OUT_ROWS = 0, A4W4_MOE_OUT_TILES = 1 };
size_t a4w4_moe_tiles_codes_bytes(int T, int topk, int E, int I);
size_t a4w4_moe_tiles_scales_bytes(int T, int topk, int E, int I);
int a4w4_moe_gemm1_ex(const void* X_bf16, int T, int D, const int32_t* sorted_rows,
                      const int32_t* block_expert, const int32_t* num_blocks, int topk,
                      const void* W1q, const void* W1s, int E, int I, int activation, int out_layout,
                      void* out_q, void* out_s, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Grouped MoE GEMM2 (down projection) with the top-k weighted per-token sum.
 * "[HIP] [CK] [FlyDSL] [Kernel] Extend MXFP4 GEMM1 replacement to A4W4",
 * Summary (stage-2 paths that consume stage 1's layout) and GEMM2 scope.
 *   Y[t, :] = sum_k topk_weights[t, k] * MXFP4(W2[e_tk]) . a~_(t*topk+k)
 * with a~ GEMM1's MXFP4 output in A4W4_MOE_OUT_TILES layout (A_q, A_s; I
 * columns), the same sort as GEMM1 (sorted_rows, block_expert, num_blocks,
 * block_m 128), topk_weights float32 [T, topk] (4-byte aligned), W2q/W2s the
 * dense preshuffled layout of the stacked [E*D, I] matrix
 * (a4w4_prepare_gemm_weight; expert e at e * a4w4_weight_codes_bytes(D, I) and
 * e * a4w4_weight_scales_bytes(D, I)), Y_bf16 [T, D].
 * Each routed row's product is scaled by its weight in fp32 and stored as an
 * fp32 row of the workspace ([T*topk, D], a4w4_moe_gemm2_workspace_bytes);
 * a second kernel adds a token's rows in k order (bitwise deterministic) and
 * rounds to BF16.  I % 256 == 0, I <= 1024, D % 256 == 0. */
size_t a4w4_moe_gemm2_workspace_bytes(int T, int topk, int D);
int a4w4_moe_gemm2(const void* A_q, const void* A_s, int T, int I, const int32_t* sorted_rows,
                   const int32_t* block_expert, const int32_t* num_blocks, int topk,
                   const float* topk_weights, const void* W2q, const void* W2s, int E, int D,
                   void* Y_bf16, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Dense A4W4 GEMM that allocates nothing (no counterpart on the source pages:
 * it exists for callers of this library).  Same arguments and result as
 * a4w4_gemm() minus the workspace: the same plan, kernels and reduction order,
 * so the output is bit-identical.  For callers that cannot allocate device
 * memory where they call the GEMM -- code under a framework allocator that
 * owns all device memory, or a latency-critical path that cannot afford
 * cudaMalloc's implicit synchronisation -- and so cannot hand a4w4_gemm() the
 * workspace its plan needs for M > 64: the activations quantised once into
 * MXFP4 tiles (64 < M <= 128 when N >= 4096, every M > 128).  Smaller M uses
 * no scratch.
 *   Scratch: a fixed 16 MiB array inside the library's device image.  It comes
 *   into being on a device with the first a4w4_gemm_noalloc call there (the
 *   CUDA runtime loads the library's device code lazily), which also looks up
 *   its device address, whatever the shape; make that first call before any
 *   stream capture.  It stays until the process exits.  No call allocates.
 *   A plan needing more than 16 MiB (a4w4_gemm_workspace_bytes(M, N, K) >
 *   16 MiB: at K = 7168, M above about 4,400 rows) is refused with
 *   A4W4_ERR_WORKSPACE.  All calls on a GPU share the array and it keeps the
 *   last call's contents (overwritten before they are read); calls that may
 *   run at the same time on one GPU (different streams) race on it --
 *   serialise them. */
int a4w4_gemm_noalloc(const void* A_bf16, int M, int K, const void* Wq, const void* Ws, int N,
                      void* C_bf16, void* stream);

/* ------------------------------------------------------------------------ */
/* Synchronises `stream`, then returns and clears the device status word:
 * A4W4_OK, A4W4_ERR_TIMEOUT, or A4W4_ERR_LAUNCH if the stream reported an error. */
int a4w4_get_device_status(void* stream);

/* Static, human-readable name of a return code. */
const char* a4w4_strerror(int code);

/* Override the in-kernel wait limit in nanoseconds (0 restores the default of
 * 2e8 ns).  Applies to launches issued after the call; used to test that an
 * expired wait is reported rather than hanging. */
void a4w4_set_wait_limit_ns(unsigned long long ns);

#ifdef __cplusplus
}
#endif

#endif /* A4W4_H_ */
