// launch.h -- host-side launchers behind the C ABI (internal).
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace a4w4 {

// Tile plan of one dense GEMM call: a pure function of (M, N, K, SM count),
// shared by a4w4_gemm and a4w4_gemm_workspace_bytes.
struct GemmPlan {
  int swap_ab;      // 1: weights are the MMA's M side (small M)
  int decode;       // 1: the decode kernel (decode.cu): M <= 16, and some M <= 32 (plan_gemm)
  int prequant;     // 1: activations quantised once into tiles first (M > 128; M > 64 when N >= 4096)
  int persistent;   // 1 (every prequant plan): the persistent large-M kernel (large.cu)
  int half_tiles;   // persistent: tiles of the last partial wave run as two 128-column halves
  size_t aq_bytes;  // workspace bytes of the quantised activation tiles (codes + scales)
  int nx;           // activation rows per CTA
  int w_tiles;      // weight-row tiles (N / 128 or N / 256)
  int x_tiles;      // activation-row tiles
  int splits;       // K splits
  int ring;         // decode kernel: weight ring depth (K tiles in flight per CTA)
  int cluster_reduce;     // 1: the splits of a tile form a cluster and reduce over DSMEM
  int kt;           // 256-wide K tiles
  size_t ws_bytes;        // workspace: the activation tiles (aq_bytes), or 0
};

GemmPlan plan_gemm(int M, int N, int K, int sms);

// Kernel function attributes (dynamic shared memory size, non-portable
// cluster sizes) belong to the current device's context.  A launcher keeps
// one bit per device in `done` and runs `set` only where that bit is clear
// (devices beyond 63 run it on every launch).  Returns 0, or -4 when the
// device cannot be read or `set` reports a failed attribute call.
template <typename SetFn>
int ensure_func_attrs(std::atomic<unsigned long long>& done, SetFn set) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -4;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return 0;
  if (!set()) return -4;
  if (bit != 0) done.fetch_or(bit, std::memory_order_release);
  return 0;
}

// Launch `kern` on a 1-D grid with programmatic stream serialisation (the
// kernels launched this way order their global reads after
// griddepcontrol.wait, so they may start while the previous grid finishes).
// Returns 0 or -4.
template <typename... Params, typename... Args>
int launch_pdl(void (*kern)(Params...), int grid, int block, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, args...) != cudaSuccess) return -4;
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Shared by the C ABI entry points (defined in api.cu): SM count of the
// current device if it is a compute capability 10.3 GPU, else a negative
// A4W4 error code; device address of the status word; the current wait limit.
int device_sms();
unsigned int* device_status_ptr();
unsigned long long wait_limit_ns();

// Test hook (a4w4_debug.h): where the activation producers of the CTAs of
// weight tile 0 also store the MXFP4 operand tiles they build in shared
// memory.  Atom a = x_tile * KT + kt: codes at codes + a * (rows per tile *
// 128) in the swizzled tile layout, scales at scales + a * 1024 in the
// scale-atom layout.  codes == nullptr: off (every product call).
struct ActDump {
  uint8_t* codes;
  uint8_t* scales;
};

int launch_mxfp4_quant(const void* x, long long rows, int cols, void* q, void* s, cudaStream_t st, int sms);
int launch_prepare_weight(const void* w, int rows, int K, int experts, int pair_I, void* wq, void* ws,
                          cudaStream_t st, int sms);
// A [M, K] -> MXFP4 tiles of 128 rows x 256 K (rows padded to 128 with zeros),
// atom x*KT + kt at aq + atom*17408: 16 KB of codes in the weight tile layout,
// then its 1 KB of scales.
int launch_quant_activation_tiles(const void* a, int M, int K, void* aq, cudaStream_t st, int sms);
// prefetch_w: weights may be read before the previous grid on the stream
// completes (the caller guarantees that grid does not write them).
int launch_gemm(const GemmPlan& plan, const void* A, int M, int K, const void* Wq, const void* Ws, int N,
                void* C, void* ws, cudaStream_t st, unsigned long long wait_ns, unsigned int* status,
                int prefetch_w, ActDump dump);
// A16WFP4 (BF16 activations x MXFP4 weights): swap-AB tiles of 16 or 32
// tokens, split-K reduced inside clusters; no workspace.
GemmPlan plan_a16w4(int M, int N, int K, int sms);
int launch_a16w4(const GemmPlan& plan, const void* A, int M, int K, const void* Wq, const void* Ws, int N, void* C,
                 cudaStream_t st, unsigned long long wait_ns, unsigned int* status, int prefetch_w);
// plan.persistent: one CTA per SM (at most `sms`) walking the 128 x 256 tiles
// of the activation tiles already quantised into `Aq`, the last
// plan.half_tiles of them as two 128-column halves each (large.cu).
int launch_large(const GemmPlan& plan, const uint8_t* Aq, int M, const void* Wq, const void* Ws, int N, void* C,
                 cudaStream_t st, unsigned long long wait_ns, unsigned int* status, int sms);
// plan.decode: the decode kernel (decode.cu); no workspace.
int launch_decode(const GemmPlan& plan, const void* A, int M, int K, const void* Wq, const void* Ws, int N,
                  void* C, cudaStream_t st, unsigned long long wait_ns, unsigned int* status, int prefetch_w,
                  ActDump dump);
// act: 0 SwiGLU (W1[e] = [2I, D] paired gate/up layout), 1 SiLU (W1[e] =
// [I, D] dense layout); out_tiles: 1 = sorted-slot operand tiles.
int launch_moe_gemm1(const void* X, int T, int D, const int32_t* sorted_rows, const int32_t* block_expert,
                     const int32_t* num_blocks, int max_blocks, int topk, const void* W1q, const void* W1s,
                     int E, int I, int act, int out_tiles, void* out_q, void* out_s, void* xq_ws, cudaStream_t st,
                     unsigned long long wait_ns, unsigned int* status, int sms, ActDump dump);
// MoE GEMM2: GEMM1's sorted-slot tiles x W2[e] ([D, I] dense layout per
// expert, I <= 1024) -> top-k weighted fp32 rows partial[T*topk, D]: one
// persistent CTA per SM walking a contiguous run of (block, 256-column tile)
// units with each block's activation tiles resident (moe2.cu).
int launch_moe_gemm2_persistent(const void* Aq, const void* As, int T, int I, const int32_t* sorted_rows,
                                const int32_t* block_expert, const int32_t* num_blocks, int max_blocks, int topk,
                                const float* topk_w, const void* W2q, const void* W2s, int E, int D, float* partial,
                                cudaStream_t st, unsigned long long wait_ns, unsigned int* status, int sms);
// Y[t, :] (BF16) = sum over k = 0..topk-1, in that order, of partial[t*topk + k, :].
int launch_moe_sum(const float* partial, int T, int topk, int D, void* Y, cudaStream_t st, int sms);
int launch_moe_sort(const int32_t* topk_ids, int T, int topk, int E, int block_m, int32_t* sorted_rows,
                    int32_t* block_expert, int32_t* num_blocks, void* ws, cudaStream_t st);
size_t moe_sort_ws_bytes(int T, int topk, int E);
// Single-launch sort with gather/scatter arrays (cooperative; E <= 4096,
// T*topk <= sms * 32768).  Workspace: histograms + 2 barrier words, zeroed once.
int launch_moe_sort_aux(const int32_t* ids, int T, int topk, int E, int bm, int32_t* sorted_rows,
                        int32_t* block_expert, int32_t* num_blocks, int32_t* sorted_tokens, int32_t* row_slot,
                        void* ws, cudaStream_t st, int sms, unsigned long long wait_ns, unsigned int* status);
size_t moe_sort_aux_ws_bytes(int T, int topk, int E, int sms);

}  // namespace a4w4
