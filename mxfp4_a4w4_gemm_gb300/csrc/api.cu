// api.cu -- the extern "C" boundary of liba4w4.so (declared in include/a4w4.h):
// argument validation, device checks, launch, and the device status word.
#include <atomic>
#include <cstdint>
#include <cstdio>

#include "a4w4.h"
#include "a4w4_debug.h"
#include "launch.h"

// Device status word: bit 0 set by a kernel whose bounded wait expired.
// Every GPU that loads the library holds these 4 bytes until exit.
static __device__ unsigned int g_status = 0u;
static constexpr unsigned int kStatusTimeout = 1u;

namespace {

constexpr unsigned long long kDefaultWaitNs = 200000000ull;   // 0.2 s
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};

constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_sms[kMaxDevices];      // 0 = unknown, -1 = unsupported, else SM count

// SM count of the current device if it is a compute capability 10.3 GPU,
// else a negative A4W4 error code.
int current_device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return A4W4_ERR_DEVICE;
  if (dev < kMaxDevices) {
    const int v = g_dev_sms[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (v < 0) return A4W4_ERR_DEVICE;
  }
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    return A4W4_ERR_DEVICE;
  }
  const int v = (major == 10 && minor == 3 && sms > 0) ? sms : -1;
  if (dev < kMaxDevices) g_dev_sms[dev].store(v, std::memory_order_relaxed);
  return v > 0 ? v : A4W4_ERR_DEVICE;
}

// Device address of g_status on the current device (looked up once per device).
std::atomic<unsigned int*> g_status_ptr[kMaxDevices];

unsigned int* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned int* p = g_status_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status) != cudaSuccess) return nullptr;
    p = static_cast<unsigned int*>(addr);
    g_status_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

// SM count for sizing a workspace; GB300's count when no device is visible.
int sizing_sms() {
  const int s = current_device_sms();
  return s > 0 ? s : 152;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

size_t padded_k(int K) { return static_cast<size_t>((K + 255) / 256) * 256; }

}  // namespace

namespace a4w4 {
int device_sms() { return current_device_sms(); }
unsigned int* device_status_ptr() { return status_ptr(); }
unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
}  // namespace a4w4

namespace {

// Shared body of a4w4_gemm_ex and the activation-export test hook.
int gemm_impl(const void* A_bf16, int M, int K, const void* Wq, const void* Ws, int N, void* C_bf16,
              void* workspace, size_t ws_bytes, unsigned int flags, void* stream, a4w4::ActDump dump) {
  if (M <= 0 || N <= 0 || K <= 0 || N % 256 != 0 || K % 128 != 0) return A4W4_ERR_ARG;
  if (!aligned16(A_bf16) || !aligned16(Wq) || !aligned16(Ws) || !aligned16(C_bf16)) return A4W4_ERR_ARG;
  if ((flags & ~static_cast<unsigned int>(A4W4_GEMM_WEIGHT_PREFETCH)) != 0) return A4W4_ERR_ARG;
  const int sms = current_device_sms();
  if (sms < 0) return sms;
  const a4w4::GemmPlan plan = a4w4::plan_gemm(M, N, K, sms);
  if (plan.ws_bytes > 0 && (ws_bytes < plan.ws_bytes || !aligned16(workspace))) return A4W4_ERR_WORKSPACE;
  unsigned int* status = status_ptr();
  if (status == nullptr) return A4W4_ERR_LAUNCH;
  return a4w4::launch_gemm(plan, A_bf16, M, K, Wq, Ws, N, C_bf16, workspace, as_stream(stream),
                           g_wait_ns.load(std::memory_order_relaxed), status,
                           (flags & A4W4_GEMM_WEIGHT_PREFETCH) ? 1 : 0, dump);
}

int moe_gemm1_impl(const void* X_bf16, int T, int D, const int32_t* sorted_rows, const int32_t* block_expert,
                   const int32_t* num_blocks, int topk, const void* W1q, const void* W1s, int E, int I, int act,
                   int out_layout, void* out_q, void* out_s, void* ws, size_t ws_bytes, void* stream,
                   a4w4::ActDump dump) {
  if (T <= 0 || D <= 0 || topk <= 0 || E <= 0 || I <= 0 || I % 128 != 0 || D % 128 != 0) return A4W4_ERR_ARG;
  if (act != A4W4_MOE_ACT_SWIGLU && act != A4W4_MOE_ACT_SILU) return A4W4_ERR_ARG;
  if (out_layout != A4W4_MOE_OUT_ROWS && out_layout != A4W4_MOE_OUT_TILES) return A4W4_ERR_ARG;
  // SiLU tiles hold 256 output columns; operand tiles are whole 256-wide K tiles
  if ((act == A4W4_MOE_ACT_SILU || out_layout == A4W4_MOE_OUT_TILES) && I % 256 != 0) return A4W4_ERR_ARG;
  if (static_cast<long long>(T) * topk > (1ll << 30)) return A4W4_ERR_ARG;
  if (!aligned16(X_bf16) || !aligned16(W1q) || !aligned16(W1s) || !aligned16(out_q) || out_s == nullptr ||
      sorted_rows == nullptr || block_expert == nullptr || num_blocks == nullptr)
    return A4W4_ERR_ARG;
  const int sms = current_device_sms();
  if (sms < 0) return sms;
  const int max_blocks = a4w4_moe_max_blocks(T, topk, E, 128);
  if (max_blocks > 65535) return A4W4_ERR_ARG;
  unsigned int* status = status_ptr();
  if (status == nullptr) return A4W4_ERR_LAUNCH;
  void* xq = nullptr;
  if (ws != nullptr || ws_bytes != 0) {
    if (!aligned16(ws) || ws_bytes < a4w4_moe_gemm1_workspace_bytes(T, D)) return A4W4_ERR_WORKSPACE;
    xq = ws;
  }
  return a4w4::launch_moe_gemm1(X_bf16, T, D, sorted_rows, block_expert, num_blocks, max_blocks, topk, W1q, W1s,
                                E, I, act, out_layout == A4W4_MOE_OUT_TILES ? 1 : 0, out_q, out_s, xq,
                                as_stream(stream), g_wait_ns.load(std::memory_order_relaxed), status, sms, dump);
}

}  // namespace

extern "C" {

size_t a4w4_weight_codes_bytes(int N, int K) {
  if (N <= 0 || K <= 0) return 0;
  return static_cast<size_t>(N) * padded_k(K) / 2;
}

size_t a4w4_weight_scales_bytes(int N, int K) {
  if (N <= 0 || K <= 0) return 0;
  return static_cast<size_t>(N) * padded_k(K) / 32;
}

int a4w4_prepare_gemm_weight(const void* W_bf16, int N, int K, void* Wq, void* Ws, void* stream) {
  if (N <= 0 || K <= 0 || N % 256 != 0 || K % 128 != 0) return A4W4_ERR_ARG;
  if (!aligned16(W_bf16) || !aligned16(Wq) || !aligned16(Ws)) return A4W4_ERR_ARG;
  const int sms = current_device_sms();
  if (sms < 0) return sms;
  return a4w4::launch_prepare_weight(W_bf16, N, K, 1, 0, Wq, Ws, as_stream(stream), sms);
}

size_t a4w4_gemm_workspace_bytes(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return a4w4::plan_gemm(M, N, K, sizing_sms()).ws_bytes;
}

int a4w4_gemm_kernel_name(int M, int N, int K, char* buf, size_t n) {
  if (M <= 0 || N <= 0 || K <= 0 || N % 256 != 0 || K % 128 != 0 || buf == nullptr || n == 0) return A4W4_ERR_ARG;
  const a4w4::GemmPlan pl = a4w4::plan_gemm(M, N, K, sizing_sms());
  if (pl.decode)
    snprintf(buf, n, "a4w4_decode_kernel<%d,%d>", pl.nx, pl.ring);
  else if (pl.persistent)
    snprintf(buf, n, "a4w4_large_kernel<prequant,persistent>");
  else
    snprintf(buf, n, "a4w4_gemm_kernel<swap,%d>", pl.nx);
  return A4W4_OK;
}

int a4w4_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (ws_bytes == 0) return A4W4_OK;
  if (!aligned16(workspace)) return A4W4_ERR_ARG;
  return cudaMemsetAsync(workspace, 0, ws_bytes, as_stream(stream)) == cudaSuccess ? A4W4_OK : A4W4_ERR_LAUNCH;
}

int a4w4_gemm_ex(const void* A_bf16, int M, int K, const void* Wq, const void* Ws, int N, void* C_bf16,
                 void* workspace, size_t ws_bytes, unsigned int flags, void* stream) {
  return gemm_impl(A_bf16, M, K, Wq, Ws, N, C_bf16, workspace, ws_bytes, flags, stream, a4w4::ActDump{});
}

int a4w4_gemm(const void* A_bf16, int M, int K, const void* Wq, const void* Ws, int N, void* C_bf16,
              void* workspace, size_t ws_bytes, void* stream) {
  return gemm_impl(A_bf16, M, K, Wq, Ws, N, C_bf16, workspace, ws_bytes, 0u, stream, a4w4::ActDump{});
}

int a4w4_gemm_a16w4(const void* A_bf16, int M, int K, const void* Wq, const void* Ws, int N, void* C_bf16,
                    unsigned int flags, void* stream) {
  if (M <= 0 || N <= 0 || K <= 0 || N % 256 != 0 || K % 128 != 0) return A4W4_ERR_ARG;
  if (!aligned16(A_bf16) || !aligned16(Wq) || !aligned16(Ws) || !aligned16(C_bf16)) return A4W4_ERR_ARG;
  if ((flags & ~static_cast<unsigned int>(A4W4_GEMM_WEIGHT_PREFETCH)) != 0) return A4W4_ERR_ARG;
  const int sms = current_device_sms();
  if (sms < 0) return sms;
  unsigned int* status = status_ptr();
  if (status == nullptr) return A4W4_ERR_LAUNCH;
  const a4w4::GemmPlan plan = a4w4::plan_a16w4(M, N, K, sms);
  return a4w4::launch_a16w4(plan, A_bf16, M, K, Wq, Ws, N, C_bf16, as_stream(stream),
                            g_wait_ns.load(std::memory_order_relaxed), status,
                            (flags & A4W4_GEMM_WEIGHT_PREFETCH) ? 1 : 0);
}

int a4w4_mxfp4_quant(const void* X_bf16, int rows, int cols, void* q, void* scales, void* stream) {
  if (rows <= 0 || cols <= 0 || cols % 32 != 0) return A4W4_ERR_ARG;
  if (!aligned16(X_bf16) || !aligned16(q) || scales == nullptr) return A4W4_ERR_ARG;
  const int sms = current_device_sms();
  if (sms < 0) return sms;
  return a4w4::launch_mxfp4_quant(X_bf16, rows, cols, q, scales, as_stream(stream), sms);
}

size_t a4w4_moe_w1_codes_bytes(int E, int two_I, int D) {
  if (E <= 0) return 0;
  return static_cast<size_t>(E) * a4w4_weight_codes_bytes(two_I, D);
}

size_t a4w4_moe_w1_scales_bytes(int E, int two_I, int D) {
  if (E <= 0) return 0;
  return static_cast<size_t>(E) * a4w4_weight_scales_bytes(two_I, D);
}

int a4w4_moe_prepare_w1(const void* W1_bf16, int E, int two_I, int D, void* W1q, void* W1s, void* stream) {
  if (E <= 0 || two_I <= 0 || D <= 0 || two_I % 256 != 0 || D % 128 != 0) return A4W4_ERR_ARG;
  if (!aligned16(W1_bf16) || !aligned16(W1q) || !aligned16(W1s)) return A4W4_ERR_ARG;
  const int sms = current_device_sms();
  if (sms < 0) return sms;
  return a4w4::launch_prepare_weight(W1_bf16, two_I, D, E, two_I / 2, W1q, W1s, as_stream(stream), sms);
}

int a4w4_moe_max_blocks(int T, int topk, int E, int block_m) {
  if (T <= 0 || topk <= 0 || E <= 0 || block_m <= 0) return 0;
  const long long n = static_cast<long long>(T) * topk;
  const long long active = n < E ? n : E;
  return static_cast<int>((n + block_m - 1) / block_m + active);
}

size_t a4w4_moe_sort_workspace_bytes(int T, int topk, int E) {
  if (T <= 0 || topk <= 0 || E <= 0) return 0;
  return a4w4::moe_sort_ws_bytes(T, topk, E);
}

int a4w4_moe_sort(const int32_t* topk_ids, int T, int topk, int E, int block_m, int32_t* sorted_rows,
                  int32_t* block_expert, int32_t* num_blocks, void* ws, size_t ws_bytes, void* stream) {
  if (T <= 0 || topk <= 0 || E <= 0 || E > 8192) return A4W4_ERR_ARG;
  if (block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128) return A4W4_ERR_ARG;
  if (static_cast<long long>(T) * topk > (1ll << 30)) return A4W4_ERR_ARG;
  if (topk_ids == nullptr || sorted_rows == nullptr || block_expert == nullptr || num_blocks == nullptr)
    return A4W4_ERR_ARG;
  if (ws == nullptr || ws_bytes < a4w4::moe_sort_ws_bytes(T, topk, E)) return A4W4_ERR_WORKSPACE;
  const int sms = current_device_sms();
  if (sms < 0) return sms;
  return a4w4::launch_moe_sort(topk_ids, T, topk, E, block_m, sorted_rows, block_expert, num_blocks, ws,
                               as_stream(stream));
}

size_t a4w4_moe_sort_aux_workspace_bytes(int T, int topk, int E) {
  if (T <= 0 || topk <= 0 || E <= 0) return 0;
  return a4w4::moe_sort_aux_ws_bytes(T, topk, E, sizing_sms());
}

int a4w4_moe_sort_aux(const int32_t* topk_ids, int T, int topk, int E, int block_m, int32_t* sorted_rows,
                      int32_t* block_expert, int32_t* num_blocks, int32_t* sorted_tokens, int32_t* row_slot,
                      void* ws, size_t ws_bytes, void* stream) {
  if (T <= 0 || topk <= 0 || E <= 0 || E > 4096) return A4W4_ERR_ARG;
  if (block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128) return A4W4_ERR_ARG;
  if (topk_ids == nullptr || sorted_rows == nullptr || block_expert == nullptr || num_blocks == nullptr ||
      sorted_tokens == nullptr || row_slot == nullptr)
    return A4W4_ERR_ARG;
  const int sms = current_device_sms();
  if (sms < 0) return sms;
  if (static_cast<long long>(T) * topk > static_cast<long long>(sms) * 32768) return A4W4_ERR_ARG;
  if (!aligned16(ws) || ws_bytes < a4w4::moe_sort_aux_ws_bytes(T, topk, E, sms)) return A4W4_ERR_WORKSPACE;
  unsigned int* status = status_ptr();
  if (status == nullptr) return A4W4_ERR_LAUNCH;
  const int rc = a4w4::launch_moe_sort_aux(topk_ids, T, topk, E, block_m, sorted_rows, block_expert, num_blocks,
                                           sorted_tokens, row_slot, ws, as_stream(stream), sms,
                                           g_wait_ns.load(std::memory_order_relaxed), status);
  return rc == -1 ? A4W4_ERR_ARG : rc;
}

size_t a4w4_moe_gemm1_workspace_bytes(int T, int D) {
  if (T <= 0 || D <= 0) return 0;
  return static_cast<size_t>(T) * (D / 2) + static_cast<size_t>(T) * (D / 32);
}

int a4w4_moe_gemm1(const void* X_bf16, int T, int D, const int32_t* sorted_rows, const int32_t* block_expert,
                   const int32_t* num_blocks, int topk, const void* W1q, const void* W1s, int E, int I,
                   void* out_q, void* out_s, void* ws, size_t ws_bytes, void* stream) {
  return moe_gemm1_impl(X_bf16, T, D, sorted_rows, block_expert, num_blocks, topk, W1q, W1s, E, I,
                        A4W4_MOE_ACT_SWIGLU, A4W4_MOE_OUT_ROWS, out_q, out_s, ws, ws_bytes, stream, a4w4::ActDump{});
}

int a4w4_moe_gemm1_ex(const void* X_bf16, int T, int D, const int32_t* sorted_rows, const int32_t* block_expert,
                      const int32_t* num_blocks, int topk, const void* W1q, const void* W1s, int E, int I,
                      int activation, int out_layout, void* out_q, void* out_s, void* ws, size_t ws_bytes,
                      void* stream) {
  return moe_gemm1_impl(X_bf16, T, D, sorted_rows, block_expert, num_blocks, topk, W1q, W1s, E, I, activation,
                        out_layout, out_q, out_s, ws, ws_bytes, stream, a4w4::ActDump{});
}

size_t a4w4_moe_tiles_codes_bytes(int T, int topk, int E, int I) {
  if (T <= 0 || topk <= 0 || E <= 0 || I <= 0) return 0;
  return static_cast<size_t>(a4w4_moe_max_blocks(T, topk, E, 128)) * ((I + 255) / 256) * 16384;
}

size_t a4w4_moe_tiles_scales_bytes(int T, int topk, int E, int I) {
  if (T <= 0 || topk <= 0 || E <= 0 || I <= 0) return 0;
  return static_cast<size_t>(a4w4_moe_max_blocks(T, topk, E, 128)) * ((I + 255) / 256) * 1024;
}

size_t a4w4_moe_gemm2_workspace_bytes(int T, int topk, int D) {
  if (T <= 0 || topk <= 0 || D <= 0) return 0;
  return static_cast<size_t>(T) * topk * D * sizeof(float);
}

int a4w4_moe_gemm2(const void* A_q, const void* A_s, int T, int I, const int32_t* sorted_rows,
                   const int32_t* block_expert, const int32_t* num_blocks, int topk, const float* topk_weights,
                   const void* W2q, const void* W2s, int E, int D, void* Y_bf16, void* ws, size_t ws_bytes,
                   void* stream) {
  if (T <= 0 || I <= 0 || topk <= 0 || E <= 0 || D <= 0 || I % 256 != 0 || D % 256 != 0 || I > 1024)
    return A4W4_ERR_ARG;
  if (static_cast<long long>(T) * topk > (1ll << 30)) return A4W4_ERR_ARG;
  if (!aligned16(A_q) || A_s == nullptr || !aligned16(W2q) || !aligned16(W2s) || !aligned16(Y_bf16) ||
      sorted_rows == nullptr || block_expert == nullptr || num_blocks == nullptr || topk_weights == nullptr ||
      (reinterpret_cast<uintptr_t>(topk_weights) & 3u) != 0)
    return A4W4_ERR_ARG;
  if (!aligned16(ws) || ws_bytes < a4w4_moe_gemm2_workspace_bytes(T, topk, D)) return A4W4_ERR_WORKSPACE;
  const int sms = current_device_sms();
  if (sms < 0) return sms;
  const int max_blocks = a4w4_moe_max_blocks(T, topk, E, 128);
  if (max_blocks > 65535) return A4W4_ERR_ARG;
  unsigned int* status = status_ptr();
  if (status == nullptr) return A4W4_ERR_LAUNCH;
  const cudaStream_t st = as_stream(stream);
  float* partial = static_cast<float*>(ws);
  // The persistent walk (each block's activation tiles resident over its
  // column tiles); the entry checks above keep I <= 1024, which it holds.
  const unsigned long long wait = g_wait_ns.load(std::memory_order_relaxed);
  const int rc = a4w4::launch_moe_gemm2_persistent(A_q, A_s, T, I, sorted_rows, block_expert, num_blocks, max_blocks,
                                                   topk, topk_weights, W2q, W2s, E, D, partial, st, wait, status, sms);
  if (rc != 0) return rc == -1 ? A4W4_ERR_ARG : rc;
  return a4w4::launch_moe_sum(partial, T, topk, D, Y_bf16, st, sms);
}

// ---------------------------------------------------------------------------
// Test hooks (a4w4_debug.h)

int a4w4_debug_gemm_activation_layout(int M, int N, int K, int* tile_rows, int* x_tiles, int* k_tiles) {
  if (M <= 0 || N <= 0 || K <= 0 || N % 256 != 0 || K % 128 != 0) return A4W4_ERR_ARG;
  if (tile_rows == nullptr || x_tiles == nullptr || k_tiles == nullptr) return A4W4_ERR_ARG;
  const a4w4::GemmPlan pl = a4w4::plan_gemm(M, N, K, sizing_sms());
  *tile_rows = pl.nx;
  *x_tiles = pl.x_tiles;
  *k_tiles = pl.kt;
  return A4W4_OK;
}

int a4w4_debug_gemm_export(const void* A_bf16, int M, int K, const void* Wq, const void* Ws, int N, void* C_bf16,
                           void* workspace, size_t ws_bytes, void* dump, size_t dump_bytes, void* stream) {
  if (M <= 0 || N <= 0 || K <= 0 || N % 256 != 0 || K % 128 != 0 || !aligned16(dump)) return A4W4_ERR_ARG;
  const int sms = current_device_sms();
  if (sms < 0) return sms;
  const a4w4::GemmPlan pl = a4w4::plan_gemm(M, N, K, sms);
  const size_t atoms = static_cast<size_t>(pl.x_tiles) * pl.kt;
  const size_t code_bytes = atoms * pl.nx * 128;
  if (dump_bytes < code_bytes + atoms * 1024) return A4W4_ERR_ARG;
  const cudaStream_t st = as_stream(stream);
  if (cudaMemsetAsync(dump, 0, code_bytes + atoms * 1024, st) != cudaSuccess) return A4W4_ERR_LAUNCH;
  a4w4::ActDump d{static_cast<uint8_t*>(dump), static_cast<uint8_t*>(dump) + code_bytes};
  // the quantise-once plans build their tiles in the workspace, not in the
  // producers: copy those out after the GEMM instead
  const int rc = gemm_impl(A_bf16, M, K, Wq, Ws, N, C_bf16, workspace, ws_bytes, 0u, stream,
                           pl.prequant ? a4w4::ActDump{} : d);
  if (rc != A4W4_OK || !pl.prequant) return rc;
  // the workspace holds 17 KB atoms (codes, then scales): split them
  const uint8_t* w8 = static_cast<const uint8_t*>(workspace);
  if (cudaMemcpy2DAsync(d.codes, 16384, w8, 17408, 16384, atoms, cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
      cudaMemcpy2DAsync(d.scales, 1024, w8 + 16384, 17408, 1024, atoms, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return A4W4_ERR_LAUNCH;
  return A4W4_OK;
}

int a4w4_debug_moe_gemm1_export(const void* X_bf16, int T, int D, const int32_t* sorted_rows,
                                const int32_t* block_expert, const int32_t* num_blocks, int topk, const void* W1q,
                                const void* W1s, int E, int I, void* out_q, void* out_s, void* ws, size_t ws_bytes,
                                void* dump, size_t dump_bytes, void* stream) {
  if (T <= 0 || D <= 0 || topk <= 0 || E <= 0 || D % 128 != 0 || !aligned16(dump)) return A4W4_ERR_ARG;
  const size_t atoms = static_cast<size_t>(a4w4_moe_max_blocks(T, topk, E, 128)) * ((D + 255) / 256);
  if (dump_bytes < atoms * (16384 + 1024)) return A4W4_ERR_ARG;
  if (cudaMemsetAsync(dump, 0, atoms * (16384 + 1024), as_stream(stream)) != cudaSuccess) return A4W4_ERR_LAUNCH;
  a4w4::ActDump d{static_cast<uint8_t*>(dump), static_cast<uint8_t*>(dump) + atoms * 16384};
  return moe_gemm1_impl(X_bf16, T, D, sorted_rows, block_expert, num_blocks, topk, W1q, W1s, E, I,
                        A4W4_MOE_ACT_SWIGLU, A4W4_MOE_OUT_ROWS, out_q, out_s, ws, ws_bytes, stream, d);
}

int a4w4_get_device_status(void* stream) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return A4W4_ERR_LAUNCH;
  unsigned int st = 0u;
  if (cudaMemcpyFromSymbol(&st, g_status, sizeof(st)) != cudaSuccess) return A4W4_ERR_LAUNCH;
  const unsigned int zero = 0u;
  if (cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) return A4W4_ERR_LAUNCH;
  return (st & kStatusTimeout) ? A4W4_ERR_TIMEOUT : A4W4_OK;
}

const char* a4w4_strerror(int code) {
  switch (code) {
    case A4W4_OK: return "ok";
    case A4W4_ERR_ARG: return "invalid argument (null or misaligned pointer, or shape outside the contract)";
    case A4W4_ERR_DEVICE: return "unsupported device (a compute capability 10.3 GPU is required)";
    case A4W4_ERR_WORKSPACE: return "workspace missing or too small";
    case A4W4_ERR_LAUNCH: return "CUDA launch or runtime error";
    case A4W4_ERR_TIMEOUT: return "an in-kernel wait expired";
    default: return "unknown error";
  }
}

void a4w4_set_wait_limit_ns(unsigned long long ns) {
  g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns, std::memory_order_relaxed);
}

}  // extern "C"
