// noalloc.cu -- a dense A4W4 GEMM entry point that allocates nothing.
//
// a4w4_gemm() needs a caller-allocated workspace whenever it splits K across
// the SMs (small M).  Some callers cannot provide one: code that runs under a
// framework allocator owning all device memory, or a latency-critical path
// where cudaMalloc's implicit synchronisation is not acceptable.  This entry
// point runs the same GEMM with its split-K scratch (fp32 partial tiles and
// tile counters) in a fixed array that is part of the library's device image.
//
// The array is kNoAllocScratchBytes (16 MiB) on every GPU that loads the
// library, kept until the process exits.  A call whose tile plan needs more
// scratch than that is refused with A4W4_ERR_WORKSPACE.  All calls on a GPU
// share its array, which keeps whatever the last call left there: the tile
// counters are cleared at the start of every call, and calls that can run at
// the same time on one GPU (issued on different streams) race on the array,
// so the caller must serialise them.
#include <atomic>
#include <cstdint>

#include "a4w4.h"
#include "launch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_gemm_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of g_gemm_scratch on the current device.  Host code only
// sees a host-side stand-in under that name, so the real address is looked up
// once per device (with that device current) and cached.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p != nullptr) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_gemm_scratch) != cudaSuccess || addr == nullptr) return nullptr;
  g_scratch_addr[dev].store(addr, std::memory_order_release);
  return addr;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

int a4w4_gemm_noalloc(const void* A_bf16, int M, int K, const void* Wq, const void* Ws, int N, void* C_bf16,
                      void* stream) {
  if (M <= 0 || N <= 0 || K <= 0 || N % 256 != 0 || K % 128 != 0) return A4W4_ERR_ARG;
  if (!aligned16(A_bf16) || !aligned16(Wq) || !aligned16(Ws) || !aligned16(C_bf16)) return A4W4_ERR_ARG;
  const int sms = a4w4::device_sms();
  if (sms < 0) return sms;
  const a4w4::GemmPlan plan = a4w4::plan_gemm(M, N, K, sms);
  if (plan.ws_bytes > kNoAllocScratchBytes) return A4W4_ERR_WORKSPACE;
  unsigned int* status = a4w4::device_status_ptr();
  if (status == nullptr) return A4W4_ERR_LAUNCH;
  void* scratch = nullptr;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (plan.ws_bytes > 0) {
    scratch = scratch_address();
    if (scratch == nullptr) return A4W4_ERR_LAUNCH;
    // The split-K tile counters must start at zero; a previous call (or one
    // that timed out) may have left them otherwise.  They follow the
    // activation tiles and the partials in the scratch layout.
    const size_t counters = plan.aq_bytes + plan.partial_bytes;
    if (plan.ws_bytes > counters &&
        cudaMemsetAsync(static_cast<unsigned char*>(scratch) + counters, 0, plan.ws_bytes - counters, st) != cudaSuccess)
      return A4W4_ERR_LAUNCH;
  }
  return a4w4::launch_gemm(plan, A_bf16, M, K, Wq, Ws, N, C_bf16, scratch, st, a4w4::wait_limit_ns(), status);
}

}  // extern "C"
