// noalloc.cu -- a dense A4W4 GEMM entry point that allocates nothing.
//
// a4w4_gemm() takes a caller-allocated workspace whenever its tile plan needs
// one: for M > 64 (64 < M <= 128 when N >= 4096; every M > 128) the activations
// are quantised once into MXFP4 tiles there.  Smaller M needs none.  Some
// callers cannot provide that memory: code running under a framework allocator
// that owns all device memory, or a latency-critical path where cudaMalloc's
// implicit device synchronisation is not acceptable.  This entry point runs the
// same plan and kernels with that scratch in a fixed array that belongs to the
// library's device image.
//
// The array holds kNoAllocScratchBytes (16 MiB).  It comes into being on a
// device when this file's module is loaded there, which with the CUDA
// runtime's lazy module loading is the first call of a4w4_gemm_noalloc on
// that device (the call that looks its address up), and stays until the
// process exits.  A plan that needs more than 16 MiB is refused with
// A4W4_ERR_WORKSPACE; at K = 7168 that is M beyond about 4,400 rows (487 KB of
// activation tiles per 128 rows).  Every call shares the array, which keeps
// whatever the previous call left there (the activation tiles are overwritten
// before they are read); calls that can run at the same time on one GPU
// (issued on different streams) race on it.
#include <atomic>
#include <cstdint>

#include "a4w4.h"
#include "launch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_gemm_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of g_gemm_scratch on the current device.  In host code the
// array's name denotes a host-side stand-in, not device memory, so the real
// address is looked up once per device (with that device current) and cached.
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
  // Looked up on every call, whatever the shape, so that the first call on a
  // device -- the one to make before any stream capture -- does the set-up
  // even when its own plan needs no scratch.
  void* scratch = scratch_address();
  if (scratch == nullptr) return A4W4_ERR_LAUNCH;
  const a4w4::GemmPlan plan = a4w4::plan_gemm(M, N, K, sms);
  if (plan.ws_bytes > kNoAllocScratchBytes) return A4W4_ERR_WORKSPACE;
  unsigned int* status = a4w4::device_status_ptr();
  if (status == nullptr) return A4W4_ERR_LAUNCH;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  return a4w4::launch_gemm(plan, A_bf16, M, K, Wq, Ws, N, C_bf16, plan.ws_bytes > 0 ? scratch : nullptr, st,
                           a4w4::wait_limit_ns(), status, 0, a4w4::ActDump{});
}

}  // extern "C"
