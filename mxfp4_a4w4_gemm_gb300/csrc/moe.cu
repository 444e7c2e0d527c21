// moe.cu -- routed-row sort for the grouped MoE GEMMs, and GEMM2's per-token
// reduction of the top-k weighted rows.
//
// "[HIP] [CK] [FlyDSL] [Kernel] Extend MXFP4 GEMM1 replacement to A4W4",
// Summary: GEMM1 consumes token->expert rows grouped per expert by an auxiliary
// sort, in blocks of block_m rows.  Output order (deterministic): experts in
// increasing order, the rows routed to each expert in increasing routed-row
// index r = t*topk + k, each expert's list padded with the sentinel T*topk to a
// multiple of block_m.
//
// Three launches, no host synchronisation:
//   1. per 2048-entry chunk, a per-expert histogram (shared-memory atomics);
//   2. one CTA: per-expert totals, padded block counts, an exclusive scan over
//      experts (block offsets, block_expert[], num_blocks, sentinel padding)
//      and, in place, each chunk's starting position inside each expert;
//   3. per chunk, one warp walks the entries in order; __match_any_sync gives
//      each entry its rank among equal experts of the same 32-entry step.
#include <atomic>

#include "device.cuh"
#include "launch.h"

namespace a4w4 {

constexpr int kSortChunk = 2048;
constexpr int kSortMaxExperts = 8192;

__global__ void __launch_bounds__(256) moe_hist_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                       int32_t* __restrict__ hist) {
  extern __shared__ int32_t sh[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  const int c0 = blockIdx.x * kSortChunk;
  const int c1 = min(n, c0 + kSortChunk);
  for (int i = c0 + threadIdx.x; i < c1; i += blockDim.x) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(sh + e, 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<long long>(blockIdx.x) * E + e] = sh[e];
}

__global__ void __launch_bounds__(1024) moe_scan_kernel(int32_t* __restrict__ hist, int nchunks, int E, int bm,
                                                        int sentinel, int32_t* __restrict__ sorted_rows,
                                                        int32_t* __restrict__ block_expert,
                                                        int32_t* __restrict__ num_blocks) {
  __shared__ int32_t warp_sums[32];
  const int per = (E + 1023) / 1024;
  const int e0 = threadIdx.x * per;
  int nb_local = 0;
  for (int e = e0; e < min(E, e0 + per); ++e) {
    int tot = 0;
    for (int c = 0; c < nchunks; ++c) tot += hist[static_cast<long long>(c) * E + e];
    nb_local += (tot + bm - 1) / bm;
  }
  // exclusive scan of nb_local over the 1024 threads (in thread order = expert order)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = nb_local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, w, d);
      if (lane >= d) w += v;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  int boff = incl - nb_local + (warp > 0 ? warp_sums[warp - 1] : 0);
  if (threadIdx.x == 1023) *num_blocks = boff + nb_local;
  for (int e = e0; e < min(E, e0 + per); ++e) {
    int pos = boff * bm;
    for (int c = 0; c < nchunks; ++c) {
      const long long h = static_cast<long long>(c) * E + e;
      const int cnt = hist[h];
      hist[h] = pos;  // where chunk c's rows of expert e start
      pos += cnt;
    }
    const int tot = pos - boff * bm;
    const int nb = (tot + bm - 1) / bm;
    for (int b = 0; b < nb; ++b) block_expert[boff + b] = e;
    for (int q = pos; q < (boff + nb) * bm; ++q) sorted_rows[q] = sentinel;
    boff += nb;
  }
}

__global__ void __launch_bounds__(32) moe_place_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                       const int32_t* __restrict__ chunk_base,
                                                       int32_t* __restrict__ sorted_rows) {
  extern __shared__ int32_t cnt[];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  const int c0 = blockIdx.x * kSortChunk;
  const int c1 = min(n, c0 + kSortChunk);
  const int32_t* base = chunk_base + static_cast<long long>(blockIdx.x) * E;
  for (int s = c0; s < c1; s += 32) {
    const int i = s + lane;
    int e = (i < c1) ? ids[i] : -1;
    const bool ok = e >= 0 && e < E;
    if (!ok) e = -1 - lane;                   // unique key: matches no other lane
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int before = ok ? cnt[e] : 0;
    if (ok) sorted_rows[base[e] + before + rank] = i;
    __syncwarp();
    if (ok && rank == 0) cnt[e] = before + __popc(peers);
    __syncwarp();
  }
}

size_t moe_sort_ws_bytes(int T, int topk, int E) {
  const long long n = static_cast<long long>(T) * topk;
  const long long nchunks = (n + kSortChunk - 1) / kSortChunk;
  return static_cast<size_t>(nchunks > 0 ? nchunks : 1) * E * sizeof(int32_t);
}

int launch_moe_sort(const int32_t* ids, int T, int topk, int E, int bm, int32_t* sorted_rows,
                    int32_t* block_expert, int32_t* num_blocks, void* ws, cudaStream_t st) {
  if (E > kSortMaxExperts) return -1;
  const int n = T * topk;
  const int nchunks = (n + kSortChunk - 1) / kSortChunk;
  int32_t* hist = static_cast<int32_t*>(ws);
  const size_t shm = static_cast<size_t>(E) * sizeof(int32_t);
  moe_hist_kernel<<<nchunks, 256, shm, st>>>(ids, n, E, hist);
  moe_scan_kernel<<<1, 1024, 0, st>>>(hist, nchunks, E, bm, n, sorted_rows, block_expert, num_blocks);
  moe_place_kernel<<<nchunks, 32, shm, st>>>(ids, n, E, hist, sorted_rows);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// ---------------------------------------------------------------------------
// Single-launch sort with the auxiliary gather/scatter arrays ("[HIP] [CK]
// [FlyDSL] [Kernel] Extend MXFP4 GEMM1 replacement to A4W4", Summary: the
// adaptive MoE auxiliary sort).  Same sorted output as the three-launch sort
// above, plus sorted_tokens[slot] (the token of each slot, T for padding) and
// row_slot[r] (the slot of each routed row).  One cooperative launch of G CTAs
// (1 for up to 2048 routed rows; at most one per SM), 16 warps each:
//   1. each warp walks its contiguous run of entries 32 at a time;
//      __match_any_sync groups equal experts and the leader adds the group to
//      the warp's own per-expert count (shared memory, no atomics); the CTA
//      publishes its per-expert totals;
//   2. grid barrier (G > 1): an arrival counter and a generation word in the
//      workspace, bounded spin;
//   3. every CTA reads all G histograms: per expert its total, the rows of
//      CTAs before it, the padded block count, and an exclusive scan over
//      experts gives each expert's first slot; experts e = c (mod G) get their
//      block_expert entries and padding sentinels from CTA c;
//   4. each warp re-walks its run: slot = expert start + rows of earlier CTAs
//      + rows of earlier warps + rows earlier in this warp + rank among equal
//      lanes of the step (stable, increasing r within each expert).
constexpr int kAuxWarps = 16;
constexpr int kAuxThreads = kAuxWarps * 32;
constexpr int kAuxMaxExperts = 4096;
constexpr int kAuxMaxPerCta = 32768;   // keeps every per-warp offset below 2^16

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__global__ void __launch_bounds__(kAuxThreads, 1)
    moe_sort_aux_kernel(const int32_t* __restrict__ ids, int n, int topk, int T, int E, int bm, int per_cta,
                        int32_t* __restrict__ sorted_rows, int32_t* __restrict__ block_expert,
                        int32_t* __restrict__ num_blocks, int32_t* __restrict__ sorted_tokens,
                        int32_t* __restrict__ row_slot, int32_t* __restrict__ hist, unsigned int* bar,
                        unsigned long long wait_ns, unsigned int* status) {
  extern __shared__ int32_t aux_sh[];
  // [kAuxWarps][E] per-warp counts, then each warp's running offset within
  // the CTA (both <= per_cta <= kAuxMaxPerCta, so 16 bits suffice)
  uint16_t* wcnt = reinterpret_cast<uint16_t*>(aux_sh);
  int32_t* start = aux_sh + (kAuxWarps * E + 1) / 2;   // [E] first slot of the expert's rows from this CTA
  int32_t* total = start + E;                          // [E] rows routed to the expert
  int32_t* first_blk = total + E;                      // [E] the expert's first block
  int32_t* scan_tmp = first_blk + E;                   // [kAuxThreads]
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  for (int i = threadIdx.x; i < kAuxWarps * E; i += kAuxThreads) wcnt[i] = 0;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  const int per_warp = per_cta / kAuxWarps;
  const int r0 = c * per_cta + warp * per_warp;
  const int r1 = min(n, r0 + per_warp);
  uint16_t* my = wcnt + warp * E;
  // 1. per-warp counts; the CTA's totals to global memory
  for (int s = r0; s < r1; s += 32) {
    const int r = s + lane;
    int e = r < r1 ? ids[r] : -1;
    const bool ok = e >= 0 && e < E;
    if (!ok) e = -1 - lane;                       // unique key: matches no other lane
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    if (ok && lane == __ffs(peers) - 1) my[e] = static_cast<uint16_t>(my[e] + __popc(peers));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kAuxThreads) {
    int tot = 0;
    for (int w = 0; w < kAuxWarps; ++w) {         // counts -> exclusive prefix over the warps
      const int v = wcnt[w * E + e];
      wcnt[w * E + e] = static_cast<uint16_t>(tot);
      tot += v;
    }
    hist[static_cast<long long>(c) * E + e] = tot;
  }
  // 2. grid barrier (one CTA: a block barrier suffices)
  __syncthreads();
  if (G > 1) {
    if (threadIdx.x == 0) {
      const unsigned int gen = ld_acquire_u32(bar + 1);
      __threadfence();
      if (atomicAdd(bar, 1u) == static_cast<unsigned int>(G - 1)) {
        bar[0] = 0u;
        __threadfence();
        atomicAdd(bar + 1, 1u);                   // release the others
      } else {
        const uint64_t t0 = global_timer_ns();
        while (ld_acquire_u32(bar + 1) == gen) {
          if (global_timer_ns() - t0 > wait_ns) {
            atomicOr(status, kStatusTimeout);
            abort_flag = 1;
            break;
          }
        }
      }
    }
    __syncthreads();
    if (abort_flag) return;
  }
  // 3. per expert: total, rows of earlier CTAs, padded blocks; exclusive scan
  //    of the block counts over experts (thread order = expert order)
  const int per_t = (E + kAuxThreads - 1) / kAuxThreads;
  const int e0 = min(E, threadIdx.x * per_t), e1 = min(E, e0 + per_t);
  int nb_local = 0;
  for (int e = e0; e < e1; ++e) {
    int tot = 0, before = 0;
    for (int g = 0; g < G; ++g) {
      const int v = __ldcg(hist + static_cast<long long>(g) * E + e);
      if (g < c) before += v;
      tot += v;
    }
    start[e] = before;
    total[e] = tot;
    nb_local += (tot + bm - 1) / bm;
  }
  scan_tmp[threadIdx.x] = nb_local;
  __syncthreads();
  for (int d = 1; d < kAuxThreads; d <<= 1) {
    const int v = threadIdx.x >= d ? scan_tmp[threadIdx.x - d] : 0;
    __syncthreads();
    scan_tmp[threadIdx.x] += v;
    __syncthreads();
  }
  int boff = scan_tmp[threadIdx.x] - nb_local;    // first block of expert e0
  if (c == 0 && threadIdx.x == kAuxThreads - 1) *num_blocks = scan_tmp[threadIdx.x];
  for (int e = e0; e < e1; ++e) {
    first_blk[e] = boff;
    start[e] += boff * bm;
    boff += (total[e] + bm - 1) / bm;
  }
  __syncthreads();
  // experts e = c (mod G): block list and padding sentinels, each expert's
  // range written by a warp of this CTA (lanes over consecutive slots)
  for (int e = c + warp * G; e < E; e += kAuxWarps * G) {
    const int b0 = first_blk[e], tot = total[e];
    const int nb_e = (tot + bm - 1) / bm;
    for (int b = lane; b < nb_e; b += 32) block_expert[b0 + b] = e;
    for (int sl = b0 * bm + tot + lane; sl < (b0 + nb_e) * bm; sl += 32) {
      sorted_rows[sl] = n;                         // sentinel T * topk
      sorted_tokens[sl] = T;
    }
  }
  // 4. place, stable: increasing r within each expert
  for (int s = r0; s < r1; s += 32) {
    const int r = s + lane;
    int e = r < r1 ? ids[r] : -1;
    const bool ok = e >= 0 && e < E;
    if (!ok) e = -1 - lane;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int before = ok ? my[e] : 0;
    if (ok) {
      const int slot = start[e] + before + rank;
      sorted_rows[slot] = r;
      sorted_tokens[slot] = r / topk;
      row_slot[r] = slot;
    } else if (r < r1) {
      row_slot[r] = -1;                            // expert id outside [0, E): not routed
    }
    __syncwarp();
    if (ok && rank == 0) my[e] = static_cast<uint16_t>(before + __popc(peers));
    __syncwarp();
  }
}

// CTAs of the aux sort: one per 2048 routed rows, at most one per SM.
static long long aux_ctas(long long n, int sms) {
  long long g = (n + 2047) / 2048;
  if (g > sms) g = sms;
  return g < 1 ? 1 : g;
}

size_t moe_sort_aux_ws_bytes(int T, int topk, int E, int sms) {
  return static_cast<size_t>(aux_ctas(static_cast<long long>(T) * topk, sms)) * E * sizeof(int32_t) + 256;
}

int launch_moe_sort_aux(const int32_t* ids, int T, int topk, int E, int bm, int32_t* sorted_rows,
                        int32_t* block_expert, int32_t* num_blocks, int32_t* sorted_tokens, int32_t* row_slot,
                        void* ws, cudaStream_t st, int sms, unsigned long long wait_ns, unsigned int* status) {
  if (E > kAuxMaxExperts) return -1;
  const long long n = static_cast<long long>(T) * topk;
  const long long g = aux_ctas(n, sms);
  // entries per CTA: a multiple of the 16 warps x 32 lanes
  long long per = (n + g - 1) / g;
  per = (per + kAuxThreads - 1) / kAuxThreads * kAuxThreads;
  if (per > kAuxMaxPerCta) return -1;
  const size_t hist_bytes = static_cast<size_t>(g) * E * sizeof(int32_t);
  unsigned int* bar = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + hist_bytes);
  const size_t shm = static_cast<size_t>((kAuxWarps * E + 1) / 2 + 3 * E + kAuxThreads) * sizeof(int32_t);
  static std::atomic<unsigned long long> attr_devs{0};
  if (ensure_func_attrs(attr_devs, [&] {
        const int max_shm = ((kAuxWarps * kAuxMaxExperts + 1) / 2 + 3 * kAuxMaxExperts + kAuxThreads) * 4;
        return cudaFuncSetAttribute(moe_sort_aux_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_shm) ==
               cudaSuccess;
      }) != 0)
    return -4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(g), 1, 1);
  cfg.blockDim = dim3(kAuxThreads, 1, 1);
  cfg.dynamicSmemBytes = shm;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;      // every CTA resident: the grid barrier cannot stall
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, moe_sort_aux_kernel, ids, static_cast<int>(n), topk, T, E, bm, static_cast<int>(per),
                         sorted_rows, block_expert, num_blocks, sorted_tokens, row_slot,
                         static_cast<int32_t*>(ws), bar, wait_ns, status) != cudaSuccess)
    return -4;
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// GEMM2's last step ("[HIP] [CK] [FlyDSL] [Kernel] Extend MXFP4 GEMM1
// replacement to A4W4", GEMM2 scope; the down projection's rows of one token
// are summed): Y[t, n] = sum_{k < topk} partial[t*topk + k, n], added in k
// order in fp32 (bitwise deterministic), rounded to BF16.  One thread per 8
// consecutive columns of a token: two 16-byte loads per routed row, one
// 16-byte store.  HBM-bound: 4*topk bytes read and 2 written per output.
__global__ void __launch_bounds__(256) moe_sum_kernel(const float4* __restrict__ part, int T, int topk, int D,
                                                      uint4* __restrict__ y) {
  griddep_wait();                 // the GEMM2 that wrote `part` has completed
  griddep_launch_dependents();
  const int g8 = D / 8;
  const long long items = static_cast<long long>(T) * g8;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < items; i += stride) {
    const long long t = i / g8;
    const int c = static_cast<int>(i - t * g8);
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const float4* src = part + (t * topk) * (D / 4) + 2 * c;
    for (int k = 0; k < topk; ++k) {
      const float4 u = __ldcs(src), v = __ldcs(src + 1);
      a[0] += u.x; a[1] += u.y; a[2] += u.z; a[3] += u.w;
      a[4] += v.x; a[5] += v.y; a[6] += v.z; a[7] += v.w;
      src += D / 4;
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(a[2 * j], a[2 * j + 1]);
      o[j] = *reinterpret_cast<const uint32_t*>(&b);
    }
    y[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

int launch_moe_sum(const float* partial, int T, int topk, int D, void* Y, cudaStream_t st, int sms) {
  const long long items = static_cast<long long>(T) * (D / 8);
  long long grid = (items + 255) / 256;
  if (grid > static_cast<long long>(sms) * 8) grid = static_cast<long long>(sms) * 8;
  if (grid < 1) grid = 1;
  return launch_pdl(moe_sum_kernel, static_cast<int>(grid), 256, st, reinterpret_cast<const float4*>(partial), T,
                    topk, D, static_cast<uint4*>(Y));
}

}  // namespace a4w4
