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
