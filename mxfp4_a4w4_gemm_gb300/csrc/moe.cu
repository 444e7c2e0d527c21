// moe.cu -- routed-row sort for the grouped MoE GEMM1.
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

}  // namespace a4w4
