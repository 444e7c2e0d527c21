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
// Sort with the auxiliary gather/scatter arrays ("[HIP] [CK] [FlyDSL] [Kernel]
// Extend MXFP4 GEMM1 replacement to A4W4", Summary: the adaptive MoE auxiliary
// sort).  Same sorted output as the three-launch sort above, plus
// sorted_tokens[slot] (the token of each slot, T for padding) and row_slot[r]
// (the slot of each routed row).  Entries are split into G runs of per_cta
// (one run per CTA, 16 warps, each warp a contiguous sub-run):
//   count  each warp walks its sub-run 32 entries at a time; __match_any_sync
//          groups equal experts and the group's leader adds it to the warp's
//          per-expert count (shared memory, no atomics);
//   scan   per expert: total, padded block count, an exclusive scan over
//          experts gives each expert's first block; block_expert[], the block
//          count and the padding sentinels are written (a warp per expert);
//   place  each warp re-walks its sub-run: slot = expert's first slot + rows
//          of earlier runs + rows of earlier warps + rows earlier in the warp
//          + rank among equal lanes of the step (stable: increasing r).
// Adaptive: up to 2048 routed rows (decode batches) one CTA does all three in
// one launch; beyond, a counting launch whose last CTA to finish (atomic
// ticket, no waiting) runs the scan, then a placing launch (programmatic
// dependent launch: it counts its run again while the first one finishes).
constexpr int kAuxWarps = 16;
constexpr int kAuxThreads = kAuxWarps * 32;
constexpr int kAuxMaxExperts = 4096;
constexpr int kAuxMaxPerCta = 32768;   // keeps every per-warp offset below 2^16
constexpr int kAuxRun = 2048;          // routed rows per CTA (at most one CTA per SM beyond)

struct AuxSmem {
  uint16_t* wcnt;     // [kAuxWarps][E]: counts, then exclusive prefix over warps, then running cursors
  int32_t* start;     // [E]
  int32_t* total;     // [E]
  int32_t* first;     // [E]
  int32_t* scan;      // [kAuxThreads]
};

__device__ __forceinline__ AuxSmem aux_smem(int32_t* sh, int E) {
  AuxSmem a;
  a.wcnt = reinterpret_cast<uint16_t*>(sh);
  a.start = sh + (kAuxWarps * E + 1) / 2;
  a.total = a.start + E;
  a.first = a.total + E;
  a.scan = a.first + E;
  return a;
}

// Per-warp counts of this CTA's run -> exclusive prefix over the warps
// (wcnt), and the run's per-expert totals into hist_row (global) when given,
// else into a.total.
__device__ void aux_count(const int32_t* __restrict__ ids, int r0, int r1, int E, AuxSmem a, int32_t* hist_row) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kAuxWarps * E; i += kAuxThreads) a.wcnt[i] = 0;
  __syncthreads();
  uint16_t* my = a.wcnt + warp * E;
  for (int s = r0; s < r1; s += 32) {
    const int r = s + lane;
    int e = r < r1 ? __ldcg(ids + r) : -1;   // L2: ids may be read before a dependency wait
    const bool ok = e >= 0 && e < E;
    if (!ok) e = -1 - lane;                       // unique key: matches no other lane
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    if (ok && lane == __ffs(peers) - 1) my[e] = static_cast<uint16_t>(my[e] + __popc(peers));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kAuxThreads) {
    int tot = 0;
    for (int w = 0; w < kAuxWarps; ++w) {
      const int v = a.wcnt[w * E + e];
      a.wcnt[w * E + e] = static_cast<uint16_t>(tot);
      tot += v;
    }
    if (hist_row != nullptr) hist_row[e] = tot;
    else a.total[e] = tot;
  }
  __syncthreads();
}

// Scan over experts of the totals in a.total: first block per expert into
// a.first (and `first_out` when not null); block_expert[], *num_blocks and
// the padding sentinels.
__device__ void aux_scan(int E, int bm_log2, int n, int T, AuxSmem a, int32_t* __restrict__ sorted_rows,
                         int32_t* __restrict__ block_expert, int32_t* __restrict__ num_blocks,
                         int32_t* __restrict__ sorted_tokens, int32_t* first_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bm = 1 << bm_log2;
  const int per_t = (E + kAuxThreads - 1) / kAuxThreads;
  const int e0 = min(E, threadIdx.x * per_t), e1 = min(E, e0 + per_t);
  int nb_local = 0;
  for (int e = e0; e < e1; ++e) nb_local += (a.total[e] + bm - 1) >> bm_log2;
  a.scan[threadIdx.x] = nb_local;
  __syncthreads();
  for (int d = 1; d < kAuxThreads; d <<= 1) {
    const int v = threadIdx.x >= d ? a.scan[threadIdx.x - d] : 0;
    __syncthreads();
    a.scan[threadIdx.x] += v;
    __syncthreads();
  }
  int boff = a.scan[threadIdx.x] - nb_local;
  if (threadIdx.x == kAuxThreads - 1) *num_blocks = a.scan[threadIdx.x];
  for (int e = e0; e < e1; ++e) {
    a.first[e] = boff;
    if (first_out != nullptr) first_out[e] = boff;
    boff += (a.total[e] + bm - 1) >> bm_log2;
  }
  __syncthreads();
  // block lists and padding of the experts that have rows: each warp scans 32
  // experts at a time and handles the non-empty ones together (lanes over slots)
  for (int base = warp * 32; base < E; base += kAuxWarps * 32) {
    const int me = base + lane;
    unsigned hit = __ballot_sync(0xFFFFFFFFu, me < E && a.total[me] > 0);
    while (hit) {
      const int e = base + __ffs(hit) - 1;
      hit &= hit - 1;
      const int b0 = a.first[e], tot = a.total[e];
      const int nb_e = (tot + bm - 1) >> bm_log2;
      for (int b = lane; b < nb_e; b += 32) block_expert[b0 + b] = e;
      for (int sl = (b0 << bm_log2) + tot + lane; sl < ((b0 + nb_e) << bm_log2); sl += 32) {
        sorted_rows[sl] = n;                        // sentinel T * topk
        sorted_tokens[sl] = T;
      }
    }
  }
}

// Stable placement of this CTA's run (a.start holds each expert's first slot
// for this run; a.wcnt each warp's prefix).
__device__ void aux_place(const int32_t* __restrict__ ids, int r0, int r1, int E, int topk, AuxSmem a,
                          int32_t* __restrict__ sorted_rows, int32_t* __restrict__ sorted_tokens,
                          int32_t* __restrict__ row_slot) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint16_t* my = a.wcnt + warp * E;
  for (int s = r0; s < r1; s += 32) {
    const int r = s + lane;
    int e = r < r1 ? __ldcg(ids + r) : -1;
    const bool ok = e >= 0 && e < E;
    if (!ok) e = -1 - lane;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int before = ok ? my[e] : 0;
    if (ok) {
      const int slot = a.start[e] + before + rank;
      sorted_rows[slot] = r;
      sorted_tokens[slot] = r / topk;
      row_slot[r] = slot;
    } else if (r < r1) {
      row_slot[r] = -1;                              // expert id outside [0, E): not routed
    }
    __syncwarp();
    if (ok && rank == 0) my[e] = static_cast<uint16_t>(before + __popc(peers));
    __syncwarp();
  }
}

// One warp, up to 32 routed rows (a decode batch of one or two tokens): only
// the experts that were hit are touched.  Lane i holds routed row i; a
// bitonic sort of the keys expert*64 + row over the warp orders the rows by
// expert, then by row; the first lane of each expert's run counts it, a scan
// over those lanes gives each expert's first block.
__global__ void __launch_bounds__(32, 1)
    moe_sort_aux_warp(const int32_t* __restrict__ ids, int n, int topk, int T, int E, int bm,
                      int32_t* __restrict__ sorted_rows, int32_t* __restrict__ block_expert,
                      int32_t* __restrict__ num_blocks, int32_t* __restrict__ sorted_tokens,
                      int32_t* __restrict__ row_slot) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x;
  int e = lane < n ? __ldcg(ids + lane) : -1;
  const bool ok = e >= 0 && e < E;
  if (lane < n && !ok) row_slot[lane] = -1;        // expert id outside [0, E): not routed
  // key: valid rows by (expert, row); everything else sorts last
  unsigned key = ok ? (static_cast<unsigned>(e) << 6) | static_cast<unsigned>(lane) : 0xFFFFFFFFu;
  for (int k = 2; k <= 32; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      const unsigned other = __shfl_xor_sync(0xFFFFFFFFu, key, j);
      const bool up = (lane & k) == 0;
      const bool lower = (lane & j) == 0;
      key = (lower == up) ? min(key, other) : max(key, other);
    }
  }
  const bool valid = key != 0xFFFFFFFFu;
  const int ke = valid ? static_cast<int>(key >> 6) : -1;
  const int kr = static_cast<int>(key & 63u);
  const int prev = __shfl_up_sync(0xFFFFFFFFu, ke, 1);
  const bool head = valid && (lane == 0 || prev != ke);
  const unsigned heads = __ballot_sync(0xFFFFFFFFu, head);
  // run of this lane's expert: [start lane, next head)
  const int run0 = 31 - __clz(heads & ((2u << lane) - 1u));        // last head at or before this lane
  const unsigned later = heads & ~((2u << lane) - 1u);
  const int nvalid = __popc(__ballot_sync(0xFFFFFFFFu, valid));
  const int run1 = later ? __ffs(later) - 1 : nvalid;
  const int cnt = run1 - run0;
  const int nblk = head ? (cnt + bm - 1) / bm : 0;
  int incl = nblk;                                  // inclusive scan of block counts over lanes
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += v;
  }
  const int first = __shfl_sync(0xFFFFFFFFu, incl - nblk, run0);   // the run's first block
  if (lane == 31) *num_blocks = incl;
  if (valid) {
    const int slot = first * bm + (lane - run0);
    sorted_rows[slot] = kr;
    sorted_tokens[slot] = kr / topk;
    row_slot[kr] = slot;
  }
  // block lists and padding, a run at a time, lanes over slots
  unsigned h = heads;
  while (h) {
    const int src = __ffs(h) - 1;
    h &= h - 1;
    const int re = __shfl_sync(0xFFFFFFFFu, ke, src);
    const int rf = __shfl_sync(0xFFFFFFFFu, first, src);
    const int rc = __shfl_sync(0xFFFFFFFFu, cnt, src);
    const int rb = (rc + bm - 1) / bm;
    for (int b = lane; b < rb; b += 32) block_expert[rf + b] = re;
    for (int sl = rf * bm + rc + lane; sl < (rf + rb) * bm; sl += 32) {
      sorted_rows[sl] = n;
      sorted_tokens[sl] = T;
    }
  }
}

// One CTA, all three steps (n <= kAuxRun).
__global__ void __launch_bounds__(kAuxThreads, 1)
    moe_sort_aux_single(const int32_t* __restrict__ ids, int n, int topk, int T, int E, int bm,
                        int32_t* __restrict__ sorted_rows, int32_t* __restrict__ block_expert,
                        int32_t* __restrict__ num_blocks, int32_t* __restrict__ sorted_tokens,
                        int32_t* __restrict__ row_slot) {
  extern __shared__ int32_t aux_sh[];
  griddep_wait();                                    // ids may come from the previous kernel
  griddep_launch_dependents();
  const AuxSmem a = aux_smem(aux_sh, E);
  const int per_warp = (n + kAuxWarps * 32 - 1) / (kAuxWarps * 32) * 32;
  const int warp = threadIdx.x >> 5;
  const int r0 = min(n, warp * per_warp), r1 = min(n, r0 + per_warp);
  aux_count(ids, r0, r1, E, a, nullptr);
  aux_scan(E, 31 - __clz(bm), n, T, a, sorted_rows, block_expert, num_blocks, sorted_tokens, nullptr);
  for (int e = threadIdx.x; e < E; e += kAuxThreads) a.start[e] = a.first[e] * bm;
  __syncthreads();
  aux_place(ids, r0, r1, E, topk, a, sorted_rows, sorted_tokens, row_slot);
}

// Counting launch (G CTAs): each CTA's run totals to hist[c][*]; the last CTA
// to finish (atomic ticket in the workspace, reset by that CTA) runs the scan.
__global__ void __launch_bounds__(kAuxThreads, 1)
    moe_sort_aux_count(const int32_t* __restrict__ ids, int n, int T, int E, int bm, int per_cta,
                       int32_t* __restrict__ sorted_rows, int32_t* __restrict__ block_expert,
                       int32_t* __restrict__ num_blocks, int32_t* __restrict__ sorted_tokens,
                       int32_t* __restrict__ hist, int32_t* __restrict__ first_out, unsigned int* ticket) {
  extern __shared__ int32_t aux_sh[];
  __shared__ int last;
  griddep_wait();
  griddep_launch_dependents();                       // the placing launch may start counting now
  const AuxSmem a = aux_smem(aux_sh, E);
  const int G = gridDim.x, c = blockIdx.x, warp = threadIdx.x >> 5;
  const int per_warp = per_cta / kAuxWarps;
  const int r0 = min(n, c * per_cta + warp * per_warp), r1 = min(n, r0 + per_warp);
  aux_count(ids, r0, r1, E, a, hist + static_cast<long long>(c) * E);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    last = atomicAdd(ticket, 1u) == static_cast<unsigned int>(G - 1);
    if (last) *ticket = 0u;                          // ready for the next call
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int e = threadIdx.x; e < E; e += kAuxThreads) {
    int tot = 0;
    for (int g = 0; g < G; ++g) tot += __ldcg(hist + static_cast<long long>(g) * E + e);
    a.total[e] = tot;
  }
  __syncthreads();
  aux_scan(E, 31 - __clz(bm), n, T, a, sorted_rows, block_expert, num_blocks, sorted_tokens, first_out);
}

// Placing launch: counts its run again (the ids only) before waiting for the
// counting launch, then reads the histograms and the experts' first blocks.
__global__ void __launch_bounds__(kAuxThreads, 1)
    moe_sort_aux_place(const int32_t* __restrict__ ids, int n, int topk, int E, int bm, int per_cta,
                       int32_t* __restrict__ sorted_rows, int32_t* __restrict__ sorted_tokens,
                       int32_t* __restrict__ row_slot, const int32_t* __restrict__ hist,
                       const int32_t* __restrict__ first_blk) {
  extern __shared__ int32_t aux_sh[];
  const AuxSmem a = aux_smem(aux_sh, E);
  const int c = blockIdx.x, warp = threadIdx.x >> 5;
  const int per_warp = per_cta / kAuxWarps;
  const int r0 = min(n, c * per_cta + warp * per_warp), r1 = min(n, r0 + per_warp);
  aux_count(ids, r0, r1, E, a, nullptr);             // ids are inputs of the sort, not of the first launch
  griddep_wait();                                    // the counting launch has completed
  for (int e = threadIdx.x; e < E; e += kAuxThreads) {
    int before = 0;
    for (int g = 0; g < c; ++g) before += __ldcg(hist + static_cast<long long>(g) * E + e);
    a.start[e] = __ldcg(first_blk + e) * bm + before;
  }
  __syncthreads();
  aux_place(ids, r0, r1, E, topk, a, sorted_rows, sorted_tokens, row_slot);
}

static long long aux_ctas(long long n, int sms) {
  long long g = (n + kAuxRun - 1) / kAuxRun;
  if (g > sms) g = sms;
  return g < 1 ? 1 : g;
}

size_t moe_sort_aux_ws_bytes(int T, int topk, int E, int sms) {
  const long long g = aux_ctas(static_cast<long long>(T) * topk, sms);
  return static_cast<size_t>(g + 1) * E * sizeof(int32_t) + 256;   // histograms, first blocks, ticket
}

int launch_moe_sort_aux(const int32_t* ids, int T, int topk, int E, int bm, int32_t* sorted_rows,
                        int32_t* block_expert, int32_t* num_blocks, int32_t* sorted_tokens, int32_t* row_slot,
                        void* ws, cudaStream_t st, int sms, unsigned long long wait_ns, unsigned int* status) {
  (void)wait_ns;
  (void)status;
  if (E > kAuxMaxExperts) return -1;
  const long long n = static_cast<long long>(T) * topk;
  const long long g = aux_ctas(n, sms);
  long long per = (n + g - 1) / g;                   // a multiple of the 16 warps x 32 lanes
  per = (per + kAuxThreads - 1) / kAuxThreads * kAuxThreads;
  if (per > kAuxMaxPerCta) return -1;
  const size_t shm = static_cast<size_t>((kAuxWarps * E + 1) / 2 + 3 * E + kAuxThreads) * sizeof(int32_t);
  static std::atomic<unsigned long long> attr_devs{0};
  if (ensure_func_attrs(attr_devs, [&] {
        const int max_shm = ((kAuxWarps * kAuxMaxExperts + 1) / 2 + 3 * kAuxMaxExperts + kAuxThreads) * 4;
        return cudaFuncSetAttribute(moe_sort_aux_single, cudaFuncAttributeMaxDynamicSharedMemorySize, max_shm) ==
                   cudaSuccess &&
               cudaFuncSetAttribute(moe_sort_aux_count, cudaFuncAttributeMaxDynamicSharedMemorySize, max_shm) ==
                   cudaSuccess &&
               cudaFuncSetAttribute(moe_sort_aux_place, cudaFuncAttributeMaxDynamicSharedMemorySize, max_shm) ==
                   cudaSuccess;
      }) != 0)
    return -4;
  auto launch = [&](auto kern, auto... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(g), 1, 1);
    cfg.blockDim = dim3(kAuxThreads, 1, 1);
    cfg.dynamicSmemBytes = shm;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...) == cudaSuccess ? 0 : -4;
  };
  int rc;
  if (n <= 32) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(32, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    rc = cudaLaunchKernelEx(&cfg, moe_sort_aux_warp, ids, static_cast<int>(n), topk, T, E, bm, sorted_rows,
                            block_expert, num_blocks, sorted_tokens, row_slot) == cudaSuccess ? 0 : -4;
  } else if (g == 1) {
    rc = launch(moe_sort_aux_single, ids, static_cast<int>(n), topk, T, E, bm, sorted_rows, block_expert, num_blocks,
                sorted_tokens, row_slot);
  } else {
    int32_t* hist = static_cast<int32_t*>(ws);
    int32_t* first_blk = hist + g * E;
    unsigned int* ticket = reinterpret_cast<unsigned int*>(first_blk + E);
    rc = launch(moe_sort_aux_count, ids, static_cast<int>(n), T, E, bm, static_cast<int>(per), sorted_rows,
                block_expert, num_blocks, sorted_tokens, hist, first_blk, ticket);
    if (rc == 0)
      rc = launch(moe_sort_aux_place, ids, static_cast<int>(n), topk, E, bm, static_cast<int>(per), sorted_rows,
                  sorted_tokens, row_slot, static_cast<const int32_t*>(hist), static_cast<const int32_t*>(first_blk));
  }
  if (rc != 0) return rc;
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
