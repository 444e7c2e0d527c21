// moe2.cu -- grouped MoE GEMM2 (down projection) over GEMM1's sorted-slot
// MXFP4 tiles: per routed row, the top-k weighted fp32 product row.
//
// "[HIP] [CK] [FlyDSL] [Kernel] Extend MXFP4 GEMM1 replacement to A4W4",
// Summary (stage-2 paths that consume stage 1's layout) and GEMM2 scope.
//
// One CTA per (sorted block of 128 slots, run of output-column tiles): the
// block's activation tiles (K = I, a few 256-wide atoms) are copied into
// shared memory once; the expert's W2 tiles of the run (256 output rows x
// 256 K, one 32 KB + 2 KB copy each) stream through a ring.  A block routed
// to one expert usually holds few valid rows, so a CTA walks many tiles with
// its operand rows resident instead of reloading them per tile.
//   warp 0      copies the activation tiles, then the weight ring;
//   warp 1      allocates TMEM, copies the activation scales to TMEM once and
//               each stage's weight scales, issues four
//               tcgen05.mma.kind::mxf4.block_scale (M = 128, N = 256, K = 64)
//               per K tile, commits the tile's accumulator to the epilogue;
//   warps 2-5   per tile: wait for the accumulator, then per 64 columns
//               tcgen05.ld, scale each valid row by its routing weight and
//               store it from registers (row `routed row` of
//               the [T*topk, D] fp32 partial buffer); then hand the
//               accumulator back (the next tile's weights keep streaming
//               meanwhile; only its MMAs wait).
#include <atomic>

#include "device.cuh"
#include "launch.h"

namespace a4w4 {

struct Moe2Args {
  const uint8_t* Aq;         // GEMM1 tiles: atom b*KT + kt, 16 KB of codes each
  const uint8_t* As;         // and 1 KB of scales each
  const uint8_t* Wq;         // W2, dense preshuffled layout of [E*D, I]
  const uint8_t* Ws;
  long long expert_code_bytes, expert_sf_bytes;
  const int32_t* sorted_rows;
  const int32_t* block_expert;
  const int32_t* num_blocks;
  const float* topk_w;
  float* partial;            // [T*topk, D] fp32
  int routed_rows, D, KT, E, tiles_per_cta;
  unsigned long long wait_ns;
  unsigned int* status;
};

constexpr int kM2Stages = 4;
constexpr int kM2MaxKT = 4;                              // I <= 1024
constexpr int kM2Threads = 192;
constexpr int kM2OffA = 0;                               // activation codes, KT x 16 KB
constexpr int kM2OffAsf = kM2OffA + kM2MaxKT * 16384;    // activation scales, KT x 1 KB
constexpr int kM2OffW = kM2OffAsf + kM2MaxKT * 1024;     // weight ring, 32 KB per stage
constexpr int kM2OffWsf = kM2OffW + kM2Stages * 32768;   // weight scales, 2 KB per stage
constexpr int kM2OffBar = kM2OffWsf + kM2Stages * 2048;
constexpr int kM2OffMisc = kM2OffBar + (2 * kM2Stages + 3) * 8;
constexpr int kM2Smem = kM2OffMisc + 32 + 1024;
constexpr int kM2TmemCols = 512;                         // 256 accumulator + scale columns
constexpr int kM2SfaCol = 256;                           // activation scales: 8 per K tile
constexpr int kM2SfbCol = kM2SfaCol + 8 * kM2MaxKT;      // weight scales: 16 per stage
static_assert(kM2SfbCol + 16 * kM2Stages <= kM2TmemCols, "TMEM budget");
static_assert(kM2Smem <= 232448, "shared memory");

__global__ void __launch_bounds__(kM2Threads, 1) a4w4_moe2_kernel(const Moe2Args p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = blockIdx.y;

  griddep_wait();                                  // GEMM1 and the sort have completed
  griddep_launch_dependents();
  if (blk >= *p.num_blocks) return;
  const int expert = p.block_expert[blk];
  if (expert < 0 || expert >= p.E) return;
  const int wt_total = p.D / 256;
  const int wt0 = blockIdx.x * p.tiles_per_cta;
  const int wt1 = min(wt_total, wt0 + p.tiles_per_cta);
  if (wt0 >= wt1) return;
  const int ntile = wt1 - wt0, KT = p.KT, nstage = ntile * KT;
  const unsigned long long drain_ns = p.wait_ns > 100000000ull ? p.wait_ns : 100000000ull;

  const uint32_t bar0 = base + kM2OffBar;
  auto w_full = [&](int s) { return bar0 + 8u * s; };
  auto w_empty = [&](int s) { return bar0 + 8u * (kM2Stages + s); };
  const uint32_t a_full = bar0 + 8u * (2 * kM2Stages);
  const uint32_t acc_full = a_full + 8u;
  const uint32_t acc_empty = acc_full + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kM2OffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kM2OffMisc + 8);
  volatile int* never = reinterpret_cast<volatile int*>(smem + kM2OffMisc + 16);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kM2Stages; ++s) {
      mbar_init(w_full(s), 1);
      mbar_init(w_empty(s), 1);
    }
    mbar_init(a_full, 1);
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 128);
    *abort_flag = 0;
    *never = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const uint8_t* wq_e = p.Wq + static_cast<long long>(expert) * p.expert_code_bytes;
  const uint8_t* ws_e = p.Ws + static_cast<long long>(expert) * p.expert_sf_bytes;
  uint32_t tmem = 0;

  if (warp == 0) {
    // ---------------- copies ----------------
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();   // each W2 tile is read by this CTA only
      const uint64_t pol_a = policy_evict_first();
      mbar_arrive_expect_tx(a_full, KT * (16384 + 1024));
      bulk_g2s(base + kM2OffA, p.Aq + static_cast<long long>(blk) * KT * 16384, KT * 16384, a_full, pol_a);
      bulk_g2s(base + kM2OffAsf, p.As + static_cast<long long>(blk) * KT * 1024, KT * 1024, a_full, pol_a);
      int i = 0;
      for (; i < nstage; ++i) {
        const int s = i % kM2Stages;
        if (i >= kM2Stages && !mbar_wait(w_empty(s), ((i / kM2Stages) & 1) ^ 1u, abort_flag, p.wait_ns, p.status))
          break;
        const int wt = wt0 + i / KT, kt = i % KT;
        const long long atom = weight_atom(2 * wt, kt, KT);   // the tile's two 128-row atoms, adjacent
        mbar_arrive_expect_tx(w_full(s), 32768 + 2048);
        bulk_g2s(base + kM2OffW + s * 32768, wq_e + atom * 16384, 32768, w_full(s), pol_w);
        bulk_g2s(base + kM2OffWsf + s * 2048, ws_e + atom * 1024, 2048, w_full(s), pol_w);
      }
      // every copy issued lands before the shared memory is released
      mbar_wait(a_full, 0, never, drain_ns, p.status);
      for (int j = (i > kM2Stages ? i - kM2Stages : 0); j < i; ++j)
        mbar_wait(w_full(j % kM2Stages), (j / kM2Stages) & 1u, never, drain_ns, p.status);
    }
  } else if (warp == 1) {
    // ---------------- TMEM + MMA ----------------
    tmem_alloc(smem_u32(tmem_slot), kM2TmemCols);
    tc_fence_before();
    __syncwarp();
    tc_fence_after();
    tmem = *tmem_slot;
    named_bar_arrive(2, 32 + 128);                 // publish the TMEM address to the epilogue
    if (lane == 0) {
      int issued_tiles = 0;
      if (mbar_wait(a_full, 0, abort_flag, p.wait_ns, p.status)) {
        tc_fence_after();
        const uint64_t asfd = sdesc_sf(base + kM2OffAsf), wsfd = sdesc_sf(base + kM2OffWsf);
        for (int kt = 0; kt < KT; ++kt)
          for (int ka = 0; ka < 2; ++ka)
            tmem_copy_sf_desc(tmem + kM2SfaCol + kt * 8 + ka * 4, asfd + ((kt * 1024 + ka * 512) >> 4));
        const uint64_t adesc0 = sdesc_sw128(base + kM2OffA), wdesc0 = sdesc_sw128(base + kM2OffW);
        const uint32_t idesc0 = idesc_mxf4(256, 0, 0), idesc2 = idesc_mxf4(256, 2, 2);
        bool ok = true;
        for (int j = 0; j < ntile && ok; ++j) {
          // the epilogue has read the previous tile's accumulator
          if (j > 0 && !mbar_wait(acc_empty, (j - 1) & 1u, abort_flag, p.wait_ns, p.status)) break;
          tc_fence_after();
          for (int kt = 0; kt < KT; ++kt) {
            const int i = j * KT + kt, s = i % kM2Stages;
            if (!mbar_wait(w_full(s), (i / kM2Stages) & 1u, abort_flag, p.wait_ns, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sfb = tmem + kM2SfbCol + s * 16;
            for (int ka = 0; ka < 2; ++ka)
              for (int a = 0; a < 2; ++a)
                tmem_copy_sf_desc(sfb + ka * 8 + a * 4, wsfd + ((s * 2048 + a * 1024 + ka * 512) >> 4));
            const uint64_t ad = adesc0 + ((kt * 16384) >> 4), wd = wdesc0 + ((s * 32768) >> 4);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const int ka = ks >> 1;
              mma_mxf4(tmem, ad + ks * 2, wd + ks * 2, (ks & 1) ? idesc2 : idesc0, tmem + kM2SfaCol + kt * 8 + ka * 4,
                       sfb + ka * 8, (kt > 0 || ks > 0) ? 1u : 0u);
            }
            mma_commit(w_empty(s));
          }
          if (!ok) break;
          mma_commit(acc_full);
          issued_tiles = j + 1;
        }
      }
      // TMEM is not released while MMAs may run: wait for the last commit
      if (issued_tiles > 0) mbar_wait(acc_full, (issued_tiles - 1) & 1u, never, drain_ns, p.status);
    }
  } else {
    // ---------------- epilogue (warps 2-5, one TMEM lane quadrant each) ----------------
    named_bar_sync(2, 32 + 128);
    tc_fence_after();
    tmem = *tmem_slot;
    const int q = warp & 3, lrow = q * 32 + lane;
    const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const int entry = p.sorted_rows[blk * 128 + lrow];
    const bool valid = entry >= 0 && entry < p.routed_rows;
    const float wgt = valid ? __ldg(p.topk_w + entry) : 0.f;
    float* out_row = p.partial + static_cast<long long>(valid ? entry : 0) * p.D;
    for (int j = 0; j < ntile; ++j) {
      // every thread waits itself (a bounded wait; no barrier that one
      // thread's early exit could leave waiting)
      if (!mbar_wait(acc_full, j & 1u, abort_flag, p.wait_ns, p.status)) break;
      tc_fence_after();
      const int wt = wt0 + j;
#pragma unroll 1
      for (int c0 = 0; c0 < 256; c0 += 64) {
        float v[64];
        tmem_ld64(tq + c0, v);
        if (valid) {
          float4* dst = reinterpret_cast<float4*>(out_row + wt * 256 + c0);
#pragma unroll
          for (int u = 0; u < 16; ++u)
            __stcs(dst + u, make_float4(wgt * v[4 * u], wgt * v[4 * u + 1], wgt * v[4 * u + 2], wgt * v[4 * u + 3]));
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kM2TmemCols);
  }
}

int launch_moe_gemm2_resident(const void* Aq, const void* As, int T, int I, const int32_t* sorted_rows,
                     const int32_t* block_expert, const int32_t* num_blocks, int max_blocks, int topk,
                     const float* topk_w, const void* W2q, const void* W2s, int E, int D, float* partial,
                     cudaStream_t st, unsigned long long wait_ns, unsigned int* status, int sms) {
  if (max_blocks <= 0) return 0;
  Moe2Args a{};
  a.Aq = static_cast<const uint8_t*>(Aq);
  a.As = static_cast<const uint8_t*>(As);
  a.Wq = static_cast<const uint8_t*>(W2q);
  a.Ws = static_cast<const uint8_t*>(W2s);
  a.KT = (I + 255) / 256;
  if (a.KT > kM2MaxKT) return -1;
  const long long kp = static_cast<long long>(a.KT) * 256;
  a.expert_code_bytes = static_cast<long long>(D) * kp / 2;
  a.expert_sf_bytes = static_cast<long long>(D) * kp / 32;
  a.sorted_rows = sorted_rows;
  a.block_expert = block_expert;
  a.num_blocks = num_blocks;
  a.topk_w = topk_w;
  a.partial = partial;
  a.routed_rows = T * topk;
  a.D = D;
  a.E = E;
  a.wait_ns = wait_ns;
  a.status = status;
  // Output-column tiles per CTA: all of them once the blocks alone give two
  // CTAs per SM; fewer (more CTAs per block) for small batches.
  const int wt_total = D / 256;
  const long long want = 2ll * sms;
  int per = static_cast<int>((static_cast<long long>(wt_total) * max_blocks + want - 1) / want);
  if (per < 1) per = 1;
  if (per > wt_total) per = wt_total;
  a.tiles_per_cta = per;
  const int groups = (wt_total + per - 1) / per;
  static std::atomic<unsigned long long> attr_devs{0};
  if (ensure_func_attrs(attr_devs, [&] {
        return cudaFuncSetAttribute(a4w4_moe2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kM2Smem) ==
               cudaSuccess;
      }) != 0)
    return -4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(groups), static_cast<unsigned>(max_blocks), 1);
  cfg.blockDim = dim3(kM2Threads, 1, 1);
  cfg.dynamicSmemBytes = kM2Smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, a4w4_moe2_kernel, a) != cudaSuccess) return -4;
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace a4w4
