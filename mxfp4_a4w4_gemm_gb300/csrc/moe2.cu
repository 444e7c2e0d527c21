// moe2.cu -- grouped MoE GEMM2 (down projection) over GEMM1's sorted-slot
// MXFP4 tiles: per routed row, the top-k weighted fp32 product row.
//
// "[HIP] [CK] [FlyDSL] [Kernel] Extend MXFP4 GEMM1 replacement to A4W4",
// Summary (stage-2 paths that consume stage 1's layout) and GEMM2 scope.
//
// Persistent: one CTA per SM takes a contiguous run of work units (sorted
// block b, 256-column output tile w), numbered block by block, so that a
// block's activation tiles (K = I, at most four 17 KB atoms) are copied into
// shared memory once and stay while the CTA walks that block's tiles; the
// expert's W2 tiles (256 output rows x 256 K, one 32 KB + 2 KB copy each)
// stream through a ring that runs on across units and blocks.
//   warp 0      copies a block's activation tiles when the block changes
//               (after the previous block's MMAs have finished), and the
//               weight ring;
//   warp 1      allocates TMEM, copies the activation scales to TMEM per
//               block and each stage's weight scales, and issues per K tile
//               eight tcgen05.mma.kind::mxf4.block_scale (M = 128, N = 128,
//               K = 64): the tile's two column halves go to two of three
//               128-column accumulator slots, so the next unit's MMAs start as
//               soon as the epilogue has read one slot;
//   warps 2-5   per slot: tcgen05.ld of the 128 columns into registers, the
//               slot handed back, each valid row scaled by its routing weight
//               and written, through a small per-warp turnaround buffer, as
//               whole 128-byte row segments of row `routed row` of the
//               [T*topk, D] fp32 partial buffer.
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
  int routed_rows, D, KT, E;
  unsigned long long wait_ns;
  unsigned int* status;
};

constexpr int kM2Stages = 4;
constexpr int kM2MaxKT = 4;                              // I <= 1024
constexpr int kM2Threads = 192;
constexpr int kM2StgPitch = 144;                         // turnaround row: 32 fp32 + 16 bytes
constexpr int kM2OffA = 0;                               // activation codes, KT x 16 KB
constexpr int kM2OffAsf = kM2OffA + kM2MaxKT * 16384;    // activation scales, KT x 1 KB
constexpr int kM2OffW = kM2OffAsf + kM2MaxKT * 1024;     // weight ring, 32 KB per stage
constexpr int kM2OffWsf = kM2OffW + kM2Stages * 32768;   // weight scales, 2 KB per stage
constexpr int kM2OffStg = kM2OffWsf + kM2Stages * 2048;  // 4 warps x 32 rows
constexpr int kM2OffBar = kM2OffStg + 4 * 32 * kM2StgPitch;
constexpr int kM2NBar = 2 * kM2Stages + 2 + 3 + 3 + 1;   // ring; A full/empty; slot full x3, empty x3; drain
constexpr int kM2OffMisc = kM2OffBar + kM2NBar * 8;
constexpr int kM2Smem = kM2OffMisc + 32 + 1024;
constexpr int kM2TmemCols = 512;
constexpr int kM2SfaCol = 384;                           // after three 128-column accumulator slots
constexpr int kM2SfbCol = kM2SfaCol + 8 * kM2MaxKT;      // weight scales: 16 per stage
static_assert(kM2OffW % 1024 == 0, "swizzled tiles start 1024-aligned");
static_assert(kM2SfbCol + 16 * kM2Stages <= kM2TmemCols, "TMEM budget");
static_assert(kM2Smem <= 232448, "shared memory");

__global__ void __launch_bounds__(kM2Threads, 1) a4w4_moe2_kernel(const Moe2Args p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long drain_ns = p.wait_ns > 100000000ull ? p.wait_ns : 100000000ull;
  const int KT = p.KT, WT = p.D / 256;

  const uint32_t bar0 = base + kM2OffBar;
  auto w_full = [&](int s) { return bar0 + 8u * s; };
  auto w_empty = [&](int s) { return bar0 + 8u * (kM2Stages + s); };
  const uint32_t a_full = bar0 + 8u * (2 * kM2Stages);    // a block's activation tiles landed
  const uint32_t a_empty = a_full + 8u;                   // the block's MMAs have finished
  auto slot_full = [&](int k) { return a_empty + 8u * (1 + k); };
  auto slot_empty = [&](int k) { return a_empty + 8u * (4 + k); };
  const uint32_t drain = a_empty + 8u * 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kM2OffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kM2OffMisc + 8);
  volatile int* never = reinterpret_cast<volatile int*>(smem + kM2OffMisc + 16);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kM2Stages; ++s) {
      mbar_init(w_full(s), 1);
      mbar_init(w_empty(s), 1);
    }
    mbar_init(a_full, 1);
    mbar_init(a_empty, 1);
    for (int k = 0; k < 3; ++k) {
      mbar_init(slot_full(k), 1);
      mbar_init(slot_empty(k), 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *never = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kM2TmemCols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();                                  // GEMM1 and the sort have completed
  griddep_launch_dependents();

  // This CTA's units [u0, u1) of nb x WT, in order; a unit whose block has
  // no valid expert is skipped by every role alike.
  const long long units = static_cast<long long>(*p.num_blocks) * WT;
  const int u0 = static_cast<int>(units * blockIdx.x / gridDim.x);
  const int u1 = static_cast<int>(units * (blockIdx.x + 1) / gridDim.x);
  auto expert_of = [&](int b) {
    const int e = p.block_expert[b];
    return (e >= 0 && e < p.E) ? e : -1;
  };

  if (warp == 0) {
    // ---------------- copies ----------------
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();   // each W2 tile is read by one CTA (about once)
      const uint64_t pol_a = policy_evict_first();
      int cur_b = -1, loads = 0, g = 0;
      bool ok = true;
      for (int u = u0; u < u1 && ok; ++u) {
        const int b = u / WT, wt = u % WT;
        const int e = expert_of(b);
        if (e < 0) continue;
        if (b != cur_b) {
          // the previous block's MMAs have finished reading its tiles
          if (loads > 0 && !mbar_wait(a_empty, static_cast<uint32_t>((loads - 1) & 1), abort_flag, p.wait_ns, p.status))
            break;
          mbar_arrive_expect_tx(a_full, KT * (16384 + 1024));
          bulk_g2s(base + kM2OffA, p.Aq + static_cast<long long>(b) * KT * 16384, KT * 16384, a_full, pol_a);
          bulk_g2s(base + kM2OffAsf, p.As + static_cast<long long>(b) * KT * 1024, KT * 1024, a_full, pol_a);
          ++loads;
          cur_b = b;
        }
        const uint8_t* wq_e = p.Wq + static_cast<long long>(e) * p.expert_code_bytes;
        const uint8_t* ws_e = p.Ws + static_cast<long long>(e) * p.expert_sf_bytes;
        for (int kt = 0; kt < KT; ++kt) {
          const int s = g % kM2Stages;
          if (!mbar_wait(w_empty(s), ((g / kM2Stages) & 1) ^ 1u, abort_flag, p.wait_ns, p.status)) {
            ok = false;
            break;
          }
          const long long atom = weight_atom(2 * wt, kt, KT);   // the tile's two 128-row atoms, adjacent
          mbar_arrive_expect_tx(w_full(s), 32768 + 2048);
          bulk_g2s(base + kM2OffW + s * 32768, wq_e + atom * 16384, 32768, w_full(s), pol_w);
          bulk_g2s(base + kM2OffWsf + s * 2048, ws_e + atom * 1024, 2048, w_full(s), pol_w);
          ++g;
        }
      }
      // every copy issued lands before the shared memory is released
      if (loads > 0) mbar_wait(a_full, static_cast<uint32_t>((loads - 1) & 1), never, drain_ns, p.status);
      for (int j = (g > kM2Stages ? g - kM2Stages : 0); j < g; ++j)
        mbar_wait(w_full(j % kM2Stages), (j / kM2Stages) & 1u, never, drain_ns, p.status);
    }
  } else if (warp == 1) {
    // ---------------- scale copies + MMA ----------------
    if (lane == 0) {
      const uint64_t asfd = sdesc_sf(base + kM2OffAsf), wsfd = sdesc_sf(base + kM2OffWsf);
      const uint64_t adesc0 = sdesc_sw128(base + kM2OffA), wdesc0 = sdesc_sw128(base + kM2OffW);
      const uint32_t idesc0 = idesc_mxf4(128, 0, 0), idesc2 = idesc_mxf4(128, 2, 2);
      int cur_b = -1, loads = 0, g = 0, pos = 0;
      bool ok = true;
      for (int u = u0; u < u1 && ok; ++u) {
        const int b = u / WT;
        if (expert_of(b) < 0) continue;
        if (b != cur_b) {
          if (cur_b >= 0) mma_commit(a_empty);   // the previous block's tiles are free once its MMAs finish
          if (!mbar_wait(a_full, static_cast<uint32_t>(loads & 1), abort_flag, p.wait_ns, p.status)) break;
          tc_fence_after();
          for (int kt = 0; kt < KT; ++kt)
            for (int ka = 0; ka < 2; ++ka)
              tmem_copy_sf_desc(tmem + kM2SfaCol + kt * 8 + ka * 4, asfd + ((kt * 1024 + ka * 512) >> 4));
          ++loads;
          cur_b = b;
        }
        // the tile's two column halves go to accumulator slots pos % 3 and
        // (pos + 1) % 3; wait until the epilogue has read their last use
        int slot[2];
        for (int h = 0; h < 2; ++h) {
          const int q = pos + h, k = q % 3, use = q / 3;
          slot[h] = k;
          if (use > 0 && !mbar_wait(slot_empty(k), static_cast<uint32_t>((use - 1) & 1), abort_flag, p.wait_ns, p.status))
            ok = false;
        }
        if (!ok) break;
        tc_fence_after();
        for (int kt = 0; kt < KT; ++kt) {
          const int s = g % kM2Stages;
          if (!mbar_wait(w_full(s), (g / kM2Stages) & 1u, abort_flag, p.wait_ns, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfb = tmem + kM2SfbCol + s * 16;
          for (int ka = 0; ka < 2; ++ka)
            for (int a = 0; a < 2; ++a)
              tmem_copy_sf_desc(sfb + ka * 8 + a * 4, wsfd + ((s * 2048 + a * 1024 + ka * 512) >> 4));
          const uint64_t ad = adesc0 + ((kt * 16384) >> 4);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint64_t wd = wdesc0 + ((s * 32768 + h * 16384) >> 4);   // rows 128h .. 128h+127 of the tile
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const int ka = ks >> 1;
              mma_mxf4(tmem + slot[h] * 128, ad + ks * 2, wd + ks * 2, (ks & 1) ? idesc2 : idesc0,
                       tmem + kM2SfaCol + kt * 8 + ka * 4, sfb + ka * 8 + h * 4, (kt > 0 || ks > 0) ? 1u : 0u);
            }
          }
          mma_commit(w_empty(s));
          ++g;
        }
        if (!ok) break;
        mma_commit(slot_full(slot[0]));
        mma_commit(slot_full(slot[1]));
        pos += 2;
      }
      // TMEM is not released while MMAs may run
      mma_commit(drain);
      mbar_wait(drain, 0, never, drain_ns, p.status);
    }
  } else {
    // ---------------- epilogue (warps 2-5, one TMEM lane quadrant each) ----------------
    const int q = warp & 3, lrow = q * 32 + lane;
    const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint8_t* stg = smem + kM2OffStg + (warp - 2) * 32 * kM2StgPitch;
    int cur_b = -1, entry = 0, pos = 0;
    bool valid = false, ok = true;
    float wgt = 0.f;
    for (int u = u0; u < u1 && ok; ++u) {
      const int b = u / WT, wt = u % WT;
      if (expert_of(b) < 0) continue;
      if (b != cur_b) {
        entry = p.sorted_rows[b * 128 + lrow];
        valid = entry >= 0 && entry < p.routed_rows;
        wgt = valid ? __ldg(p.topk_w + entry) : 0.f;
        cur_b = b;
      }
      for (int h = 0; h < 2; ++h) {
        const int qq = pos + h, k = qq % 3, use = qq / 3;
        if (!mbar_wait(slot_full(k), static_cast<uint32_t>(use & 1), abort_flag, p.wait_ns, p.status)) {
          ok = false;
          break;
        }
        __syncwarp();
        tc_fence_after();
        float v[128];
        tmem_ld64(tq + k * 128, v);
        tmem_ld64(tq + k * 128 + 64, v + 64);
        tc_fence_before();
        mbar_arrive(slot_empty(k));              // the slot may take the next unit's MMAs
        const int n0 = wt * 256 + h * 128;
        uint4* mine = reinterpret_cast<uint4*>(stg + lane * kM2StgPitch);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float* x = v + c * 32 + 4 * t;
            mine[t] = make_uint4(__float_as_uint(wgt * x[0]), __float_as_uint(wgt * x[1]), __float_as_uint(wgt * x[2]),
                                 __float_as_uint(wgt * x[3]));
          }
          __syncwarp();
#pragma unroll
          for (int r4 = 0; r4 < 8; ++r4) {
            const int r = r4 * 4 + (lane >> 3), seg = lane & 7;
            const int er = __shfl_sync(0xffffffffu, entry, r);
            const int vr = __shfl_sync(0xffffffffu, valid ? 1 : 0, r);
            const uint4 val = *reinterpret_cast<const uint4*>(stg + r * kM2StgPitch + seg * 16);
            if (vr)
              __stcs(reinterpret_cast<uint4*>(p.partial + static_cast<long long>(er) * p.D + n0 + c * 32 + seg * 4), val);
          }
          __syncwarp();
        }
      }
      pos += 2;
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

int launch_moe_gemm2_persistent(const void* Aq, const void* As, int T, int I, const int32_t* sorted_rows,
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
  // one CTA per SM, or one per unit when the blocks can give fewer units
  const long long max_units = static_cast<long long>(max_blocks) * (D / 256);
  const int grid = static_cast<int>(max_units < sms ? max_units : sms);
  if (grid < 1) return 0;
  static std::atomic<unsigned long long> attr_devs{0};
  if (ensure_func_attrs(attr_devs, [&] {
        return cudaFuncSetAttribute(a4w4_moe2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kM2Smem) ==
               cudaSuccess;
      }) != 0)
    return -4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
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
