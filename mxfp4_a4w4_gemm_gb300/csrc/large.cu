// large.cu -- persistent large-M dense A4W4 GEMM (sm_103a).
//
// "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM", Summary/Implementation
// and the M = 1 ... 2048 microbenchmark: MXFP4 activations (quantised once
// beforehand at large M, the page's separate-quant path) times preshuffled
// MXFP4 weights, fp32 accumulation, BF16 output with M-tail masking.
//
// One CTA per SM walks a list of work units; a unit is a 128 x 256 output
// tile (activation tile x, weight tile w), or one 128-column half of a tile of
// the last, partial wave (two CTAs take the two halves: the wave's operand
// bytes per SM drop from 51 KB to 34 KB per K step, its own output columns
// each, nothing to reduce).  The operand ring runs on across units: the next
// unit's copies land while the epilogue drains the accumulator.  The ring's
// 204 KB hold four 51 KB stages of one K step for whole tiles, or three 68 KB
// stages of two K steps for halves (the SM's bulk-copy pipe turns a stage
// over in no less than ~0.42 us whatever its size up to ~51 KB, so a half
// unit's 34 KB per K step would leave it a third idle); a CTA whose walk goes
// on from whole tiles to halves lets the whole-tile stages drain before it
// reuses their bytes.
//   warp 0     producer: per 256-wide K step one 17 KB activation atom, the
//              two adjacent 16 KB weight atoms and their 2 KB of scales (one
//              atom and 1 KB for a half unit, two K steps to a stage);
//   warp 1     TMEM owner and MMA issuer: scale copies into TMEM, four
//              tcgen05.mma.kind::mxf4.block_scale (M = 128, N = 256 or 128,
//              K = 64) per step; before a unit's first MMA it waits until the
//              epilogue has read the previous unit's accumulator;
//   warps 2-5  epilogue (one per TMEM lane quadrant, a thread per row):
//              the accumulator row -> packed BF16 registers, TMEM handed
//              back, then 64-column chunks turned around in a small per-warp
//              buffer so that each store writes whole 128-byte row segments.
#include "device.cuh"
#include "launch.h"

namespace a4w4 {

struct LargeArgs {
  const uint8_t* Aq;        // activation tiles: atom (x_tile, kt) = 17408 bytes (codes, then scales)
  const uint8_t* Wq;        // preshuffled weight codes
  const uint8_t* Ws;        // preshuffled weight scales
  uint16_t* C;              // [M, N] BF16
  int M, N, KT, w_tiles;
  int full_units;           // tiles 0 .. full_units-1 run whole
  int units;                // full_units + 2 x (tiles run as two 128-column halves)
  unsigned long long wait_ns;
  unsigned int* status;
};

struct LCfg {
  static constexpr int THREADS = 192;
  static constexpr int A_BYTES = 17408;          // 128 rows x 256 K: codes + scales
  static constexpr int ATOM_BYTES = 16384;       // one 128-row weight atom, one K step
  static constexpr int ATOM_SF_BYTES = 1024;     // its scales
  static constexpr int RING_BYTES = 4 * (A_BYTES + 2 * (ATOM_BYTES + ATOM_SF_BYTES));
  // epilogue turnaround: per warp 32 rows x 64 BF16 columns, rows padded to
  // 144 bytes (conflict-free 16-byte accesses row-wise and column-wise)
  static constexpr int STG_PITCH = 144;
  static constexpr int STG_BYTES = 32 * STG_PITCH;
  static constexpr int OFF_STG = RING_BYTES;
  static constexpr int OFF_BAR = OFF_STG + 4 * STG_BYTES;
  // full, empty per stage of the two rings; acc_full, acc_empty, drain
  static constexpr int NBAR = 2 * (4 + 3) + 3;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 32 + 1024;
  static constexpr int ACC_COLS = 256;
  static constexpr int SFA_COLS = 8;             // 2 K halves x 4 columns
  static constexpr int SFB_COLS = 16;            // 2 K halves x 2 weight atoms x 4 columns
  static constexpr int SF_STAGE_COLS = SFA_COLS + SFB_COLS;
  static constexpr int TMEM_COLS = 512;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// The two ring geometries over the same bytes.  A stage holds KTS K steps:
// their activation atoms side by side (consecutive K steps of a row tile are
// adjacent in the activation tiles, one copy), then per K step the weight
// atom(s) and their scales; each geometry keeps the activation, weight and
// scale parts of all its stages in three separate arrays.  Barriers BAR ..
// BAR+STAGES-1 are the stages' "landed" barriers, the next STAGES their
// "consumed" ones.
template <bool HALF>
struct LRing {
  static constexpr int STAGES = HALF ? 3 : 4;
  static constexpr int KTS = HALF ? 2 : 1;       // K steps per stage
  static constexpr int ATOMS = HALF ? 1 : 2;     // weight atoms per K step
  static constexpr int W_STEP = ATOMS * LCfg::ATOM_BYTES;
  static constexpr int WSF_STEP = ATOMS * LCfg::ATOM_SF_BYTES;
  static constexpr int A_STAGE = KTS * LCfg::A_BYTES;
  static constexpr int W_STAGE = KTS * W_STEP;
  static constexpr int WSF_STAGE = KTS * WSF_STEP;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_W = OFF_A + STAGES * A_STAGE;
  static constexpr int OFF_WSF = OFF_W + STAGES * W_STAGE;
  static constexpr int BAR = HALF ? 8 : 0;
  static constexpr uint32_t TX_STEP = LCfg::A_BYTES + W_STEP + WSF_STEP;   // bytes per K step
  static_assert(LCfg::A_BYTES % 1024 == 0 && OFF_W % 1024 == 0 && W_STEP % 1024 == 0,
                "swizzled tiles start 1024-aligned");
  static_assert(OFF_WSF + STAGES * WSF_STAGE <= LCfg::RING_BYTES, "ring bytes");
  static_assert(LCfg::ACC_COLS + STAGES * KTS * LCfg::SF_STAGE_COLS <= LCfg::TMEM_COLS, "TMEM budget");
  static __device__ __forceinline__ uint32_t full(uint32_t bar0, int s) { return bar0 + 8u * (BAR + s); }
  static __device__ __forceinline__ uint32_t empty(uint32_t bar0, int s) { return bar0 + 8u * (BAR + STAGES + s); }
};
static_assert(LRing<true>::BAR == 2 * LRing<false>::STAGES, "barrier layout");
static_assert(2 * (LRing<false>::STAGES + LRing<true>::STAGES) + 3 == LCfg::NBAR, "barrier count");

// Unit u -> tile and column half (-1: the whole 256 columns).
__device__ __forceinline__ void large_unit(const LargeArgs& p, int u, int& tile, int& half) {
  if (u < p.full_units) {
    tile = u;
    half = -1;
  } else {
    const int v = u - p.full_units;
    tile = p.full_units + (v >> 1);
    half = v & 1;
  }
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Producer: the K steps of one unit into ring R, KTS per stage (fewer in the
// last stage when KT is not a multiple); g counts the stages issued on R.
// False when a wait gave up.
template <bool HALF>
__device__ __forceinline__ bool large_produce(const LargeArgs& p, uint32_t base, uint32_t bar0, int tile, int half,
                                              int& g, uint64_t pol, volatile int* abort_flag) {
  using R = LRing<HALF>;
  const int x_tile = tile / p.w_tiles, w_tile = tile % p.w_tiles;
  for (int kt = 0; kt < p.KT; kt += R::KTS) {
    const int nk = p.KT - kt < R::KTS ? p.KT - kt : R::KTS;
    const int s = g % R::STAGES;
    if (!mbar_wait(R::empty(bar0, s), ((g / R::STAGES) & 1) ^ 1u, abort_flag, p.wait_ns, p.status)) return false;
    const long long aatom = static_cast<long long>(x_tile) * p.KT + kt;
    const uint32_t fb = R::full(bar0, s);
    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nk) * R::TX_STEP);
    bulk_g2s(base + R::OFF_A + s * R::A_STAGE, p.Aq + aatom * LCfg::A_BYTES, nk * LCfg::A_BYTES, fb, pol);
    for (int k2 = 0; k2 < nk; ++k2) {
      const long long watom = weight_atom(2 * w_tile, kt + k2, p.KT) + (half > 0 ? 1 : 0);
      bulk_g2s(base + R::OFF_W + s * R::W_STAGE + k2 * R::W_STEP, p.Wq + watom * LCfg::ATOM_BYTES, R::W_STEP, fb, pol);
      bulk_g2s(base + R::OFF_WSF + s * R::WSF_STAGE + k2 * R::WSF_STEP, p.Ws + watom * LCfg::ATOM_SF_BYTES,
               R::WSF_STEP, fb, pol);
    }
    ++g;
  }
  return true;
}

// MMA issuer: the K steps of one unit from ring R into the accumulator.
template <bool HALF>
__device__ __forceinline__ bool large_mma(const LargeArgs& p, uint32_t base, uint32_t bar0, uint32_t tmem, int& g,
                                          volatile int* abort_flag) {
  using R = LRing<HALF>;
  constexpr int N = HALF ? 128 : 256;
  const uint32_t idesc0 = idesc_mxf4(N, 0, 0), idesc2 = idesc_mxf4(N, 2, 2);
  const uint64_t adesc0 = sdesc_sw128(base + R::OFF_A), bdesc0 = sdesc_sw128(base + R::OFF_W);
  const uint64_t asfd0 = sdesc_sf(base + R::OFF_A + 16384), bsfd0 = sdesc_sf(base + R::OFF_WSF);
  for (int kt = 0; kt < p.KT; kt += R::KTS) {
    const int nk = p.KT - kt < R::KTS ? p.KT - kt : R::KTS;
    const int s = g % R::STAGES;
    if (!mbar_wait(R::full(bar0, s), (g / R::STAGES) & 1u, abort_flag, p.wait_ns, p.status)) return false;
    tc_fence_after();
#pragma unroll
    for (int k2 = 0; k2 < R::KTS; ++k2) {
      if (k2 < nk) {
        const uint32_t sfa = tmem + LCfg::ACC_COLS + (s * R::KTS + k2) * LCfg::SF_STAGE_COLS;
        const uint32_t sfb = sfa + LCfg::SFA_COLS;
        const uint32_t aoff = s * R::A_STAGE + k2 * LCfg::A_BYTES;
        const uint64_t ad = adesc0 + (aoff >> 4), bd = bdesc0 + ((s * R::W_STAGE + k2 * R::W_STEP) >> 4);
        const uint64_t asd = asfd0 + (aoff >> 4), bsd = bsfd0 + ((s * R::WSF_STAGE + k2 * R::WSF_STEP) >> 4);
#pragma unroll
        for (int ka = 0; ka < 2; ++ka) {
          tmem_copy_sf_desc(sfa + ka * 4, asd + ka * (512 >> 4));
          tmem_copy_sf_desc(sfb + ka * 8, bsd + (ka * 512) / 16);
          if (!HALF) tmem_copy_sf_desc(sfb + ka * 8 + 4, bsd + (1024 + ka * 512) / 16);
        }
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const int ka = ks >> 1;
          mma_mxf4(tmem, ad + ks * 2, bd + ks * 2, (ks & 1) ? idesc2 : idesc0, sfa + ka * 4, sfb + ka * 8,
                   (kt + k2 > 0 || ks > 0) ? 1u : 0u);
        }
      }
    }
    mma_commit(R::empty(bar0, s));
    ++g;
  }
  return true;
}

__global__ void __launch_bounds__(LCfg::THREADS, 1) a4w4_large_kernel(const LargeArgs p) {
  using Cf = LCfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const unsigned long long drain_ns = p.wait_ns > 100000000ull ? p.wait_ns : 100000000ull;

  const uint32_t bar0 = base + Cf::OFF_BAR;
  const uint32_t acc_full = bar0 + 8u * (Cf::NBAR - 3);   // a unit's accumulator is complete
  const uint32_t acc_empty = acc_full + 8u;               // the epilogue has read it
  const uint32_t drain = acc_empty + 8u;                  // every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cf::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cf::OFF_MISC + 8);
  volatile int* never = reinterpret_cast<volatile int*>(smem + Cf::OFF_MISC + 16);

  if (threadIdx.x == 0) {
    for (int b = 0; b < Cf::NBAR - 3; ++b) mbar_init(bar0 + 8u * b, 1);
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 128);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *never = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cf::TMEM_COLS);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The activation tiles come from the kernel just before this one.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();   // operands are re-read by other tiles from L2
      int g = 0, gh = 0;                          // stages issued on each ring (a ring runs on across units)
      bool ok = true, on_half = false;
      int u = blockIdx.x;
      for (; u < p.full_units && ok; u += G) ok = large_produce<false>(p, base, bar0, u, -1, g, pol, abort_flag);
      if (ok && u < p.units) {
        // the half-unit ring reuses the whole-tile ring's bytes: every
        // whole-tile stage issued has been consumed first
        constexpr int S = LRing<false>::STAGES;
        for (int j = (g > S ? g - S : 0); j < g && ok; ++j)
          ok = mbar_wait(LRing<false>::empty(bar0, j % S), (j / S) & 1u, abort_flag, p.wait_ns, p.status);
        on_half = ok;
        for (; u < p.units && ok; u += G) {
          int tile, half;
          large_unit(p, u, tile, half);
          ok = large_produce<true>(p, base, bar0, tile, half, gh, pol, abort_flag);
        }
      }
      // every copy issued lands before the CTA's shared memory is released
      if (on_half) {
        constexpr int S = LRing<true>::STAGES;
        for (int j = (gh > S ? gh - S : 0); j < gh; ++j)
          mbar_wait(LRing<true>::full(bar0, j % S), (j / S) & 1u, never, drain_ns, p.status);
      } else {
        constexpr int S = LRing<false>::STAGES;
        for (int j = (g > S ? g - S : 0); j < g; ++j)
          mbar_wait(LRing<false>::full(bar0, j % S), (j / S) & 1u, never, drain_ns, p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // (a half stage's scales reuse a whole-tile stage's TMEM columns only
    // after the producer has seen every whole-tile stage consumed)
    if (lane == 0) {
      int g = 0, gh = 0, j = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units && ok; u += G, ++j) {
        // the epilogue has read the previous unit's accumulator
        if (j > 0) {
          if (!mbar_wait(acc_empty, static_cast<uint32_t>((j - 1) & 1), abort_flag, p.wait_ns, p.status)) break;
          tc_fence_after();
        }
        ok = u < p.full_units ? large_mma<false>(p, base, bar0, tmem, g, abort_flag)
                              : large_mma<true>(p, base, bar0, tmem, gh, abort_flag);
        if (ok) mma_commit(acc_full);
      }
      // TMEM is released only after every MMA issued has completed.
      mma_commit(drain);
      mbar_wait(drain, 0, never, drain_ns, p.status);
    }
  } else {
    // ---------------- epilogue (4 warps, one per TMEM lane quadrant) ----------------
    const int q = warp & 3;
    const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint8_t* stg = smem + Cf::OFF_STG + (warp - 2) * Cf::STG_BYTES;
    int j = 0;
    for (int u = blockIdx.x; u < p.units; u += G, ++j) {
      int tile, half;
      large_unit(p, u, tile, half);
      const int x_tile = tile / p.w_tiles, w_tile = tile % p.w_tiles;
      if (!mbar_wait(acc_full, static_cast<uint32_t>(j & 1), abort_flag, p.wait_ns, p.status)) break;
      __syncwarp();
      tc_fence_after();
      const int row0 = x_tile * 128 + q * 32;       // this warp's 32 rows
      const int cols = half < 0 ? 256 : 128;
      const int n0 = w_tile * 256 + (half > 0 ? 128 : 0);
      // The whole accumulator row into registers first (packed BF16), so
      // that TMEM goes back to the MMA warp before any store is issued.
      uint32_t pk[128];
#pragma unroll
      for (int c0 = 0; c0 < 256; c0 += 64) {
        if (c0 < cols) {
          float v[64];
          tmem_ld64(tq + c0, v);
#pragma unroll
          for (int t = 0; t < 32; ++t) pk[c0 / 2 + t] = bf16x2_bits(v[2 * t], v[2 * t + 1]);
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty);
      // per 64-column chunk: row lane -> buffer row; then 8 lanes per row,
      // 4 rows per store
      uint4* mine = reinterpret_cast<uint4*>(stg + lane * Cf::STG_PITCH);
#pragma unroll
      for (int c0 = 0; c0 < 256; c0 += 64) {
        if (c0 < cols) {
#pragma unroll
          for (int t = 0; t < 8; ++t)
            mine[t] = make_uint4(pk[c0 / 2 + 4 * t], pk[c0 / 2 + 4 * t + 1], pk[c0 / 2 + 4 * t + 2],
                                 pk[c0 / 2 + 4 * t + 3]);
          __syncwarp();
#pragma unroll
          for (int r4 = 0; r4 < 8; ++r4) {
            const int r = r4 * 4 + (lane >> 3), seg = lane & 7;
            const uint4 val = *reinterpret_cast<const uint4*>(stg + r * Cf::STG_PITCH + seg * 16);
            if (row0 + r < p.M)
              *reinterpret_cast<uint4*>(p.C + static_cast<long long>(row0 + r) * p.N + n0 + c0 + seg * 8) = val;
          }
          __syncwarp();
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, Cf::TMEM_COLS);
  }
}

int launch_large(const GemmPlan& pl, const uint8_t* Aq, int M, const void* Wq, const void* Ws, int N, void* C,
                 cudaStream_t st, unsigned long long wait_ns, unsigned int* status, int sms) {
  const int tiles = pl.x_tiles * pl.w_tiles;
  const int units = tiles + pl.half_tiles;
  if (tiles < 1 || pl.half_tiles < 0 || pl.half_tiles > tiles || sms < 1) return -4;
  static std::atomic<unsigned long long> attr_devs{0};   // bit d: attribute set on device d
  if (ensure_func_attrs(attr_devs, [&] {
        return cudaFuncSetAttribute(a4w4_large_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    LCfg::SMEM_BYTES) == cudaSuccess;
      }) != 0)
    return -4;
  LargeArgs a{};
  a.Aq = Aq;
  a.Wq = static_cast<const uint8_t*>(Wq);
  a.Ws = static_cast<const uint8_t*>(Ws);
  a.C = static_cast<uint16_t*>(C);
  a.M = M; a.N = N; a.KT = pl.kt; a.w_tiles = pl.w_tiles;
  a.full_units = tiles - pl.half_tiles;
  a.units = units;
  a.wait_ns = wait_ns;
  a.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units < sms ? units : sms, 1, 1);
  cfg.blockDim = dim3(LCfg::THREADS, 1, 1);
  cfg.dynamicSmemBytes = LCfg::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, a4w4_large_kernel, a) != cudaSuccess) return -4;
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace a4w4
