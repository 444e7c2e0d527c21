// a16w4.cu -- A16WFP4 GEMM: BF16 activations (not quantised) x MXFP4 weights.
//
// "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM", Summary (BF16
// activation x decoded MXFP4 weight): C = A W^T with W the E2M1 codes times
// their E8M0 block scales, BF16 operands, fp32 accumulation, BF16 output.
//
// Work layout as in the decode kernel (swap-AB: a 128-row weight tile is the
// MMA's M side, up to NX tokens its N side, the K range split over the CTAs
// of a thread-block cluster), but the weights reach the tensor core as BF16
// decoded on chip, one CTA per SM:
//
//   warp 0      weight producer: 16 KB + 1 KB bulk copies per 256-wide K
//               tile into an SW-deep ring; a slot is handed back as soon as
//               the decoders have read it, so the next copies overlap the
//               decoding and the MMAs;
//   warp 1      TMEM owner and MMA issuer: per K tile 16 tcgen05.mma.kind::f16
//               (K = 16 each) with the decoded weights in TMEM (A operand)
//               and the tokens in shared memory (B operand), spread round
//               robin over four accumulators summed at the end;
//   warps 2..17 decoders: warp w serves TMEM lane quadrant w % 4 (the lanes
//               a warp may access) and K quarter (w - 2) / 4 of every K tile,
//               so thread (w, lane) expands the two 32-blocks of weight row
//               32 (w % 4) + lane in that quarter to BF16 in registers and
//               writes them to its lane with one tcgen05.st; the decoders
//               also stage the tokens' BF16 chunks.  The first four then drain
//               the accumulator, and all of them reduce split-K partials over
//               DSMEM exactly as the decode kernel does.
//
// Decoding without conversion instructions.  Within each group of 8 K
// elements the weights are written in the order (0,4,1,5,2,6,3,7) and the
// tokens staged in the same order: one permutation applied to both operands
// of a dot product leaves it unchanged.  Elements j and j+4 of a 32-bit word
// of eight E2M1 codes then form one BF16x2 word with two shifts and two
// masks: the code's 3 magnitude bits (exponent e, mantissa m) placed at bits
// 6..8 of a BF16 read as exactly the code's value times 2^-126 (e = 0, m = 1,
// the value 0.5, becomes the subnormal 2^-127), and the sign goes to bit 15.
// One BF16x2 multiply by 2^(s-1) then applies the E8M0 scale s exactly; when
// 2^(s-1) is not a BF16 normal (s > 128) two multiplies do it, by 2^126 and
// by 2^(s-127).
#include "device.cuh"
#include "launch.h"

#include <atomic>

namespace a4w4 {

namespace {

struct A16W4Args {
  const uint16_t* A;   // activations [M, K] BF16
  const uint8_t* Wq;   // preshuffled weight codes
  const uint8_t* Ws;   // preshuffled weight scales
  uint16_t* C;         // [M, N] BF16
  int M, N, K, KT, splits;
  int prefetch_w;      // 1: weights may be read before the previous grid on the stream completes
  unsigned long long wait_ns;
  unsigned int* status;
};

constexpr int kMaxA16W4Splits = 16;   // non-portable cluster size

template <int NX, int SW>
struct HCfg {
  static constexpr int DWARPS = 16;                               // decoder warps: 4 per lane quadrant
  static constexpr int THREADS = 64 + 32 * DWARPS;
  static constexpr int SB = 3;                                    // decoded-tile slots (TMEM + token tile)
  static constexpr int W_STAGE = 16384, WSF_STAGE = 1024;
  static constexpr int X_STAGE = NX * 512;                        // 4 atoms of 64 K: NX rows x 128 B each
  static constexpr int OFF_W = 0;
  static constexpr int OFF_WSF = OFF_W + SW * W_STAGE;
  static constexpr int OFF_X = OFF_WSF + SW * WSF_STAGE;
  // push buffer: up to 16 rank slots of ceil(G / S) float4 groups, G = 32 x tokens
  static constexpr int PUSH_BYTES = NX * 512 + 256;
  static constexpr int OFF_PUSH = OFF_X + SB * X_STAGE;
  static constexpr int OFF_BAR = OFF_PUSH + PUSH_BYTES;
  static constexpr int NBAR = 2 * SW + 2 * SB + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 32 + 1024;        // + slack to align the base to 1024
  // TMEM: NACC accumulators in columns [32 a, 32 a + NX); decoded weight
  // slot s (128 rows x 256 K as BF16 pairs) in columns [128 (s + 1), 128 (s + 2)).
  // Consecutive MMAs of a K tile go to different accumulators: MMAs chained
  // on one accumulator run one after another, each waiting for the last.
  static constexpr int NACC = 4;
  static constexpr int A_COL0 = 128;
  static constexpr int TMEM_COLS = 512;
  static constexpr int XCH = (NX * 32 + 32 * DWARPS - 1) / (32 * DWARPS);   // token chunks per thread
  static_assert(NX % 16 == 0 && NX <= 32, "token tile");
  static_assert(SW >= 2, "ring");
  static_assert(A_COL0 + SB * 128 <= TMEM_COLS && NX <= 32 && NACC * 32 <= A_COL0, "TMEM budget");
  static_assert(OFF_X % 1024 == 0 && X_STAGE % 1024 == 0, "swizzled token tiles");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(2 * (SMEM_BYTES + 1024) > 233472, "one CTA per SM (the whole TMEM)");
  static_assert(NX * 128 * 4 <= SW * W_STAGE, "a staged partial must fit in the drained weight ring");
};

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
         "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
         "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
         "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D (TMEM, fp32) (+)= A (TMEM, BF16 pairs, K-major rows) x B (shared memory
// descriptor), kind::f16.
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Eight E2M1 codes (element i in bits 4i..4i+3) -> four BF16x2 words holding
// elements (j, j+4), each the code's value times 2^-126.
__device__ __forceinline__ void e2m1x8_to_bf16x2_pow2m126(uint32_t w, uint32_t* o) {
  constexpr uint32_t kMag = 0x01C001C0u, kSign = 0x80008000u;
  o[0] = ((w << 6) & kMag) | ((w << 12) & kSign);
  o[1] = ((w << 2) & kMag) | ((w << 8) & kSign);
  o[2] = ((w >> 2) & kMag) | ((w << 4) & kSign);
  o[3] = ((w >> 6) & kMag) | (w & kSign);
}

// Two 32-blocks of E2M1 codes with their E8M0 scales -> 32 BF16x2 words in
// the permuted K order above.
__device__ __forceinline__ void decode_two_blocks(uint4 c0, uint4 c1, uint32_t s0, uint32_t s1, uint32_t* o) {
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int q = 0; q < 8; ++q) e2m1x8_to_bf16x2_pow2m126(w[q], o + 4 * q);
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const uint32_t s = b ? s1 : s0;
    if (s <= 128u) {
      const uint32_t f = ((s + 126u) << 7) * 0x00010001u;     // 2^(s-1) in both halves
#pragma unroll
      for (int j = 0; j < 16; ++j) o[16 * b + j] = mul_bf16x2(o[16 * b + j], f);
    } else {
      const uint32_t f = ((s & 0xFFu) << 7) * 0x00010001u;    // 2^(s-127) (s = 255: the NaN scale -> inf)
#pragma unroll
      for (int j = 0; j < 16; ++j) o[16 * b + j] = mul_bf16x2(mul_bf16x2(o[16 * b + j], 0x7E807E80u), f);
    }
  }
}

template <int NX, int SW>
__global__ void __launch_bounds__(HCfg<NX, SW>::THREADS, 1) a4w4_a16w4_kernel(const A16W4Args p) {
  using Cf = HCfg<NX, SW>;
  constexpr int SB = Cf::SB;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w_tile = blockIdx.x, x_tile = blockIdx.y, split = blockIdx.z;
  const int kt0 = static_cast<int>(static_cast<long long>(split) * p.KT / p.splits);
  const int kt1 = static_cast<int>(static_cast<long long>(split + 1) * p.KT / p.splits);
  const int nk = kt1 - kt0;
  const int m0 = x_tile * NX;
  const int mvalid = min(NX, p.M - m0);
  const unsigned long long drain_ns = p.wait_ns > 100000000ull ? p.wait_ns : 100000000ull;

  const uint32_t bar0 = base + Cf::OFF_BAR;
  auto full_w = [&](int s) { return bar0 + 8u * s; };
  auto empty_w = [&](int s) { return bar0 + 8u * (SW + s); };
  auto full_b = [&](int s) { return bar0 + 8u * (2 * SW + s); };
  auto empty_b = [&](int s) { return bar0 + 8u * (2 * SW + SB + s); };
  const uint32_t tmem_full = bar0 + 8u * (2 * SW + 2 * SB);
  const uint32_t red_bar = tmem_full + 8u;   // peers' pushes into this CTA's slice
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cf::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cf::OFF_MISC + 8);
  volatile int* never = reinterpret_cast<volatile int*>(smem + Cf::OFF_MISC + 16);
  volatile int* epi_ready = reinterpret_cast<volatile int*>(smem + Cf::OFF_MISC + 24);
  volatile int* owner_ready = reinterpret_cast<volatile int*>(smem + Cf::OFF_MISC + 28);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(full_w(s), 1);
      mbar_init(empty_w(s), Cf::DWARPS);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(full_b(s), Cf::DWARPS);
      mbar_init(empty_b(s), 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(red_bar, 1);
    *abort_flag = 0;
    *never = 0;
    *epi_ready = 0;
    fence_barrier_init();
    if (p.splits > 1) {
      // this CTA's slice receives S x (its groups) x 16 bytes
      const int S = p.splits, G = mvalid * 32;
      const int rank = static_cast<int>(cluster_ctarank());
      const int g0 = static_cast<int>(static_cast<long long>(rank) * G / S);
      const int g1 = static_cast<int>(static_cast<long long>(rank + 1) * G / S);
      mbar_arrive_expect_tx(red_bar, static_cast<uint32_t>(S * (g1 - g0) * 16));
    }
  }
  // Token rows beyond M are never written by the decoders: zeroed here once
  // for every slot.
  for (int i = threadIdx.x; i < SB * Cf::X_STAGE / 16; i += Cf::THREADS)
    reinterpret_cast<uint4*>(smem + Cf::OFF_X)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  __syncthreads();
  if (p.splits > 1) cluster_arrive_relaxed();  // paired with cluster_wait() before the first push / the exit
  bool cluster_waited = false;

  const uint64_t pol = policy_evict_first();   // every weight byte is read once
  auto issue_w = [&](int i) {
    const int s = i % SW;
    const long long atom = weight_atom(w_tile, kt0 + i, p.KT);
    mbar_arrive_expect_tx(full_w(s), Cf::W_STAGE + Cf::WSF_STAGE);
    bulk_g2s(base + Cf::OFF_W + s * Cf::W_STAGE, p.Wq + atom * 16384, 16384, full_w(s), pol);
    bulk_g2s(base + Cf::OFF_WSF + s * Cf::WSF_STAGE, p.Ws + atom * 1024, 1024, full_w(s), pol);
  };
  int issued = 0;
  if (warp == 0 && lane == 0) {
    // The first ring pass needs no empty-slot wait.  Weights are read before
    // the grid dependency resolves only on request: the previous kernel on
    // the stream must not write them.
    if (!p.prefetch_w) griddep_wait();
    issued = nk < SW ? nk : SW;
    for (int i = 0; i < issued; ++i) issue_w(i);
  }
  uint32_t tmem = 0;
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cf::TMEM_COLS);
    tc_fence_before();
    __syncwarp();
    tc_fence_after();
    tmem = *tmem_slot;
  }
  // every role needs the TMEM address (the decoders write their tiles there)
  __syncthreads();
  tc_fence_after();
  tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- weight producer ----------------
    griddep_wait();
    griddep_launch_dependents();
    if (lane == 0 && nk > 0) {
      int i = issued;
      for (; i < nk; ++i) {
        const int s = i % SW;
        if (!mbar_wait(empty_w(s), ((i / SW) & 1) ^ 1u, abort_flag, p.wait_ns, p.status)) break;
        issue_w(i);
      }
      // every copy issued lands before the CTA's shared memory is released
      for (int j = (i > SW ? i - SW : 0); j < i; ++j)
        mbar_wait(full_w(j % SW), (j / SW) & 1u, never, drain_ns, p.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    griddep_launch_dependents();
    if (lane == 0) {
      const uint64_t xdesc0 = sdesc_sw128(base + Cf::OFF_X);
      const uint32_t idesc = idesc_bf16(NX);
      bool ok = true;
      for (int i = 0; i < nk; ++i) {
        const int s = i % SB;
        if (!mbar_wait(full_b(s), (i / SB) & 1u, abort_flag, p.wait_ns, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_col = tmem + Cf::A_COL0 + s * 128;
        const uint64_t xd = xdesc0 + ((s * Cf::X_STAGE) >> 4);
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int j = g * 4 + kk;
            mma_bf16_tmem_a(tmem + (j % Cf::NACC) * 32, a_col + g * 32 + kk * 8, xd + ((g * NX * 128) >> 4) + kk * 2,
                            idesc, (i > 0 || j >= Cf::NACC) ? 1u : 0u);
          }
        // a slot is handed back only if a later K tile will refill it
        if (i + SB < nk) mma_commit(empty_b(s));
      }
      (void)ok;
      mma_commit(tmem_full);
      // TMEM is never released while MMAs may still run, whoever gave up.
      mbar_wait(tmem_full, 0, never, drain_ns, p.status);
    }
    griddep_wait();
  } else {
    // ---------------- decoders ----------------
    griddep_wait();                          // A is written by the previous grid
    griddep_launch_dependents();
    const int dw = warp - 2;
    const int quad = warp & 3, kq = dw >> 2;
    const int r = quad * 32 + lane;           // weight row of the tile (TMEM lane)
    const int dt = dw * 32 + lane;            // token-chunk index base
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t code_off0 = (r >> 3) * 1024 + (r & 7) * 128;
    const int cb = 2 * kq;                    // first of this thread's two 32-blocks
    const uint32_t sf_off = (cb >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (cb & 3);
    for (int i = 0; i < nk; ++i) {
      const int s = i % SB, sw = i % SW;
      // this stage's token chunks (8 BF16 each; zero beyond K), loads in flight
      // while the weights are waited for and decoded
      const int kbase = (kt0 + i) * 256;
      uint4 xv[Cf::XCH];
#pragma unroll
      for (int u = 0; u < Cf::XCH; ++u) {
        const int item = dt + u * 32 * Cf::DWARPS, n = item >> 5, k = kbase + (item & 31) * 8;
        xv[u] = (n < mvalid && k < p.K) ? ld_global_nc_v4(p.A + static_cast<long long>(m0 + n) * p.K + k)
                                        : make_uint4(0u, 0u, 0u, 0u);
      }
      if (!mbar_wait(full_w(sw), (i / SW) & 1u, abort_flag, p.wait_ns, p.status)) break;
      const uint8_t* wt = smem + Cf::OFF_W + sw * Cf::W_STAGE;
      const uint4 c0 = *reinterpret_cast<const uint4*>(wt + code_off0 + ((cb ^ (r & 7)) << 4));
      const uint4 c1 = *reinterpret_cast<const uint4*>(wt + code_off0 + (((cb + 1) ^ (r & 7)) << 4));
      const uint32_t sc = *reinterpret_cast<const uint16_t*>(smem + Cf::OFF_WSF + sw * Cf::WSF_STAGE + sf_off);
      uint32_t o[32];
      decode_two_blocks(c0, c1, sc & 0xFFu, sc >> 8, o);
      // the raw slot is free once every lane of every decoder warp has read it
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_w(sw));
      if (!mbar_wait(empty_b(s), ((i / SB) & 1) ^ 1u, abort_flag, p.wait_ns, p.status)) break;
      tc_fence_after();
      tmem_st32(t_lane + Cf::A_COL0 + s * 128 + kq * 32, o);
      uint8_t* xt = smem + Cf::OFF_X + s * Cf::X_STAGE;
#pragma unroll
      for (int u = 0; u < Cf::XCH; ++u) {
        const int item = dt + u * 32 * Cf::DWARPS, n = item >> 5, c16 = item & 31;
        if (n < mvalid) {
          // K order (0,4,1,5,2,6,3,7) within the chunk, as the weights
          const uint4 v = xv[u];
          const uint4 pv = make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                                      __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
          *reinterpret_cast<uint4*>(xt + (c16 >> 3) * (NX * 128) + (n >> 3) * 1024 + (n & 7) * 128 +
                                    (((c16 & 7) ^ (n & 7)) << 4)) = pv;
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(full_b(s));
    }

    // ---------------- epilogue ----------------
    // warps 2..5 (one per TMEM lane quadrant) drain the accumulator; with
    // split-K every decoder thread then takes part in the reduction, since
    // the DSMEM stores of one thread complete one after another
    float* red = reinterpret_cast<float*>(smem + Cf::OFF_W);   // partial [token][weight row], drained ring
    constexpr int P = 32 * Cf::DWARPS;
    if (warp < 6) {
      const int lrow = quad * 32 + lane;
      if (warp == 2 && lane == 0)
        *epi_ready = (mbar_wait(tmem_full, 0, abort_flag, p.wait_ns, p.status) && !*abort_flag && nk > 0) ? 1 : 0;
      named_bar_sync(1, 128);
      const int ready = *epi_ready;
      __syncwarp();
      tc_fence_after();
      const int n = w_tile * 128 + lrow;
      // the accumulators' sum, in accumulator order
      auto load_sum = [&](int c0, float* v) {
        tmem_ld16(t_lane + c0, v);
#pragma unroll
        for (int a = 1; a < Cf::NACC; ++a) {
          float u[16];
          tmem_ld16(t_lane + a * 32 + c0, u);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] += u[j];
        }
      };
      if (p.splits == 1) {
        if (ready) {
#pragma unroll
          for (int c0 = 0; c0 < NX; c0 += 16) {
            if (c0 < mvalid) {
              float v[16];
              load_sum(c0, v);
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < mvalid)
                  p.C[static_cast<long long>(m0 + c0 + j) * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
            }
          }
        }
      } else if (ready) {
#pragma unroll
        for (int c0 = 0; c0 < NX; c0 += 16) {
          if (c0 < mvalid) {
            float v[16];
            load_sum(c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) red[(c0 + j) * 128 + lrow] = v[j];
          }
        }
      }
    }
    if (p.splits > 1) {
      named_bar_sync(3, P);                    // partial staged, readiness published
      const int ready = *epi_ready;
      cluster_wait();                          // every owner's mbarrier is initialised
      cluster_waited = true;
      const int S = p.splits;
      const uint32_t rank = cluster_ctarank();
      const int G = mvalid * 32;               // float4 groups of the valid partial
      const int slot = (G + S - 1) / S;
      const float4* red4 = reinterpret_cast<const float4*>(red);
      // group g belongs to owner o = max{o : floor(o*G/S) <= g}; sent whatever
      // happened before, so that every owner's byte count completes
      for (int g = dt; g < G; g += P) {
        const int o = static_cast<int>((static_cast<long long>(g + 1) * S - 1) / G);
        const int og0 = static_cast<int>(static_cast<long long>(o) * G / S);
        const uint32_t dst = cluster_map_shared(
            base + Cf::OFF_PUSH + static_cast<uint32_t>((static_cast<int>(rank) * slot + (g - og0)) * 16),
            static_cast<uint32_t>(o));
        st_async_v4(dst, red4[g], cluster_map_shared(red_bar, static_cast<uint32_t>(o)));
      }
      // this CTA's slice: wait for all S x slice bytes (the limit exceeds any
      // peer's bounded path to its stores), sum the slots in rank order
      if (dt == 0) {
        const unsigned long long lim = 32ull * (p.wait_ns > drain_ns ? p.wait_ns : drain_ns);
        *owner_ready = mbar_wait_cluster(red_bar, 0, lim, p.status) && ready ? 1 : 0;
      }
      named_bar_sync(3, P);
      if (*owner_ready) {
        const int g0 = static_cast<int>(static_cast<long long>(rank) * G / S);
        const int g1 = static_cast<int>(static_cast<long long>(rank + 1) * G / S);
        const float4* push = reinterpret_cast<const float4*>(smem + Cf::OFF_PUSH);
        for (int g = g0 + dt; g < g1; g += P) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int c = 0; c < S; ++c) {
            const float4 v = push[c * slot + (g - g0)];
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
          }
          const int t = g >> 5, r4 = (g & 31) * 4;
          uint2 ov;
          ov.x = (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.y))) << 16) |
                 __bfloat16_as_ushort(__float2bfloat16_rn(acc.x));
          ov.y = (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.w))) << 16) |
                 __bfloat16_as_ushort(__float2bfloat16_rn(acc.z));
          *reinterpret_cast<uint2*>(p.C + static_cast<long long>(m0 + t) * p.N + w_tile * 128 + r4) = ov;
        }
      }
    }
  }

  if (p.splits > 1 && !cluster_waited) cluster_wait();

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, Cf::TMEM_COLS);
  }
}

constexpr int kRing = 6;   // 256-wide K tiles of weights in flight per CTA

template <int NX>
int set_attrs() {
  using Cf = HCfg<NX, kRing>;
  auto kern = a4w4_a16w4_kernel<NX, kRing>;
  static std::atomic<unsigned long long> attr_devs{0};   // bit d: attributes set on device d
  return ensure_func_attrs(attr_devs, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM_BYTES) == cudaSuccess &&
           cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  });
}

// Clusters of `splits` CTAs (one per SM) that can be resident at once.
template <int NX>
int active_clusters(int splits) {
  using Cf = HCfg<NX, kRing>;
  if (set_attrs<NX>() != 0) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, static_cast<unsigned>(splits));
  cfg.blockDim = dim3(Cf::THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cf::SMEM_BYTES;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 1;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = static_cast<unsigned>(splits);
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, a4w4_a16w4_kernel<NX, kRing>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// active_clusters per (device, token tile, splits), filled on first use
// (0: not known yet)
constexpr int kMaxDevices = 64;
std::atomic<int> g_active[kMaxDevices][2][kMaxA16W4Splits + 1];

int active_clusters_cached(int nx, int splits) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::atomic<int>* slot = (dev >= 0 && dev < kMaxDevices) ? &g_active[dev][nx == 16 ? 0 : 1][splits] : nullptr;
  int v = slot != nullptr ? slot->load(std::memory_order_relaxed) : 0;
  if (v == 0) {
    v = nx == 16 ? active_clusters<16>(splits) : active_clusters<32>(splits);
    if (v > 0 && slot != nullptr) slot->store(v, std::memory_order_relaxed);
  }
  return v;
}

template <int NX>
int launch_cfg(const A16W4Args& a, dim3 grid, cudaStream_t st) {
  using Cf = HCfg<NX, kRing>;
  if (set_attrs<NX>() != 0) return -4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Cf::THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cf::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (a.splits > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = 1;
    attrs[n].val.clusterDim.y = 1;
    attrs[n].val.clusterDim.z = static_cast<unsigned>(a.splits);
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  if (cudaLaunchKernelEx(&cfg, a4w4_a16w4_kernel<NX, kRing>, a) != cudaSuccess) return -4;
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace

// Split-K for one CTA per SM: the split count s (at most the K tiles and 16)
// that minimises (waves of clusters) x (K tiles of the longest split + 2), where a
// wave is as many clusters of s CTAs as the device can hold at once (clusters
// are placed within a GPC, so large ones leave SMs idle); ties go to fewer
// splits (less reduction traffic).
GemmPlan plan_a16w4(int M, int N, int K, int sms) {
  GemmPlan pl{};
  pl.kt = (K + 255) / 256;
  pl.swap_ab = 1;
  pl.nx = M <= 16 ? 16 : 32;
  pl.w_tiles = N / 128;
  pl.x_tiles = (M + pl.nx - 1) / pl.nx;
  const long long tiles = static_cast<long long>(pl.w_tiles) * pl.x_tiles;
  int best = 1;
  long long best_cost = -1;
  const int smax = pl.kt < kMaxA16W4Splits ? pl.kt : kMaxA16W4Splits;
  for (int s = 1; s <= smax; ++s) {
    const int act = s == 1 ? sms : active_clusters_cached(pl.nx, s);
    if (act <= 0) continue;
    const long long waves = (tiles + act - 1) / act;
    // a CTA's fixed cost (start-up, first weight fetch, reduction) is about
    // two K tiles' worth of decoding
    const long long cost = waves * ((pl.kt + s - 1) / s + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  pl.splits = best;
  pl.cluster_reduce = best > 1;
  return pl;
}

int launch_a16w4(const GemmPlan& pl, const void* A, int M, int K, const void* Wq, const void* Ws, int N, void* C,
                 cudaStream_t st, unsigned long long wait_ns, unsigned int* status, int prefetch_w) {
  if (pl.splits < 1 || pl.splits > kMaxA16W4Splits) return -4;
  A16W4Args a{};
  a.A = static_cast<const uint16_t*>(A);
  a.Wq = static_cast<const uint8_t*>(Wq);
  a.Ws = static_cast<const uint8_t*>(Ws);
  a.C = static_cast<uint16_t*>(C);
  a.M = M; a.N = N; a.K = K; a.KT = pl.kt; a.splits = pl.splits;
  a.prefetch_w = prefetch_w;
  a.wait_ns = wait_ns;
  a.status = status;
  const dim3 grid(pl.w_tiles, pl.x_tiles, pl.splits);
  return pl.nx == 16 ? launch_cfg<16>(a, grid, st) : launch_cfg<32>(a, grid, st);
}

}  // namespace a4w4
