// decode.cu -- decode-size dense A4W4 GEMM (M <= 16; M <= 32 when one CTA
// holds a whole K range): weights stream at HBM rate through the tcgen05
// block-scaled MMA with the tokens on its N side.
//
// "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM", Summary/Implementation:
// BF16 activations quantised inline to MXFP4 and multiplied with preshuffled
// MXFP4 weights, fp32 accumulation, BF16 output with M-tail masking.
//
// Layout of the work: the 128-row weight tile of CTA (w_tile, x_tile, split)
// is the MMA's A operand (M = 128), up to NX tokens its B operand, and the K
// range is split over the `splits` CTAs of a thread-block cluster.  Shapes are
// planned so that a CTA's whole K range fits its SW-deep weight ring, so every
// weight copy is issued at once; with weight prefetch on, before the grid
// dependency resolves, i.e. while the previous kernel on the stream still runs.
//
//   warp 0      weight producer: 16 KB + 1 KB bulk copies per 256-wide K tile;
//   warp 1      TMEM owner and MMA issuer: copies each weight tile's scale
//               atoms to TMEM as soon as they land (before the activations
//               exist), then per K tile one activation scale copy and four
//               tcgen05.mma.kind::mxf4.block_scale (K = 64 each);
//   warps 2..   activation producers: rounds of up to SX K tiles, their
//               (tile, token row, 32-block) items spread over all producer
//               threads with the BF16 loads in flight together, E8M0 + E2M1
//               quantisation into the SX-deep operand ring, one proxy fence
//               per round; the first four then drain TMEM and reduce the
//               split-K partials over DSMEM.
//
// Split-K reduction (splits > 1): the CTAs of a cluster each own a slice of
// the tile's outputs (float4 groups of [token][weight row]).  Every CTA parks
// its fp32 partial in its drained weight ring and sends each group, one
// thread per group, with st.async into the owning CTA's push buffer (slot =
// sender's cluster rank); the stores count their bytes on the owner's
// mbarrier, whose expected byte count the owner set at start-up.  An owner
// waits for all bytes, sums the slots in rank order (bitwise deterministic)
// and writes BF16.  Remote stores of one thread complete one after another,
// so the work is spread over all threads; no CTA reads a peer's shared
// memory, and a CTA leaves only after every byte destined to it has landed.
// One split cluster barrier (arrive at set-up, wait before the first store)
// guarantees every owner's mbarrier exists before anyone stores.
#include "device.cuh"
#include "launch.h"

namespace a4w4 {

struct DecodeArgs {
  const uint16_t* A;   // activations [M, K] BF16
  const uint8_t* Wq;   // preshuffled weight codes
  const uint8_t* Ws;   // preshuffled weight scales
  uint16_t* C;         // [M, N] BF16
  int M, N, K, KT, splits;
  int prefetch_w;      // 1: weights may be read before the previous grid on the stream completes
  unsigned long long wait_ns;
  unsigned int* status;
  // test hook (ActDump): the CTAs of weight tile 0 also store the activation
  // tiles their producers build; nullptr in every product call
  uint8_t* dump_codes;
  uint8_t* dump_scales;
};

template <int NX, int SW, int SX>
struct DCfg {
  static constexpr int QWARPS = NX <= 16 ? 4 : 8;                // activation producer warps
  static constexpr int THREADS = 64 + 32 * QWARPS;
  static constexpr int W_STAGE = 16384, WSF_STAGE = 1024;
  static constexpr int X_STAGE = NX * 128;
  static constexpr int XSF_STAGE = 1024;                          // 2 atoms (K halves) x 512 B
  static constexpr int OFF_W = 0;
  static constexpr int OFF_X = OFF_W + SW * W_STAGE;
  static constexpr int OFF_WSF = OFF_X + SX * X_STAGE;
  static constexpr int OFF_XSF = OFF_WSF + SW * WSF_STAGE;
  // push buffer: up to 16 rank slots of ceil(G / S) float4 groups, G = 32 x tokens
  // (S * ceil(G / S) <= G + S groups)
  static constexpr int PUSH_BYTES = NX * 512 + 256;
  static constexpr int OFF_PUSH = OFF_XSF + SX * XSF_STAGE;
  static constexpr int OFF_BAR = OFF_PUSH + PUSH_BYTES;
  static constexpr int NBAR = 2 * SW + 4;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 32 + 1024;       // + slack to align the base to 1024
  static constexpr int MIN_BLOCKS_SMEM = 233472 / (SMEM_BYTES + 1024);
  static constexpr int MIN_BLOCKS = MIN_BLOCKS_SMEM >= 3 ? 3 : (MIN_BLOCKS_SMEM >= 2 ? 2 : 1);
  static constexpr int ACC_COLS = NX;
  static constexpr int WSF_COLS = 8;                              // per weight stage: 2 atoms x 4 columns
  static constexpr int XSF_COLS = 8;                              // scale columns start 4-aligned
  static constexpr int WSF_COL0 = ACC_COLS;
  static constexpr int XSF_COL0 = WSF_COL0 + SW * WSF_COLS;
  static constexpr int TMEM_NEED = XSF_COL0 + SX * XSF_COLS;
  static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128 : 256;
  static constexpr int A_CHUNK = 4;                               // A blocks a producer thread keeps in flight
  static_assert(NX % 16 == 0 && NX <= 128, "token tile");
  static_assert(SW >= 2 && SX >= 2 && SX <= SW, "rings");
  static_assert(TMEM_NEED <= 256, "TMEM budget");
  static_assert(MIN_BLOCKS * TMEM_COLS <= 512, "co-resident CTAs must fit in TMEM");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(NX * 128 * 4 <= SW * W_STAGE, "a staged partial must fit in the drained weight ring");
};

template <int NX, int SW, int SX>
__global__ void __launch_bounds__(DCfg<NX, SW, SX>::THREADS, DCfg<NX, SW, SX>::MIN_BLOCKS)
    a4w4_decode_kernel(const DecodeArgs p) {
  using Cf = DCfg<NX, SW, SX>;
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
  // the activation ring is filled and drained in rounds of up to SX K tiles:
  // one full / one empty barrier whose phases alternate per round
  const uint32_t full_x = bar0 + 8u * (2 * SW);
  const uint32_t empty_x = full_x + 8u;
  const uint32_t tmem_full = empty_x + 8u;
  const uint32_t red_bar = tmem_full + 8u;   // peers' pushes into this CTA's slice
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cf::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cf::OFF_MISC + 8);
  volatile int* never = reinterpret_cast<volatile int*>(smem + Cf::OFF_MISC + 16);
  volatile int* epi_ready = reinterpret_cast<volatile int*>(smem + Cf::OFF_MISC + 24);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(full_w(s), 1);
      mbar_init(empty_w(s), 1);
    }
    mbar_init(full_x, Cf::QWARPS * 32);
    mbar_init(empty_x, 1);
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
  // Token rows beyond M are never written by the producers: their codes and
  // scales are zeroed here once for every operand slot.
  for (int i = threadIdx.x; i < SX * Cf::X_STAGE / 16; i += Cf::THREADS)
    reinterpret_cast<uint4*>(smem + Cf::OFF_X)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < SX * Cf::XSF_STAGE / 16; i += Cf::THREADS)
    reinterpret_cast<uint4*>(smem + Cf::OFF_XSF)[i] = make_uint4(0u, 0u, 0u, 0u);
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
    named_bar_arrive(2, 32 + 128);
  }

  if (warp == 0) {
    // ---------------- weight producer ----------------
    // Later ring passes wait for MMAs, hence for the activations: nothing is
    // lost by taking the grid dependency here.
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
    // The weight scale copies need only the weights, so they run as soon as a
    // weight tile lands; everything touching the activations waits for the
    // previous grid (through the producers' full_x barriers).
    griddep_launch_dependents();
    if (lane == 0) {
      const uint64_t adesc0 = sdesc_sw128(base + Cf::OFF_W), bdesc0 = sdesc_sw128(base + Cf::OFF_X);
      const uint64_t wsfd0 = sdesc_sf(base + Cf::OFF_WSF), xsfd0 = sdesc_sf(base + Cf::OFF_XSF);
      const uint32_t idesc0 = idesc_mxf4(NX, 0, 0), idesc2 = idesc_mxf4(NX, 2, 2);
      const uint32_t wsf_col = tmem + Cf::WSF_COL0, xsf_col = tmem + Cf::XSF_COL0;
      bool ok = true;
      auto copy_w_sf = [&](int i) {
        const int s = i % SW;
        if (!mbar_wait(full_w(s), (i / SW) & 1u, abort_flag, p.wait_ns, p.status)) return false;
        tc_fence_after();
        const uint64_t d = wsfd0 + ((s * Cf::WSF_STAGE) >> 4);
        tmem_copy_sf_desc(wsf_col + s * Cf::WSF_COLS, d);
        tmem_copy_sf_desc(wsf_col + s * Cf::WSF_COLS + 4, d + (512 >> 4));
        return true;
      };
      const int pre = nk < SW ? nk : SW;
      for (int i = 0; i < pre && ok; ++i) ok = copy_w_sf(i);
      for (int r0 = 0, rnd = 0; r0 < nk && ok; r0 += SX, ++rnd) {
        const int ns = nk - r0 < SX ? nk - r0 : SX;
        for (int j = 0; j < ns && ok; ++j)
          if (r0 + j >= pre) ok = copy_w_sf(r0 + j);
        if (!ok || !mbar_wait(full_x, static_cast<uint32_t>(rnd & 1), abort_flag, p.wait_ns, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int j = 0; j < ns; ++j) {
          const int i = r0 + j, sw = i % SW;
          const uint64_t xd = xsfd0 + ((j * Cf::XSF_STAGE) >> 4);
          tmem_copy_sf_desc(xsf_col + j * Cf::XSF_COLS, xd);
          tmem_copy_sf_desc(xsf_col + j * Cf::XSF_COLS + 4, xd + (512 >> 4));
          const uint64_t ad = adesc0 + ((sw * Cf::W_STAGE) >> 4), bd = bdesc0 + ((j * Cf::X_STAGE) >> 4);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const int ka = ks >> 1;
            mma_mxf4(tmem, ad + ks * 2, bd + ks * 2, (ks & 1) ? idesc2 : idesc0, wsf_col + sw * Cf::WSF_COLS + ka * 4,
                     xsf_col + j * Cf::XSF_COLS + ka * 4, (i > 0 || ks > 0) ? 1u : 0u);
          }
          // a weight slot is handed back only if a later K tile will refill it
          if (i + SW < nk) mma_commit(empty_w(sw));
        }
        if (r0 + SX < nk) mma_commit(empty_x);
      }
      mma_commit(tmem_full);
      // TMEM is never released while MMAs may still run, whoever gave up.
      mbar_wait(tmem_full, 0, never, drain_ns, p.status);
    }
    griddep_wait();
  } else {
    // ---------------- activation producers ----------------
    griddep_wait();                          // A is written by the previous grid
    griddep_launch_dependents();
    // Work items are (K tile, valid token row, 32-block) triples of a round
    // of up to SX K tiles, spread over all producer threads (rows beyond M
    // are never touched: zeroed at set-up), loaded CH at a time with all
    // loads in flight; one proxy fence and one arrival per round.
    const int qt = threadIdx.x - 64;
    constexpr int P = Cf::QWARPS * 32;
    constexpr int CH = Cf::A_CHUNK;
    const int blk = mvalid * 8;                    // valid blocks per stage
    const bool dump = p.dump_codes != nullptr && w_tile == 0;
    bool stop = false;
    for (int r0 = 0, rnd = 0; r0 < nk && !stop; r0 += SX, ++rnd) {
      const int ns = nk - r0 < SX ? nk - r0 : SX;
      const int total = ns * blk;
      bool waited = rnd == 0;
      for (int t0 = qt; t0 < total && !stop; t0 += CH * P) {
        uint32_t w[CH][16];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int t = t0 + c * P;
          const int j = t / blk, rb = t - j * blk;
          const int k = (kt0 + r0 + j) * 256 + (rb & 7) * 32;
          if (t < total && k < p.K) {
            const uint4* src = reinterpret_cast<const uint4*>(p.A + static_cast<long long>(m0 + (rb >> 3)) * p.K + k);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 v = ld_global_nc_v4(src + q);
              w[c][4 * q] = v.x; w[c][4 * q + 1] = v.y; w[c][4 * q + 2] = v.z; w[c][4 * q + 3] = v.w;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) w[c][q] = 0u;
          }
        }
        // the ring's slots are reused from the second round on: wait (once,
        // with the first chunk's loads already in flight) for the MMAs of the
        // previous round
        if (!waited) {
          waited = true;
          if (!mbar_wait(empty_x, static_cast<uint32_t>((rnd - 1) & 1), abort_flag, p.wait_ns, p.status)) {
            stop = true;
            break;
          }
        }
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int t = t0 + c * P;
          if (t < total) {
            const int j = t / blk, rb = t - j * blk;
            const int r = rb >> 3, kb = rb & 7;
            uint8_t* xt = smem + Cf::OFF_X + j * Cf::X_STAGE;
            uint8_t* xs = smem + Cf::OFF_XSF + j * Cf::XSF_STAGE;
            uint32_t code[4];
            const uint32_t e = quant32_bf16(w[c], code);
            const uint32_t code_off = (r >> 3) * 1024 + (r & 7) * 128 + ((kb ^ (r & 7)) << 4);
            const uint32_t sf_off = (kb >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (kb & 3);
            const uint4 cv = make_uint4(code[0], code[1], code[2], code[3]);
            *reinterpret_cast<uint4*>(xt + code_off) = cv;
            xs[sf_off] = static_cast<uint8_t>(e);
            if (dump) {
              // test hook: the same bytes at the same offsets of a global copy
              const long long atom = static_cast<long long>(x_tile) * p.KT + kt0 + r0 + j;
              *reinterpret_cast<uint4*>(p.dump_codes + atom * Cf::X_STAGE + code_off) = cv;
              p.dump_scales[atom * Cf::XSF_STAGE + sf_off] = static_cast<uint8_t>(e);
            }
          }
        }
      }
      // every thread, with items or not, arrives for round rnd only after
      // round rnd-1 was consumed, so no arrival can count toward an earlier phase
      if (!stop && !waited && !mbar_wait(empty_x, static_cast<uint32_t>((rnd - 1) & 1), abort_flag, p.wait_ns, p.status))
        stop = true;
      if (stop) break;
      fence_proxy_async_smem();
      mbar_arrive(full_x);
    }

    // ---------------- epilogue ----------------
    // warps 2..5 (one per TMEM lane quadrant) drain the accumulator; with
    // split-K every producer thread then takes part in the reduction, since
    // the DSMEM stores of one thread complete one after another
    volatile int* owner_ready = reinterpret_cast<volatile int*>(smem + Cf::OFF_MISC + 28);
    float* red = reinterpret_cast<float*>(smem + Cf::OFF_W);   // partial [token][weight row], drained ring
    if (warp < 6) {
      named_bar_sync(2, 32 + 128);             // TMEM address published by the MMA warp
      tc_fence_after();
      tmem = *tmem_slot;
      const int q = warp & 3;
      const int lrow = q * 32 + lane;
      const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
      if (warp == 2 && lane == 0)
        *epi_ready = (mbar_wait(tmem_full, 0, abort_flag, p.wait_ns, p.status) && !*abort_flag && nk > 0) ? 1 : 0;
      named_bar_sync(1, 128);
      const int ready = *epi_ready;
      __syncwarp();
      tc_fence_after();
      const int n = w_tile * 128 + lrow;
      if (p.splits == 1) {
        if (ready) {
#pragma unroll
          for (int c0 = 0; c0 < NX; c0 += 16) {
            if (c0 < mvalid) {
              float v[16];
              tmem_ld16(tq + c0, v);
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
            tmem_ld16(tq + c0, v);
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
      const int et = qt;
      const uint32_t rank = cluster_ctarank();
      const int G = mvalid * 32;                   // float4 groups of the valid partial
      const int slot = (G + S - 1) / S;
      const float4* red4 = reinterpret_cast<const float4*>(red);
      // group g belongs to owner o = max{o : floor(o*G/S) <= g}; sent whatever
      // happened before, so that every owner's byte count completes
      for (int g = et; g < G; g += P) {
        const int o = static_cast<int>((static_cast<long long>(g + 1) * S - 1) / G);
        const int og0 = static_cast<int>(static_cast<long long>(o) * G / S);
        const uint32_t dst = cluster_map_shared(
            base + Cf::OFF_PUSH + static_cast<uint32_t>((static_cast<int>(rank) * slot + (g - og0)) * 16), static_cast<uint32_t>(o));
        st_async_v4(dst, red4[g], cluster_map_shared(red_bar, static_cast<uint32_t>(o)));
      }
      // this CTA's slice: wait for all S x slice bytes (the limit exceeds any
      // peer's bounded path to its stores), sum the slots in rank order
      if (et == 0) {
        const unsigned long long lim = 32ull * (p.wait_ns > drain_ns ? p.wait_ns : drain_ns);
        *owner_ready = mbar_wait_cluster(red_bar, 0, lim, p.status) && ready ? 1 : 0;
      }
      named_bar_sync(3, P);
      if (*owner_ready) {
        const int g0 = static_cast<int>(static_cast<long long>(rank) * G / S);
        const int g1 = static_cast<int>(static_cast<long long>(rank + 1) * G / S);
        const float4* push = reinterpret_cast<const float4*>(smem + Cf::OFF_PUSH);
        for (int g = g0 + et; g < g1; g += P) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int c = 0; c < S; ++c) {
            const float4 v = push[c * slot + (g - g0)];
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
          }
          const int t = g >> 5, r4 = (g & 31) * 4;
          uint2 o;
          o.x = (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.y))) << 16) |
                __bfloat16_as_ushort(__float2bfloat16_rn(acc.x));
          o.y = (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.w))) << 16) |
                __bfloat16_as_ushort(__float2bfloat16_rn(acc.z));
          *reinterpret_cast<uint2*>(p.C + static_cast<long long>(m0 + t) * p.N + w_tile * 128 + r4) = o;
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

template <int NX, int SW, int SX>
static int launch_decode_cfg(const DecodeArgs& a, dim3 grid, cudaStream_t st) {
  using Cf = DCfg<NX, SW, SX>;
  auto kern = a4w4_decode_kernel<NX, SW, SX>;
  static std::atomic<unsigned long long> attr_devs{0};   // bit d: attributes set on device d
  if (ensure_func_attrs(attr_devs, [&] {
        // clusters of up to 16 CTAs (more than the portable 8)
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM_BYTES) ==
                   cudaSuccess &&
               cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
      }) != 0)
    return -4;
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
  if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return -4;
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int launch_decode(const GemmPlan& pl, const void* A, int M, int K, const void* Wq, const void* Ws, int N, void* C,
                  cudaStream_t st, unsigned long long wait_ns, unsigned int* status, int prefetch_w, ActDump dump) {
  if (pl.splits < 1 || pl.splits > 16) return -4;   // push buffer and cluster limits
  DecodeArgs a{};
  a.A = static_cast<const uint16_t*>(A);
  a.Wq = static_cast<const uint8_t*>(Wq);
  a.Ws = static_cast<const uint8_t*>(Ws);
  a.C = static_cast<uint16_t*>(C);
  a.M = M; a.N = N; a.K = K; a.KT = pl.kt; a.splits = pl.splits;
  a.prefetch_w = prefetch_w;
  a.dump_codes = dump.codes;
  a.dump_scales = dump.scales;
  a.wait_ns = wait_ns;
  a.status = status;
  const dim3 grid(pl.w_tiles, pl.x_tiles, pl.splits);
  switch (pl.nx * 8 + pl.ring) {
    case 16 * 8 + 3: return launch_decode_cfg<16, 3, 3>(a, grid, st);
    case 16 * 8 + 4: return launch_decode_cfg<16, 4, 4>(a, grid, st);
    case 32 * 8 + 4: return launch_decode_cfg<32, 4, 4>(a, grid, st);
    default: return -4;
  }
}

}  // namespace a4w4
