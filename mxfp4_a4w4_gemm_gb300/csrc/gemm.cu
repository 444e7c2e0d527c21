// gemm.cu -- warp-specialised tcgen05 block-scaled MXFP4 GEMM (sm_103a).
//
// "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM", Summary/Implementation:
// BF16 activations quantised inline to MXFP4 and multiplied with preshuffled
// MXFP4 weights on the scaled-FP4 tensor cores, BF16 direct output with M-tail
// masking.  "[gfx1250] Fuse A4W4 stage1 FP4 quantization", Summary: the MoE
// GEMM1 variant emits MXFP4 codes + E8M0 scales after SwiGLU.
//
// One CTA computes a (weight rows) x (activation rows) tile over a K range:
//   warp 0      TMA producer: 16 KB bulk copies of preshuffled weight tiles
//               and their 1 KB scale atoms into a STAGES-deep smem ring;
//   warp 1      allocates TMEM, copies each stage's scale atoms smem->TMEM
//               (tcgen05.cp) and issues tcgen05.mma.kind::mxf4.block_scale
//               (M=128, K=64 per instruction, 4 per 256-wide stage), then
//               tcgen05.commit to free the stage;
//   warps 2..   activation producers: 16-byte BF16 loads, per-32-block amax,
//               E8M0 + E2M1 round-to-nearest-even into the 128-byte-swizzled
//               smem operand tile and the 128x4 scale atom; the first four
//               of them then run the epilogue (tcgen05.ld -> BF16 -> global,
//               or split-K partials, or SwiGLU + MXFP4 requant for MoE).
// Swap-AB (small M): the weights are the MMA's 128-row A operand and the
// tokens its N side (16..128), so the tensor core does no work on padding
// rows and the kernel streams weights at HBM rate; the K range is split over
// the SMs and the last CTA of a tile sums the fp32 partials in split order.
#include "device.cuh"
#include "launch.h"

namespace a4w4 {

// kSwap: weights x inline-quantised tokens (17 <= M <= 128; larger M runs in
// the persistent kernel of large.cu); kMoe: inline-quantised gathered sorted
// rows x an expert's weights with the SwiGLU / SiLU + requant epilogue;
// kMoePre: kMoe gathering rows that were quantised once beforehand (plain
// MXFP4 layout) instead of quantising them per tile.  (MoE GEMM2 runs in the
// persistent kernel of moe2.cu.)
enum Mode { kSwap = 0, kMoe = 1, kMoePre = 2 };

// MoE GEMM1 epilogue activation (a4w4.h: A4W4_MOE_ACT_*)
constexpr int kActSwiglu = 0, kActSilu = 1;

struct GemmArgs {
  const uint16_t* A;  // dense: activations [M, K]; MoE: tokens X [T, D]
  const uint8_t* Aq;  // kMoePre: tokens quantised once, MXFP4 codes [T, K/2]
  const uint8_t* As;  // kMoePre: their E8M0 scales [T, K/32]
  const uint8_t* Wq;
  const uint8_t* Ws;
  uint16_t* C;        // [M, N] BF16
  int M, N, K, KT, splits, w_tiles;
  int cluster_reduce;   // 1: the `splits` CTAs of a tile form a cluster and reduce over DSMEM
  int prefetch_w;       // 1: weights may be read before the previous grid on the stream completes
  unsigned long long wait_ns;
  unsigned int* status;
  // MoE GEMM1
  const int32_t* sorted_rows;
  const int32_t* block_expert;
  const int32_t* num_blocks;
  int topk, routed_rows, I, E;
  long long expert_code_bytes, expert_sf_bytes;
  uint8_t* out_q;
  uint8_t* out_s;
  int act;              // kActSwiglu or kActSilu
  int out_tiles;        // 1: GEMM1 output in sorted-slot operand tiles (KT_out K tiles per block)
  int KT_out;
  // test hook (ActDump): the CTAs of weight tile 0 also store the activation
  // tiles their producers build; nullptr in every product call
  uint8_t* dump_codes;
  uint8_t* dump_scales;
};

constexpr int kMaxClusterSplits = 8;  // portable cluster size
constexpr int kMaxDecodeSplits = 16;  // decode kernel: non-portable clusters (a GPC holds at least 16 SMs)

template <int MODE, int NX, int STAGES>
struct Cfg {
  static constexpr bool kSwapAB = MODE == kSwap;
  static constexpr int NW = kSwapAB ? 128 : 256;                 // weight rows per CTA
  static constexpr int W_ATOMS = NW / 128;
  static constexpr int MMA_N = kSwapAB ? NX : NW;
  static constexpr bool kMoeAny = MODE == kMoe || MODE == kMoePre;  // MoE GEMM1
  static constexpr bool kRouted = kMoeAny;                       // blocks of sorted routed rows
  static constexpr bool kGatherQ = MODE == kMoePre;              // producers copy pre-quantised rows
  static constexpr int QWARPS = (kSwapAB && NX <= 32) ? 4 : 8;   // producer warps
  // epilogue warps (the first of the producer warps): MoE's SwiGLU + requant
  // epilogue splits each TMEM lane quadrant's columns over two warps
  static constexpr int EPI_WARPS = kMoeAny ? 8 : 4;
  static constexpr int EPI_THREADS = EPI_WARPS * 32;
  static constexpr int THREADS = 32 * (2 + QWARPS);
  static constexpr int MIN_BLOCKS = (kSwapAB && NX <= 16) ? 3 : (kSwapAB && NX <= 32) ? 2 : 1;
  static constexpr int W_CODE_BYTES = W_ATOMS * 16384;
  static constexpr int X_CODE_BYTES = NX * 128;
  static constexpr int W_SF_BYTES = W_ATOMS * 1024;
  static constexpr int X_SF_BYTES = 1024;
  static constexpr int OFF_W = 0;
  static constexpr int OFF_X = OFF_W + STAGES * W_CODE_BYTES;
  static constexpr int OFF_WSF = OFF_X + STAGES * X_CODE_BYTES;
  static constexpr int OFF_XSF = OFF_WSF + STAGES * W_SF_BYTES;
  // swap-AB split-K: peers push fp32 partial slices here (owner-indexed slots)
  static constexpr int PUSH_BYTES = kSwapAB ? (NX + 8) * 512 : 0;
  static constexpr int OFF_PUSH = OFF_XSF + STAGES * X_SF_BYTES;
  static constexpr int OFF_BAR = OFF_PUSH + PUSH_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + (3 * STAGES + 1) * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 32 + 1024;       // + slack to align the base to 1024
  static constexpr int ACC_COLS = MMA_N;
  static constexpr int SFA_COLS = 8;                             // 2 K-atoms x 4 columns
  static constexpr int SFB_COLS = 8 * ((MMA_N + 127) / 128);
  static constexpr int SF_STAGE_COLS = SFA_COLS + SFB_COLS;
  static constexpr int TMEM_NEED = ACC_COLS + STAGES * SF_STAGE_COLS;
  static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128 : (TMEM_NEED <= 256 ? 256 : 512);
  static constexpr int BLOCKS_PER_STAGE = NX * 8;                // (row, 32-block) pairs
  static constexpr int PER_THREAD = (BLOCKS_PER_STAGE + QWARPS * 32 - 1) / (QWARPS * 32);
  static constexpr int A_DEPTH = PER_THREAD == 1 ? 4 : 2;        // stages of A loads in flight per thread
  static_assert(NX % 16 == 0 && NX <= 128, "activation tile");
  static_assert(TMEM_NEED <= 512, "TMEM budget");
  static_assert(MIN_BLOCKS * TMEM_COLS <= 512, "co-resident CTAs must fit in TMEM");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(MIN_BLOCKS * (SMEM_BYTES + 1024) <= 233472, "co-resident CTAs must fit in shared memory");
  static_assert(!kSwapAB || NX * 128 * 4 <= OFF_PUSH, "a staged split-K partial must fit in the drained ring");
};

template <int MODE, int NX, int STAGES>
__global__ void __launch_bounds__(Cfg<MODE, NX, STAGES>::THREADS, Cfg<MODE, NX, STAGES>::MIN_BLOCKS)
    a4w4_gemm_kernel(const GemmArgs p) {
  using Cf = Cfg<MODE, NX, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int w_tile = blockIdx.x;
  const int x_tile = blockIdx.y;
  const int split = blockIdx.z;

  int expert = 0;
  if (Cf::kRouted) {
    griddep_wait();                                // the sort that wrote num_blocks has finished
    if (x_tile >= *p.num_blocks) return;           // block does not exist for this routing
    expert = p.block_expert[x_tile];
    if (expert < 0 || expert >= p.E) return;
  }
  const int kt0 = static_cast<int>(static_cast<long long>(split) * p.KT / p.splits);
  const int kt1 = static_cast<int>(static_cast<long long>(split + 1) * p.KT / p.splits);
  const int nk = kt1 - kt0;
  // Waits that only drain work already in flight (bulk copies landing in this
  // CTA's shared memory, MMAs reading TMEM) before the CTA releases them keep
  // a floor of 0.1 s whatever limit the caller set for ordinary waits.
  const unsigned long long drain_ns = p.wait_ns > 100000000ull ? p.wait_ns : 100000000ull;

  const uint32_t bar0 = base + Cf::OFF_BAR;
  auto full_w = [&](int s) { return bar0 + 8u * s; };
  auto full_x = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto empty = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
  const uint32_t tmem_full = bar0 + 8u * (3 * STAGES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cf::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cf::OFF_MISC + 8);
  volatile int* never = reinterpret_cast<volatile int*>(smem + Cf::OFF_MISC + 24);
  volatile int* epi_ready = reinterpret_cast<volatile int*>(smem + Cf::OFF_MISC + 28);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_w(s), 1);
      mbar_init(full_x(s), Cf::QWARPS * 32);
      mbar_init(empty(s), 1);
    }
    mbar_init(tmem_full, 1);
    *abort_flag = 0;
    *never = 0;
    *epi_ready = 0;
    fence_barrier_init();
  }
  // Activation rows that do not exist (beyond M, or padding of a routed
  // block) are never written by the producers: their codes and scales are
  // zeroed here once for every stage.
  for (int i = threadIdx.x; i < STAGES * Cf::X_CODE_BYTES / 16; i += Cf::THREADS)
    reinterpret_cast<uint4*>(smem + Cf::OFF_X)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < STAGES * Cf::X_SF_BYTES / 16; i += Cf::THREADS)
    reinterpret_cast<uint4*>(smem + Cf::OFF_XSF)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  __syncthreads();                                 // barriers initialised
  // Start streaming weights before TMEM allocation: the first ring pass needs
  // no empty-slot wait (fresh barriers).
  const uint8_t* wq_e = p.Wq + static_cast<long long>(expert) * p.expert_code_bytes;
  const uint8_t* ws_e = p.Ws + static_cast<long long>(expert) * p.expert_sf_bytes;
  // Swap-AB and MoE GEMM1 stream every weight byte once.
  const uint64_t pol = policy_evict_first();
  auto issue_stage = [&](int i) {
    const int s = i % STAGES;
    mbar_arrive_expect_tx(full_w(s), Cf::W_ATOMS * (16384 + 1024));
    // the W_ATOMS atoms of this K tile are adjacent (weight_atom): one copy
    // of codes, one of scales
    const long long watom = weight_atom(w_tile * Cf::W_ATOMS, kt0 + i, p.KT);
    bulk_g2s(base + Cf::OFF_W + s * Cf::W_CODE_BYTES, wq_e + watom * 16384, Cf::W_ATOMS * 16384, full_w(s), pol);
    bulk_g2s(base + Cf::OFF_WSF + s * Cf::W_SF_BYTES, ws_e + watom * 1024, Cf::W_ATOMS * 1024, full_w(s), pol);
  };
  int issued = 0;
  if (warp == 0 && lane == 0) {
    // Weights are read before the grid dependency resolves only on request
    // (the previous kernel on the stream must not write them).
    if (!p.prefetch_w) griddep_wait();
    issued = nk < STAGES ? nk : STAGES;
    for (int i = 0; i < issued; ++i) issue_stage(i);
  }
  // TMEM is allocated off the data path: the MMA warp allocates and signals
  // the epilogue warps through a named barrier (arrive: non-blocking).
  uint32_t tmem = 0;
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cf::TMEM_COLS);
    tc_fence_before();
    __syncwarp();
    tc_fence_after();
    tmem = *tmem_slot;
    named_bar_arrive(2, 32 + Cf::EPI_THREADS);
  }
  // The set-up above may overlap the previous grid on the stream (programmatic
  // dependent launch); global memory is read and written only after it has
  // completed.  The next grid may start its own set-up from here on.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ---------------- weight producer ----------------
    if (lane == 0 && nk > 0) {
      int i = issued;
      for (; i < nk; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!mbar_wait(empty(s), ph ^ 1u, abort_flag, p.wait_ns, p.status)) break;
        issue_stage(i);
      }
      // Let every copy already issued land before the CTA's smem is released
      // (immediate on the normal path; matters when another role gave up).
      for (int j = (i > STAGES ? i - STAGES : 0); j < i; ++j)
        mbar_wait(full_w(j % STAGES), (j / STAGES) & 1u, never, drain_ns, p.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // One thread issues everything; the tensor pipe is in order, so the loop
    // is kept lean: every descriptor is built once and advanced by additions.
    if (lane == 0) {
      bool ok = true;
      const uint32_t a_tile0 = base + (Cf::kSwapAB ? Cf::OFF_W : Cf::OFF_X);
      const uint32_t b_tile0 = base + (Cf::kSwapAB ? Cf::OFF_X : Cf::OFF_W);
      const uint32_t a_sf0 = base + (Cf::kSwapAB ? Cf::OFF_WSF : Cf::OFF_XSF);
      const uint32_t b_sf0 = base + (Cf::kSwapAB ? Cf::OFF_XSF : Cf::OFF_WSF);
      constexpr uint32_t A_STAGE = Cf::kSwapAB ? Cf::W_CODE_BYTES : Cf::X_CODE_BYTES;
      constexpr uint32_t B_STAGE = Cf::kSwapAB ? Cf::X_CODE_BYTES : Cf::W_CODE_BYTES;
      constexpr uint32_t ASF_STAGE = Cf::kSwapAB ? Cf::W_SF_BYTES : Cf::X_SF_BYTES;
      constexpr uint32_t BSF_STAGE = Cf::kSwapAB ? Cf::X_SF_BYTES : Cf::W_SF_BYTES;
      const uint64_t adesc0 = sdesc_sw128(a_tile0), bdesc0 = sdesc_sw128(b_tile0);
      const uint64_t asfd0 = sdesc_sf(a_sf0), bsfd0 = sdesc_sf(b_sf0);
      const uint32_t idesc0 = idesc_mxf4(Cf::MMA_N, 0, 0), idesc2 = idesc_mxf4(Cf::MMA_N, 2, 2);
      const uint32_t sf_col0 = tmem + Cf::ACC_COLS;
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nk; ++i) {
        if (!mbar_wait(full_w(s), ph, abort_flag, p.wait_ns, p.status) ||
            !mbar_wait(full_x(s), ph, abort_flag, p.wait_ns, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sfa = sf_col0 + s * Cf::SF_STAGE_COLS;
        const uint32_t sfb = sfa + Cf::SFA_COLS;
        const uint64_t ad = adesc0 + ((s * A_STAGE) >> 4), bd = bdesc0 + ((s * B_STAGE) >> 4);
        const uint64_t asd = asfd0 + ((s * ASF_STAGE) >> 4), bsd = bsfd0 + ((s * BSF_STAGE) >> 4);
#pragma unroll
        for (int ka = 0; ka < 2; ++ka) {
          tmem_copy_sf_desc(sfa + ka * 4, asd + ka * (512 >> 4));
          if (Cf::kSwapAB) {
            tmem_copy_sf_desc(sfb + ka * 4, bsd + ka * (512 >> 4));
          } else {
#pragma unroll
            for (int j = 0; j < Cf::W_ATOMS; ++j)
              tmem_copy_sf_desc(sfb + ka * 8 + j * 4, bsd + (j * 1024 + ka * 512) / 16);
          }
        }
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const int ka = ks >> 1;
          mma_mxf4(tmem, ad + ks * 2, bd + ks * 2, (ks & 1) ? idesc2 : idesc0, sfa + ka * 4,
                   sfb + ka * (Cf::kSwapAB ? 4 : 8), (i > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(empty(s));
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      mma_commit(tmem_full);
      // Never release TMEM while MMAs may still be running, whichever role
      // (this one or the epilogue) gave up.
      mbar_wait(tmem_full, 0, never, drain_ns, p.status);
      (void)ok;
    }
  } else {
    // ---------------- activation producers ----------------
    const int qt = threadIdx.x - 64;
    constexpr int P = Cf::QWARPS * 32;
    constexpr int PER = Cf::PER_THREAD;
    const uint16_t* rowp[PER];
    bool rvalid[PER];
    int tok[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int j = qt + u * P;
      const int r = j >> 3;
      rowp[u] = p.A;
      rvalid[u] = false;
      tok[u] = 0;
      if (j < Cf::BLOCKS_PER_STAGE) {
        if (Cf::kMoeAny) {
          const int entry = p.sorted_rows[x_tile * 128 + r];
          if (entry >= 0 && entry < p.routed_rows) {
            rvalid[u] = true;
            rowp[u] = p.A + static_cast<long long>(entry / p.topk) * p.K;
            tok[u] = entry / p.topk;
          }
        } else {
          const int gm = x_tile * NX + r;
          if (gm < p.M) {
            rvalid[u] = true;
            rowp[u] = p.A + static_cast<long long>(gm) * p.K;
          }
        }
      }
    }
    // One stage's BF16 blocks of this thread -> registers (zeros outside A).
    auto load_stage = [&](int i, uint32_t (&w)[PER][16]) {
      const int kbase = (kt0 + i) * 256;
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int j = qt + u * P;
        const int k = kbase + (j & 7) * 32;
        if (j < Cf::BLOCKS_PER_STAGE && rvalid[u] && k < p.K) {
          const uint4* src = reinterpret_cast<const uint4*>(rowp[u] + k);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint4 v = ld_global_nc_v4(src + t);
            w[u][4 * t] = v.x; w[u][4 * t + 1] = v.y; w[u][4 * t + 2] = v.z; w[u][4 * t + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) w[u][t] = 0u;
        }
      }
    };
    // Test hook: the CTAs of weight tile 0 store each code chunk and scale
    // byte at the same offsets in a global copy of the tile as well.
    const bool dump = p.dump_codes != nullptr && w_tile == 0;
    auto dump_store = [&](int i, uint32_t code_off, uint32_t sf_off, uint4 c, uint32_t e) {
      const long long atom = static_cast<long long>(x_tile) * p.KT + kt0 + i;
      *reinterpret_cast<uint4*>(p.dump_codes + atom * Cf::X_CODE_BYTES + code_off) = c;
      p.dump_scales[atom * Cf::X_SF_BYTES + sf_off] = static_cast<uint8_t>(e);
    };
    // Quantise them into stage i's swizzled operand tile and scale atom.
    auto quant_stage = [&](int i, const uint32_t (&w)[PER][16]) {
      const int s = i % STAGES;
      uint8_t* xt = smem + Cf::OFF_X + s * Cf::X_CODE_BYTES;
      uint8_t* xs = smem + Cf::OFF_XSF + s * Cf::X_SF_BYTES;
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int j = qt + u * P;
        if (j < Cf::BLOCKS_PER_STAGE && rvalid[u]) {
          const int r = j >> 3, kb = j & 7;
          uint32_t c[4];
          const uint32_t e = quant32_bf16(w[u], c);
          const uint32_t code_off = (r >> 3) * 1024 + (r & 7) * 128 + ((kb ^ (r & 7)) << 4);
          const uint32_t sf_off = (kb >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (kb & 3);
          const uint4 cv = make_uint4(c[0], c[1], c[2], c[3]);
          *reinterpret_cast<uint4*>(xt + code_off) = cv;
          xs[sf_off] = static_cast<uint8_t>(e);
          if (dump) dump_store(i, code_off, sf_off, cv, e);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(full_x(s));
    };
    const int nq = nk;
    if constexpr (Cf::kGatherQ) {
      // Rows were quantised once beforehand (codes [T, K/2], scales [T, K/32]):
      // copy this thread's 16-byte code chunks and scale bytes of a stage into
      // the swizzled tile and the scale atom; loads run ahead of the stores in
      // a register ring (below).
      auto gload = [&](int i, uint4 (&c)[PER], uint32_t (&e)[PER]) {
#pragma unroll
        for (int u = 0; u < PER; ++u) {
          const int j = qt + u * P;
          const int kb = (kt0 + i) * 8 + (j & 7);
          c[u] = make_uint4(0u, 0u, 0u, 0u);
          e[u] = 0u;
          if (j < Cf::BLOCKS_PER_STAGE && rvalid[u] && kb * 32 < p.K) {
            c[u] = ld_global_nc_v4(p.Aq + static_cast<long long>(tok[u]) * (p.K / 2) + kb * 16);
            e[u] = __ldg(p.As + static_cast<long long>(tok[u]) * (p.K / 32) + kb);
          }
        }
      };
      auto gstore = [&](int i, const uint4 (&c)[PER], const uint32_t (&e)[PER]) {
        const int s = i % STAGES;
        uint8_t* xt = smem + Cf::OFF_X + s * Cf::X_CODE_BYTES;
        uint8_t* xs = smem + Cf::OFF_XSF + s * Cf::X_SF_BYTES;
#pragma unroll
        for (int u = 0; u < PER; ++u) {
          const int j = qt + u * P;
          if (j < Cf::BLOCKS_PER_STAGE && rvalid[u]) {
            const int r = j >> 3, kb = j & 7;
            const uint32_t code_off = (r >> 3) * 1024 + (r & 7) * 128 + ((kb ^ (r & 7)) << 4);
            const uint32_t sf_off = (kb >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (kb & 3);
            *reinterpret_cast<uint4*>(xt + code_off) = c[u];
            xs[sf_off] = static_cast<uint8_t>(e[u]);
            if (dump) dump_store(i, code_off, sf_off, c[u], e[u]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(full_x(s));
      };
      // a register ring of GQ stages: the gathers of stages i+1 .. i+GQ-1 are
      // in flight while stage i is stored (full expert blocks gather 16 KB of
      // scattered rows per stage; one stage ahead left each stage waiting on
      // most of an L2 round trip)
      constexpr int GQ = 3;
      uint4 cq[GQ][PER];
      uint32_t eq[GQ][PER];
#pragma unroll
      for (int r = 0; r < GQ; ++r)
        if (r < nq) gload(r, cq[r], eq[r]);
      bool stop = false;
      for (int i0 = 0; i0 < nq && !stop; i0 += GQ) {
#pragma unroll
        for (int r = 0; r < GQ; ++r) {
          const int i = i0 + r;
          if (i >= nq) break;
          if (!mbar_wait(empty(i % STAGES), ((i / STAGES) & 1) ^ 1u, abort_flag, p.wait_ns, p.status)) {
            stop = true;
            break;
          }
          gstore(i, cq[r], eq[r]);
          if (i + GQ < nq) gload(i + GQ, cq[r], eq[r]);
        }
      }
    } else if (PER <= 2) {
      // A register ring: the loads of stages i+1 .. i+R-1 are in flight while
      // stage i is quantised, so a CTA pays the L2 latency of A about once,
      // not once per stage or two.
      constexpr int R = Cf::A_DEPTH;
      uint32_t wr[R][PER][16];
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (r < nq) load_stage(r, wr[r]);
      bool stop = false;
      for (int i0 = 0; i0 < nq && !stop; i0 += R) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int i = i0 + r;
          if (i >= nq) break;
          if (!mbar_wait(empty(i % STAGES), ((i / STAGES) & 1) ^ 1u, abort_flag, p.wait_ns, p.status)) {
            stop = true;
            break;
          }
          quant_stage(i, wr[r]);
          if (i + R < nq) load_stage(i + R, wr[r]);
        }
      }
    } else {
      for (int i = 0; i < nq; ++i) {
        if (!mbar_wait(empty(i % STAGES), ((i / STAGES) & 1) ^ 1u, abort_flag, p.wait_ns, p.status)) break;
        uint32_t w[PER][16];
        load_stage(i, w);
        quant_stage(i, w);
      }
    }

    // ---------------- epilogue (4 warps, one per TMEM lane quadrant) ----------------
    if (warp < 2 + Cf::EPI_WARPS) {
      named_bar_sync(2, 32 + Cf::EPI_THREADS);     // TMEM address published by the MMA warp
      tc_fence_after();
      tmem = *tmem_slot;
      const int q = warp & 3;
      const int lrow = q * 32 + lane;
      const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
      // One thread decides for all four epilogue warps, so that every named
      // barrier below is reached by all of them or by none.
      if (warp == 2 && lane == 0)
        *epi_ready = (mbar_wait(tmem_full, 0, abort_flag, p.wait_ns, p.status) && !*abort_flag && nk > 0) ? 1 : 0;
      named_bar_sync(1, Cf::EPI_THREADS);
      const int ready = *epi_ready;
      __syncwarp();
      tc_fence_after();
      if (ready) {
        if (Cf::kSwapAB) {
          const int n = w_tile * 128 + lrow;
          const int m0 = x_tile * NX;
          const int mvalid = min(NX, p.M - m0);
          if (p.splits == 1) {
#pragma unroll
            for (int c0 = 0; c0 < NX; c0 += 16) {
              float v[16];
              tmem_ld16(tq + c0, v);
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < mvalid) p.C[static_cast<long long>(m0 + c0 + j) * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
            }
          } else if (p.cluster_reduce) {
            // Stage the fp32 partial [token][weight row] in the drained ring,
            // then hand owner CTA o its tokens [o*U, (o+1)*U) as one contiguous
            // slice, written with 16-byte DSMEM stores into slot [this split]
            // of the owner's push buffer.
            const int S = p.splits;
            const int U = (NX + S - 1) / S;
            float* red = reinterpret_cast<float*>(smem);
#pragma unroll
            for (int c0 = 0; c0 < NX; c0 += 16) {
              float v[16];
              tmem_ld16(tq + c0, v);
#pragma unroll
              for (int j = 0; j < 16; ++j) red[(c0 + j) * 128 + lrow] = v[j];
            }
            named_bar_sync(1, 128);
            const int et = threadIdx.x - 64;
            const uint32_t slot = base + Cf::OFF_PUSH + static_cast<uint32_t>(split * U * 128 * 4);
            for (int o = 0; o < S; ++o) {
              const int t0 = o * U;
              const int t1 = min(t0 + U, mvalid);
              if (t0 >= t1) break;
              const float4* src = reinterpret_cast<const float4*>(red + t0 * 128);
              const int n4 = (t1 - t0) * 32;
              for (int i = et; i < n4; i += 128)
                st_shared_cluster_v4(cluster_map_shared(slot + static_cast<uint32_t>(i * 16), static_cast<uint32_t>(o)), src[i]);
            }
          }
        } else {  // kMoe, kMoePre: activation + MXFP4 requant of the CTA's output columns
          // SwiGLU: 128 output columns per CTA (accumulator columns 0..127
          // gate, 128..255 up); SiLU: 256 output columns, one accumulator
          // column each.  Two warps per TMEM lane quadrant split the columns.
          const int slot = x_tile * 128 + lrow;
          const int entry = p.sorted_rows[slot];
          const bool valid = entry >= 0 && entry < p.routed_rows;
          const bool silu_only = p.act == kActSilu;
          const int groups = silu_only ? 4 : 2;        // 32-column groups per warp
          const int jc0 = w_tile * (silu_only ? 256 : 128);
          const int half = (warp - 2) >> 2;
#pragma unroll 1
          for (int gi = 0; gi < groups; ++gi) {
            const int g4 = groups * half + gi;
            float g[32], h[32];
            tmem_ld16(tq + g4 * 32, g);
            tmem_ld16(tq + g4 * 32 + 16, g + 16);
            if (silu_only) {
#pragma unroll
              for (int i = 0; i < 32; ++i) h[i] = __fdividef(g[i], 1.0f + __expf(-g[i]));
            } else {
              float u[32];
              tmem_ld16(tq + 128 + g4 * 32, u);
              tmem_ld16(tq + 128 + g4 * 32 + 16, u + 16);
#pragma unroll
              for (int i = 0; i < 32; ++i) h[i] = __fdividef(g[i], 1.0f + __expf(-g[i])) * u[i];
            }
            uint32_t c[4];
            const uint32_t e = quant32_f32(h, c);
            const int col = jc0 + g4 * 32;
            if (p.out_tiles) {
              // sorted-slot operand tiles (GEMM2's A operand): every slot is
              // written; a padding slot's accumulator row is zero, so are its
              // codes and scale
              const long long atom = static_cast<long long>(x_tile) * p.KT_out + col / 256;
              const int j = (col % 256) / 32;
              *reinterpret_cast<uint4*>(p.out_q + atom * 16384 + (lrow >> 3) * 1024 + (lrow & 7) * 128 +
                                        ((j ^ (lrow & 7)) << 4)) = make_uint4(c[0], c[1], c[2], c[3]);
              p.out_s[atom * 1024 + (j >> 2) * 512 + (lrow & 31) * 16 + (lrow >> 5) * 4 + (j & 3)] =
                  static_cast<uint8_t>(e);
            } else if (valid) {
              *reinterpret_cast<uint4*>(p.out_q + static_cast<long long>(entry) * (p.I / 2) + col / 2) = make_uint4(c[0], c[1], c[2], c[3]);
              p.out_s[static_cast<long long>(entry) * (p.I / 32) + col / 32] = static_cast<uint8_t>(e);
            }
          }
        }
      }
    }
  }

  if (Cf::kSwapAB && p.cluster_reduce) {
    // Split-K over the cluster: every CTA has pushed its slices of the fp32
    // partial into their owners' push buffers; CTA `rank` owns tokens
    // [rank*U, rank*U + U) and sums the pushed slots locally in split order
    // (bitwise deterministic).  Every thread of every CTA reaches the cluster
    // barrier, so that all pushes have landed.
    cluster_sync_all();
    if (warp >= 2 && warp < 6) {
      const int et = threadIdx.x - 64;
      const int S = p.splits;
      const uint32_t rank = cluster_ctarank();
      const int m0 = x_tile * NX;
      const int mvalid = min(NX, p.M - m0);
      const int n = w_tile * 128 + et;
      const int U = (NX + S - 1) / S;
      const float* push = reinterpret_cast<const float*>(smem + Cf::OFF_PUSH);
      const int t0 = static_cast<int>(rank) * U;
      const int t1 = min(t0 + U, mvalid);
      for (int t = t0; t < t1; ++t) {
        float acc = 0.f;
        for (int c = 0; c < S; ++c) acc += push[(c * U + (t - t0)) * 128 + et];
        p.C[static_cast<long long>(m0 + t) * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
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

// ---------------------------------------------------------------------------
// Host side

template <int MODE, int NX, int STAGES>
static int launch_cfg(const GemmArgs& a, dim3 grid, cudaStream_t st) {
  using Cf = Cfg<MODE, NX, STAGES>;
  auto kern = a4w4_gemm_kernel<MODE, NX, STAGES>;
  static std::atomic<unsigned long long> attr_devs{0};   // bit d: attributes set on device d
  if (ensure_func_attrs(attr_devs, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM_BYTES) == cudaSuccess;
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
  if (a.cluster_reduce) {
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

static int swap_nx(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

// Decode kernel: K splits per 128-row weight tile.  The fewest that let each
// CTA hold its whole K range in its `ring`-deep weight ring (every weight copy
// in flight at once); once split-K is needed at all, raised until the grid
// fills two CTAs per SM (more weight streams in flight), keeping at least one
// K tile per CTA and at most 16 CTAs per cluster (non-portable size).
static int decode_splits(int kt, int ring, int w_tiles, int sms) {
  int splits = (kt + ring - 1) / ring;
  if (splits > 1) {
    int fill = 2 * sms / (w_tiles > 0 ? w_tiles : 1);
    if (fill > kt) fill = kt;
    if (fill > splits) splits = fill;
  }
  if (splits > kMaxDecodeSplits) splits = kMaxDecodeSplits;
  return splits < 1 ? 1 : splits;
}

// Quantise-once plans (M > 128, or M > 64 with N >= 4096): the persistent
// large-M kernel (large.cu) walks the 128 x 256 tiles, one CTA per SM; a last
// wave of r < sms tiles with 2r <= sms (every tile, when they are that few)
// runs as 2r 128-column halves.  No split-K: the activation tiles are the
// whole workspace.
static void plan_persistent(GemmPlan& pl, int M, int N, int sms) {
  pl.swap_ab = 0;
  pl.prequant = 1;
  pl.persistent = 1;
  pl.nx = 128;
  pl.w_tiles = N / 256;
  pl.x_tiles = (M + 127) / 128;
  pl.splits = 1;
  const int tiles = pl.w_tiles * pl.x_tiles;
  const int r = tiles % (sms > 0 ? sms : 1);
  pl.half_tiles = (r > 0 && 2 * r <= sms) ? r : 0;
  pl.aq_bytes = static_cast<size_t>(pl.x_tiles) * pl.kt * (16384 + 1024);
  pl.ws_bytes = pl.aq_bytes;
}

GemmPlan plan_gemm(int M, int N, int K, int sms) {
  GemmPlan pl{};
  pl.kt = (K + 255) / 256;
  if (M > 128 || (M > 64 && N / 256 >= 16)) {
    // 128 x 256 tiles with the tokens on the MMA's 128-row side: fewer
    // operand bytes per weight byte than swap-AB once M passes 64 (for N <
    // 4096, swap-AB's split-K spreads the few tiles better up to 128 rows).
    // The activations are quantised once into tiles (every weight tile's CTA
    // would otherwise load the same BF16 rows, 4x the bytes of their codes).
    plan_persistent(pl, M, N, sms);
    return pl;
  }
  if (M <= 16 || (M <= 32 && (pl.kt <= 4 || decode_splits(pl.kt, 4, N / 128, sms) > kMaxClusterSplits))) {
    // Decode kernel (decode.cu), no workspace.  16 tokens: 3 CTAs fit per SM,
    // so a 3-deep ring (room for the next grid's CTAs to start early and
    // stream their weights), 4 deep when 3 would need over 16 splits.  17-32
    // tokens whose whole K range fits one CTA's ring (K <= 1024) run as two
    // 16-token tiles, each CTA quantising half the rows (32x7168x768: 4.8
    // against 5.6 us in one 32-token tile).  Otherwise 32 tokens fit 2 per SM
    // (4-deep ring); the swap-AB kernel reduces their 16 KB split-K partials
    // as fast, so they come here only when 16-wide clusters give the grid
    // more CTAs than its 8-wide ones (two 16-token tiles with split-K read
    // every weight byte twice: 14.3 against 10.4 us at 32x7168x4224).
    pl.swap_ab = 1;
    pl.decode = 1;
    pl.w_tiles = N / 128;
    if (M <= 16 || pl.kt <= 4) {
      pl.nx = 16;
      pl.x_tiles = (M + 15) / 16;
      pl.ring = M > 16 ? (pl.kt <= 3 ? 3 : 4) : ((pl.kt + 2) / 3 <= kMaxDecodeSplits ? 3 : 4);
    } else {
      pl.nx = 32;
      pl.x_tiles = 1;
      pl.ring = 4;
    }
    pl.splits = decode_splits(pl.kt, pl.ring, pl.w_tiles * pl.x_tiles, sms);
    pl.cluster_reduce = pl.splits > 1;
    return pl;
  }
  // Swap-AB (17 <= M <= 128): weights on the MMA's 128-row side, up to 128
  // tokens on N; K split over the SMs, reduced inside a cluster (at most 8).
  pl.swap_ab = 1;
  pl.nx = swap_nx(M);
  pl.w_tiles = N / 128;
  pl.x_tiles = (M + pl.nx - 1) / pl.nx;
  const int ctas_per_sm = pl.nx <= 32 ? 2 : 1;
  const int tiles = pl.w_tiles * pl.x_tiles;
  int splits = (sms * ctas_per_sm) / (tiles > 0 ? tiles : 1);
  if (splits > pl.kt) splits = pl.kt;
  if (splits > kMaxClusterSplits) splits = kMaxClusterSplits;
  if (splits < 1) splits = 1;
  pl.splits = splits;
  pl.cluster_reduce = splits > 1;
  return pl;
}

int launch_gemm(const GemmPlan& pl, const void* A, int M, int K, const void* Wq, const void* Ws, int N, void* C,
                void* ws, cudaStream_t st, unsigned long long wait_ns, unsigned int* status, int prefetch_w,
                ActDump dump) {
  GemmArgs a{};
  a.prefetch_w = prefetch_w;
  a.dump_codes = dump.codes;
  a.dump_scales = dump.scales;
  a.status = status;
  a.A = static_cast<const uint16_t*>(A);
  a.Wq = static_cast<const uint8_t*>(Wq);
  a.Ws = static_cast<const uint8_t*>(Ws);
  a.C = static_cast<uint16_t*>(C);
  a.M = M; a.N = N; a.K = K; a.KT = pl.kt; a.splits = pl.splits; a.w_tiles = pl.w_tiles;
  a.cluster_reduce = pl.cluster_reduce;
  a.wait_ns = wait_ns;
  const dim3 grid(pl.w_tiles, pl.x_tiles, pl.splits);
  if (pl.decode) return launch_decode(pl, A, M, K, Wq, Ws, N, C, st, wait_ns, status, prefetch_w, dump);
  if (pl.swap_ab) {
    switch (pl.nx) {
      case 32: return launch_cfg<kSwap, 32, 4>(a, grid, st);
      case 64: return launch_cfg<kSwap, 64, 5>(a, grid, st);
      default: return launch_cfg<kSwap, 128, 4>(a, grid, st);
    }
  }
  if (pl.persistent) {
    // workspace: the activation tiles (17 KB atoms: codes then scales)
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    uint8_t* aq = static_cast<uint8_t*>(ws);
    const int rc = launch_quant_activation_tiles(A, M, K, aq, st, sms);
    if (rc != 0) return rc;
    return launch_large(pl, aq, M, Wq, Ws, N, C, st, wait_ns, status, sms);
  }
  return -4;   // every plan is one of the above
}

int launch_moe_gemm1(const void* X, int T, int D, const int32_t* sorted_rows, const int32_t* block_expert,
                     const int32_t* num_blocks, int max_blocks, int topk, const void* W1q, const void* W1s, int E,
                     int I, int act, int out_tiles, void* out_q, void* out_s, void* xq_ws, cudaStream_t st,
                     unsigned long long wait_ns, unsigned int* status, int sms, ActDump dump) {
  GemmArgs a{};
  a.status = status;
  a.dump_codes = dump.codes;
  a.dump_scales = dump.scales;
  a.A = static_cast<const uint16_t*>(X);
  a.Wq = static_cast<const uint8_t*>(W1q);
  a.Ws = static_cast<const uint8_t*>(W1s);
  const int rows = act == kActSwiglu ? 2 * I : I;     // weight rows per expert (SwiGLU: gate + up)
  a.M = T; a.N = rows; a.K = D; a.KT = (D + 255) / 256; a.splits = 1; a.w_tiles = rows / 256;
  a.wait_ns = wait_ns;
  a.sorted_rows = sorted_rows;
  a.block_expert = block_expert;
  a.num_blocks = num_blocks;
  a.topk = topk;
  a.routed_rows = T * topk;
  a.I = I;
  a.E = E;
  a.act = act;
  a.out_tiles = out_tiles;
  a.KT_out = (I + 255) / 256;
  const long long kp = static_cast<long long>(a.KT) * 256;
  a.expert_code_bytes = static_cast<long long>(rows) * kp / 2;
  a.expert_sf_bytes = static_cast<long long>(rows) * kp / 32;
  a.out_q = static_cast<uint8_t*>(out_q);
  a.out_s = static_cast<uint8_t*>(out_s);
  if (max_blocks <= 0) return 0;
  if (xq_ws != nullptr) {
    // quantise every token once (plain MXFP4 layout), then gather those rows
    uint8_t* xq = static_cast<uint8_t*>(xq_ws);
    uint8_t* xs = xq + static_cast<size_t>(T) * (D / 2);
    const int rc = launch_mxfp4_quant(X, T, D, xq, xs, st, sms);
    if (rc != 0) return rc;
    a.Aq = xq;
    a.As = xs;
    return launch_cfg<kMoePre, 128, 4>(a, dim3(a.w_tiles, max_blocks, 1), st);
  }
  return launch_cfg<kMoe, 128, 4>(a, dim3(a.w_tiles, max_blocks, 1), st);
}

}  // namespace a4w4
