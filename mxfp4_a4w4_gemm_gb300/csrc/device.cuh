// device.cuh -- sm_103a primitives shared by the A4W4 kernels: mbarriers with
// bounded waits, TMA bulk copies, tcgen05 (TMEM alloc, smem->TMEM copy,
// block-scaled MMA, commit, TMEM loads) and the MXFP4 32-block quantiser.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace a4w4 {

// Bit set in the device status word (passed to kernels by address) when a
// bounded wait expires; read and cleared by a4w4_get_device_status().
constexpr unsigned int kStatusTimeout = 1u;

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with parity `parity` to complete.  Gives up
// after `limit_ns` (setting *abort and the status word) or as soon as another
// role of the CTA has set *abort.  Returns true on success.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns, unsigned int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA bulk copy global -> shared, completion counted on an mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}
// Bulk copy shared -> global (both 16-byte aligned, bytes a multiple of 16),
// tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void bulk_s2g(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" :: "l"(gdst), "r"(ssrc), "r"(bytes)
               : "memory");
}
// Close the bulk async-group and wait until its shared-memory sources have
// been read (the shared memory may then be released; the global writes
// complete with the grid).
__device__ __forceinline__ void bulk_commit_wait_read() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Generic-proxy shared-memory writes -> visible to the async proxy (tcgen05).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t threads) {
  asm volatile("bar.arrive %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(slot_smem), "r"(cols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format, version 1).
//   K-major, 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
  d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                   // 128-byte swizzle
  return d;
}
//   Scale-factor source of a 32x128b copy: 32 rows of 16 bytes, no swizzle,
//   8-row groups 128 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptor of tcgen05.mma.kind::mxf4.block_scale: E2M1 x E2M1,
// UE8M0 scales, both operands K-major, D in fp32, dense, M=128, MMA-K = 64.
// sf_a/sf_b select the byte pair of the 32-bit scale words (0 or 2 with two
// 32-blocks per MMA).
__device__ __forceinline__ uint32_t idesc_mxf4(uint32_t n, uint32_t sf_a, uint32_t sf_b) {
  return (sf_b << 4)            // B scale-factor id
         | (1u << 7)            // A type E2M1
         | (1u << 10)           // B type E2M1
         | ((n >> 3) << 17)     // N / 8
         | (1u << 23)           // scale type UE8M0
         | ((128u >> 7) << 27)  // M / 128
         | (sf_a << 29);        // A scale-factor id
}

// Instruction descriptor of tcgen05.mma.kind::f16 with BF16 A and B (both
// K-major), fp32 D, dense, M = 128, MMA-K = 16: D format at bits 4-5 (1 =
// fp32), A and B formats at 7-9 and 10-12 (1 = BF16), N / 8 at 17-22,
// M / 16 at 24-28.
__device__ __forceinline__ uint32_t idesc_bf16(uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

// Copy a 128-row x 4-block scale atom (512 bytes, layout (r%32)*16+(r/32)*4+j)
// from shared memory into 4 TMEM columns (replicated over the 4 lane groups).
__device__ __forceinline__ void tmem_copy_sf(uint32_t taddr, uint32_t saddr) {
  const uint64_t d = sdesc_sf(saddr);
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(d) : "memory");
}

// Same copy with a prebuilt source descriptor (sdesc_sf of the atom's address).
__device__ __forceinline__ void tmem_copy_sf_desc(uint32_t taddr, uint64_t d) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(d) : "memory");
}

__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Arrives on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(bar) : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
// 64 consecutive columns of this warp's lane quadrant: four loads in flight,
// one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[16 * q + 0]), "=r"(r[16 * q + 1]), "=r"(r[16 * q + 2]), "=r"(r[16 * q + 3]), "=r"(r[16 * q + 4]),
          "=r"(r[16 * q + 5]), "=r"(r[16 * q + 6]), "=r"(r[16 * q + 7]), "=r"(r[16 * q + 8]), "=r"(r[16 * q + 9]),
          "=r"(r[16 * q + 10]), "=r"(r[16 * q + 11]), "=r"(r[16 * q + 12]), "=r"(r[16 * q + 13]),
          "=r"(r[16 * q + 14]), "=r"(r[16 * q + 15])
        : "r"(taddr + 16 * q));
  }
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------------------
// MXFP4 quantisation of one 32-element block (OCP MX rule):
//   e = floor(log2 amax) - 2 clamped to [-127, 127]  ->  E8M0 code
//   = max(biased_exponent(amax) - 2, 0) (BF16 and FP32 share the 8-bit
//   exponent field, and finite amax has a biased exponent <= 254);
//   y = |x| * 2^-e exactly (2^-e = 2^(127-code) is a normal float; a product
//   that underflows is far below the first rounding midpoint 0.25);
//   E2M1 by the hardware's round-to-nearest-even saturating conversion;
//   the sign bit of x is copied, so a negative value that rounds to zero
//   gives code 8.

// Four pairs of non-negative floats -> 8 packed E2M1 codes (element 2j low nibble).
__device__ __forceinline__ uint32_t cvt_e2m1x8(float y0, float y1, float y2, float y3, float y4, float y5,
                                               float y6, float y7) {
  uint32_t w;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(w)
      : "f"(y0), "f"(y1), "f"(y2), "f"(y3), "f"(y4), "f"(y5), "f"(y6), "f"(y7));
  return w;
}

// Per 16-bit lane: the BF16 value of larger magnitude, with its sign replaced
// by the xor of the two inputs' signs.
__device__ __forceinline__ uint32_t max_abs_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}


// x: 32 BF16 values as 16 words (element 2j in the low half of w[j]).
// Returns the E8M0 code; codes[0..3] receive the 16 packed code bytes.  The
// signed values go through the conversion as they are: E2M1 is
// sign-magnitude and round-to-nearest-even and saturation are symmetric, so
// the code of -x is the code of x with bit 3 set, a negative value that
// rounds to zero included (code 8), as the rule wants.
__device__ __forceinline__ uint32_t quant32_bf16(const uint32_t* w, uint32_t* codes) {
  // the larger magnitude of each BF16 lane pair, one instruction per word
  // (finite inputs: magnitude order is the order of the unsigned bit patterns
  // with the sign cleared; the result's sign bits are dropped below)
  uint32_t m = w[0];
#pragma unroll
  for (int j = 1; j < 16; ++j) m = max_abs_bf16x2(m, w[j]);
  m &= 0x7FFF7FFFu;
  const uint32_t amax = max(m & 0xFFFFu, m >> 16);
  const uint32_t ebits = amax >> 7;
  const uint32_t code = ebits > 2u ? ebits - 2u : 0u;
  const float inv = __uint_as_float((254u - code) << 23);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float y[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t a = w[4 * q + j];
      y[2 * j] = __uint_as_float(a << 16) * inv;
      y[2 * j + 1] = __uint_as_float(a & 0xFFFF0000u) * inv;
    }
    codes[q] = cvt_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
  }
  return code;
}

// h: 32 fp32 values.  Same rule as quant32_bf16.
__device__ __forceinline__ uint32_t quant32_f32(const float* h, uint32_t* codes) {
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = max(amax, __float_as_uint(h[i]) & 0x7FFFFFFFu);
  const uint32_t ebits = amax >> 23;
  const uint32_t code = ebits > 2u ? ebits - 2u : 0u;
  const float inv = __uint_as_float((254u - code) << 23);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float y[8];
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t b = __float_as_uint(h[8 * q + i]);
      y[i] = __uint_as_float(b & 0x7FFFFFFFu) * inv;
      s |= (b >> 31) << (4 * i + 3);
    }
    codes[q] = cvt_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]) | s;
  }
  return code;
}

// Weight operand layout (a4w4.h): 128-row x 256-K atoms grouped in pairs of
// row tiles, so that a 256-row tile's two atoms of one K tile are adjacent:
// atom (nt, kt) is number ((nt / 2) * KT + kt) * 2 + nt % 2, at 16 KB (codes)
// and 1 KB (scales) per atom.
__device__ __forceinline__ long long weight_atom(int nt, int kt, int KT) {
  return (static_cast<long long>(nt >> 1) * KT + kt) * 2 + (nt & 1);
}

__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

}  // namespace a4w4

namespace a4w4 {

// ---------------------------------------------------------------------------
// Programmatic dependent launch: a grid launched with the programmatic
// stream-serialisation attribute may start before the previous grid on the
// stream has finished; griddep_wait() returns once that grid has completed and
// its memory is visible.  griddep_launch_dependents() lets the next grid start.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters: a barrier over every thread of every CTA in the
// cluster (release/acquire orders shared-memory writes before peer reads),
// and loads from a peer CTA's shared memory.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Split cluster barrier: arrive early (relaxed; mbarrier inits are published
// by fence_barrier_init), wait before the first access to a peer's memory.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void fence_acq_rel_cluster() {
  asm volatile("fence.acq_rel.cluster;" ::: "memory");
}
// 16-byte store into a peer CTA's shared memory whose completion is counted
// (complete_tx, release at cluster scope) on an mbarrier of that same peer;
// `dst` and `bar` are shared::cluster addresses from cluster_map_shared.
__device__ __forceinline__ void st_async_v4(uint32_t dst, float4 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
               :: "r"(dst), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar) : "memory");
}
// Arrive (release, cluster scope) on an mbarrier in a peer CTA's shared
// memory (`remote` from cluster_map_shared).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(remote) : "memory");
}
// Wait (acquire, cluster scope) for a phase of a local mbarrier that peers
// arrive on; bounded like mbar_wait (no abort flag: the caller must not leave
// before the peers' writes have landed unless the limit passes).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                  unsigned int* status) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    if (ok) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}
__device__ __forceinline__ uint32_t cluster_map_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_shared_cluster_f32x2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_shared_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_shared_cluster_v4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

}  // namespace a4w4
