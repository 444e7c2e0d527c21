// quant.cu -- MXFP4 quantisation kernels: the standalone plain-layout quant and
// the one-time weight quant + preshuffle into the tensor-core tile layout.
//
// "[gfx1250] Fuse A4W4 stage1 FP4 quantization", Summary (standalone quant kept
// as the fallback); "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM",
// Implementation (one-time packed E2M1 weight and E8M0 scale preshuffle).
#include "device.cuh"
#include "launch.h"

namespace a4w4 {

// One thread per 32-element block; blocks are contiguous in a row-major
// [rows, cols] matrix with cols % 32 == 0, so block b starts at element 32b.
// Reads 64 bytes and writes 16 + 1 bytes per block: HBM-bound.
__global__ void __launch_bounds__(256) mxfp4_quant_kernel(const uint4* __restrict__ x, uint4* __restrict__ q,
                                                          uint8_t* __restrict__ s, long long nblocks) {
  // programmatic dependent launch: x may come from the previous kernel; the
  // next one (a GEMM that waits for this grid before reading q) may start its
  // set-up now
  griddep_wait();
  griddep_launch_dependents();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long b = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblocks; b += stride) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = ld_global_nc_v4(x + 4 * b + i);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
    uint32_t c[4];
    const uint32_t e = quant32_bf16(w, c);
    q[b] = make_uint4(c[0], c[1], c[2], c[3]);
    s[b] = static_cast<uint8_t>(e);
  }
}

// Weights, once: one thread per (row, 32-block) of the padded matrix [rows,
// KP]; writes the 16 code bytes into the 128-byte-swizzled tile and the scale
// byte into the 128x4 scale atom (layout documented in a4w4.h), atoms grouped
// in pairs of row tiles (weight_atom), codes in wq, scales in ws.  With
// `pair_I` > 0 the preshuffled row n of each expert is gate row
// 128*(n/256) + n%256 when n%256 < 128, else up row pair_I + 128*(n/256) + n%256 - 128.
__global__ void __launch_bounds__(256) prepare_weight_kernel(const uint16_t* __restrict__ w, int rows, int K, int KT,
                                                             int experts, int pair_I, uint8_t* __restrict__ wq,
                                                             uint8_t* __restrict__ ws) {
  // w may come from the previous kernel on the stream; the trigger for the
  // next grid stays at completion, since a GEMM with weight prefetch reads its
  // weights before its own grid dependency resolves
  griddep_wait();
  const int kblocks = KT * 8;
  const long long total = static_cast<long long>(experts) * rows * kblocks;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int kb = static_cast<int>(i % kblocks);
    const long long rr = i / kblocks;
    const int n = static_cast<int>(rr % rows);
    const int e = static_cast<int>(rr / rows);
    int src_row = n;
    if (pair_I > 0) {
      const int j = n / 256, within = n % 256;
      src_row = within < 128 ? 128 * j + within : pair_I + 128 * j + (within - 128);
    }
    uint32_t c[4] = {0u, 0u, 0u, 0u};
    uint32_t code = 0;
    if (kb * 32 < K) {
      const uint4* src = reinterpret_cast<const uint4*>(w + (static_cast<long long>(e) * rows + src_row) * K + kb * 32);
      uint32_t v[16];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint4 u = src[t];
        v[4 * t] = u.x; v[4 * t + 1] = u.y; v[4 * t + 2] = u.z; v[4 * t + 3] = u.w;
      }
      code = quant32_bf16(v, c);
    }
    const int nt = n / 128, r = n % 128, kt = kb / 8, j = kb % 8;
    const uint32_t code_off = (r / 8) * 1024 + (r % 8) * 128 + ((j ^ (r % 8)) * 16);
    const uint32_t sf_off = (j / 4) * 512 + (r % 32) * 16 + (r / 32) * 4 + (j % 4);
    const long long atom = static_cast<long long>(e) * (rows / 128) * KT + weight_atom(nt, kt, KT);
    *reinterpret_cast<uint4*>(wq + atom * 16384 + code_off) = make_uint4(c[0], c[1], c[2], c[3]);
    ws[atom * 1024 + sf_off] = static_cast<uint8_t>(code);
  }
}

// Activation tiles of the quantise-once GEMM plans: one thread per (row,
// 32-block) of the matrix padded to whole 128-row and 256-column tiles, item
// i = row * (KT * 8) + block, so a warp's lanes read adjacent 64-byte blocks of
// one row.  Writes the 16 code bytes into the 128-byte-swizzled tile and the
// four scale bytes of four adjacent blocks (adjacent lanes) as one 32-bit
// word of the 128x4 scale atom; atom (x_tile, kt) = 16 KB of codes then 1 KB
// of scales at aq + (x_tile * KT + kt) * 17408.  Rows >= M and blocks past K
// get zeros.  32-bit index arithmetic, no loop: `total` (rows x KT x 8, rows
// a multiple of 128) is a multiple of the block size.
__global__ void __launch_bounds__(256) quant_act_tiles_kernel(const uint16_t* __restrict__ a, int M, int K, int KT,
                                                              uint8_t* __restrict__ aq) {
  griddep_wait();                 // A may come from the previous kernel on the stream
  // the GEMM that follows waits for this grid before reading the tiles, so it
  // may start its set-up now
  griddep_launch_dependents();
  const uint32_t kblocks = static_cast<uint32_t>(KT) * 8u;
  const uint32_t item = blockIdx.x * 256u + threadIdx.x;
  const uint32_t n = item / kblocks, kb = item - n * kblocks;
  uint32_t c[4] = {0u, 0u, 0u, 0u};
  uint32_t e = 0u;
  if (n < static_cast<uint32_t>(M) && kb * 32u < static_cast<uint32_t>(K)) {
    const uint4* src = reinterpret_cast<const uint4*>(a + static_cast<size_t>(n) * K + kb * 32u);
    uint32_t v[16];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint4 u = ld_global_nc_v4(src + t);
      v[4 * t] = u.x; v[4 * t + 1] = u.y; v[4 * t + 2] = u.z; v[4 * t + 3] = u.w;
    }
    e = quant32_bf16(v, c);
  }
  const uint32_t nt = n >> 7, r = n & 127u, kt = kb >> 3, j = kb & 7u;
  uint8_t* at = aq + (static_cast<size_t>(nt) * KT + kt) * 17408u;
  *reinterpret_cast<uint4*>(at + (r >> 3) * 1024u + (r & 7u) * 128u + ((j ^ (r & 7u)) << 4)) =
      make_uint4(c[0], c[1], c[2], c[3]);
  // blocks 4q..4q+3 of a row sit in lanes 4m..4m+3 (kblocks is a multiple of
  // 8, so a group of four never straddles two rows): one word per group
  const uint32_t w4 = (e & 0xFFu) | ((__shfl_down_sync(0xFFFFFFFFu, e, 1) & 0xFFu) << 8) |
                      ((__shfl_down_sync(0xFFFFFFFFu, e, 2) & 0xFFu) << 16) |
                      ((__shfl_down_sync(0xFFFFFFFFu, e, 3) & 0xFFu) << 24);
  if ((j & 3u) == 0u)
    *reinterpret_cast<uint32_t*>(at + 16384u + (j >> 2) * 512u + (r & 31u) * 16u + (r >> 5) * 4u) = w4;
}

static int grid_for(long long items, int threads, int sms, int per_sm) {
  long long g = (items + threads - 1) / threads;
  const long long cap = static_cast<long long>(sms) * per_sm;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

int launch_mxfp4_quant(const void* x, long long rows, int cols, void* q, void* s, cudaStream_t st, int sms) {
  const long long nblocks = rows * (cols / 32);
  return launch_pdl(mxfp4_quant_kernel, grid_for(nblocks, 256, sms, 8), 256, st, static_cast<const uint4*>(x),
                    static_cast<uint4*>(q), static_cast<uint8_t*>(s), nblocks);
}

int launch_prepare_weight(const void* w, int rows, int K, int experts, int pair_I, void* wq, void* ws,
                          cudaStream_t st, int sms) {
  const int KT = (K + 255) / 256;
  const long long items = static_cast<long long>(experts) * rows * KT * 8;
  return launch_pdl(prepare_weight_kernel, grid_for(items, 256, sms, 8), 256, st, static_cast<const uint16_t*>(w),
                    rows, K, KT, experts, pair_I, static_cast<uint8_t*>(wq), static_cast<uint8_t*>(ws));
}

int launch_quant_activation_tiles(const void* a, int M, int K, void* aq, cudaStream_t st, int sms) {
  (void)sms;
  const int KT = (K + 255) / 256;
  const long long rows = (static_cast<long long>(M) + 127) / 128 * 128;
  const long long items = rows * KT * 8;          // a multiple of 1024
  if (items > 0xFFFFFFFFll || items % 256 != 0) return -4;
  return launch_pdl(quant_act_tiles_kernel, static_cast<int>(items / 256), 256, st, static_cast<const uint16_t*>(a),
                    M, K, KT, static_cast<uint8_t*>(aq));
}

}  // namespace a4w4
