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

// One thread per (row, 32-block) of the padded matrix [rows, KP]; writes the
// 16 code bytes into the 128-byte-swizzled tile and the scale byte into the
// 128x4 scale atom (layout documented in a4w4.h).  Rows >= valid_rows (the
// padding of an activation matrix to whole 128-row tiles) get zeros.
// Weights (act_tiles == 0): atoms grouped in pairs of row tiles (weight_atom),
// codes in wq, scales in ws.  Activation tiles of the quantise-once GEMM
// (act_tiles == 1): atom nt*KT + kt holds its 16 KB of codes followed by its
// 1 KB of scales at wq + atom * 17408, so one bulk copy brings both.  With
// `pair_I` > 0 the preshuffled row n of each expert is gate row
// 128*(n/256) + n%256 when n%256 < 128, else up row pair_I + 128*(n/256) + n%256 - 128.
__global__ void __launch_bounds__(256) prepare_weight_kernel(const uint16_t* __restrict__ w, int rows, int valid_rows,
                                                             int K, int KT, int experts, int pair_I,
                                                             uint8_t* __restrict__ wq, uint8_t* __restrict__ ws,
                                                             int act_tiles) {
  griddep_wait();                // w may come from the previous kernel on the stream
  // Activation tiles: the GEMM that follows waits for this grid before
  // reading them, so it may start its set-up now.  Weights: the trigger stays
  // at completion, since a GEMM with weight prefetch reads its weights early.
  if (act_tiles) griddep_launch_dependents();
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
    if (kb * 32 < K && n < valid_rows) {
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
    if (act_tiles) {
      uint8_t* at = wq + (static_cast<long long>(nt) * KT + kt) * 17408;
      *reinterpret_cast<uint4*>(at + code_off) = make_uint4(c[0], c[1], c[2], c[3]);
      at[16384 + sf_off] = static_cast<uint8_t>(code);
    } else {
      const long long atom = static_cast<long long>(e) * (rows / 128) * KT + weight_atom(nt, kt, KT);
      *reinterpret_cast<uint4*>(wq + atom * 16384 + code_off) = make_uint4(c[0], c[1], c[2], c[3]);
      ws[atom * 1024 + sf_off] = static_cast<uint8_t>(code);
    }
  }
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
                    rows, rows, K, KT, experts, pair_I, static_cast<uint8_t*>(wq), static_cast<uint8_t*>(ws), 0);
}

int launch_quant_activation_tiles(const void* a, int M, int K, void* aq, cudaStream_t st, int sms) {
  const int KT = (K + 255) / 256;
  const int rows = (M + 127) / 128 * 128;
  const long long items = static_cast<long long>(rows) * KT * 8;
  return launch_pdl(prepare_weight_kernel, grid_for(items, 256, sms, 8), 256, st, static_cast<const uint16_t*>(a),
                    rows, M, K, KT, 1, 0, static_cast<uint8_t*>(aq), static_cast<uint8_t*>(nullptr), 1);
}

}  // namespace a4w4
