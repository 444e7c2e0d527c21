"""CPU oracle for the MXFP4 A4W4 GEMM path -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously correct float64 restatement of what
the GPU library computes.  It exists to judge the CUDA path, never to stand in
for it: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it.  The product package
(``mxfp4_a4w4_gemm_gb300``) never imports it and has no CPU fallback.

It shares no code with the CUDA path: no kernels, headers, helpers, tables or
constant generators.  The only module both sides use is ``workloads`` (seeded
synthetic inputs), which holds none of the method's arithmetic.

Sources (web pages, cited by title and section):

* "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM" -- Summary (BF16
  activations quantised inline to MXFP4, E2M1 weights with E8M0 scales,
  scaled-FP4 product), Implementation (weights quantised and preshuffled once;
  M-tail masking; ceil-based scale accounting), Scope (N % 256 == 0,
  K % 128 == 0), Kernel microbenchmark (relative L2 2.42%-4.15%).
* "[gfx1250] Fuse A4W4 stage1 FP4 quantization" -- Summary (MoE GEMM1
  epilogue that emits MXFP4 codes and E8M0 scales after the SiLU or SwiGLU
  activation, scale taken from the FP32 activation).
* "[HIP] [CK] [FlyDSL] [Kernel] Extend MXFP4 GEMM1 replacement to A4W4" --
  Summary (auxiliary sort of routed rows; stage-2 paths that consume stage
  1's output layout) and GEMM2 scope.
* The block-scale rule itself is not stated on the pages.  The oracle uses the
  OCP Microscaling Formats (MX) v1.0 rule: shared exponent
  floor(log2(amax)) - 2 over 32 elements, clamped to the E8M0 range; E2M1
  elements rounded to nearest, ties to even, saturating at +-6.

Modules:
  mxfp4  -- E2M1/E8M0 format, block quantiser, packing, BF16 rounding
  gemm   -- the dense A4W4 GEMM (exact products, fp64 sums, BF16 output)
  moe    -- routed-row sort, the grouped GEMM1 + SwiGLU (or SiLU) + MXFP4
            requant, and GEMM2 (down projection, top-k weighted sum)

Parity status of every function is pinned by ``tests/test_oracle_*.py``
(-m "not gpu"); none is "parity unpinned".
"""

from . import mxfp4, gemm, moe  # noqa: F401
