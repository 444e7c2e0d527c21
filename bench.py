"""Benchmark of the MXFP4 A4W4 GEMM path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload all|decode|small|large|stress|moe]

Prints ONE JSON line (rank 0).  The default (``all``) measures every workload
of the metric "M = 1-2048" in one invocation:

* ``decode`` (the headline: ``value``, ``roofline``, ``e2e``, ``cpu_baseline``)
  -- the nine decode-size GEMMs M in {1, 8, 32} x (N, K) in {(7168, 4224),
  (1536, 7168), (7168, 768)}, BF16 activations N(0,1) with 1% x20 outlier
  channels, MXFP4 weights from N(0,0.02);
* ``large`` -- M in {128, 512, 2048} x (N, K) in {(8448, 7168), (7168, 4224)};
* ``stress`` -- M in {37, 513, 2047}, N = 1536, K = 4224, scale-edge blocks;
* ``moe`` -- grouped MoE GEMM1 + SwiGLU + MXFP4 requant, T in {1, 16, 256,
  4096}, E = 896, topk = 16, D = 3584, I = 768 (sort + GEMM1 per T);

each under ``configs`` with its own step time, per-GEMM table, roofline,
end-to-end figures, clocks and CPU-oracle baseline.  A step is one pass over
the workload's GEMMs, each one launch of the fused quant + tcgen05
block-scaled GEMM + epilogue (the quantise-once plans add the activation
pre-pass).  Weights are prepared once, outside timing, as on the source page.

Timing: W warm-up steps, then K steps replayed from CUDA graphs, bracketed by
a barrier and torch.cuda.synchronize(), CUDA events on the launching stream.
Each GEMM call in a step reads a different copy of its weights, rotating over
copies totalling more than twice the L2 size, so weights stream from HBM.

value  = sum of algorithmic bytes (N*K/2 + N*K/32 + 2*M*K + 2*M*N per GEMM)
         over the step / step time, in TB/s (whole job: all ranks' bytes over
         the slowest rank's time).
e2e    = the same metric with each step's activations copied from pinned host
         memory and its outputs copied back inside the timed region (graphs of
         the C ABI calls; ``e2e_eager`` issues every C ABI call from Python
         instead, so the host cost of the calls is inside the time too).
N > 1: replicas only (the GEMMs of different ranks are independent; no
collective on the data path).

``--impl reference`` times the CPU oracle (oracle/) on a bounded sample of the
headline workload on the host cores and prints the same line with "impl":
"reference".
"""

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "A4W4 GEMM µs & TFLOPS/TB/s vs GB300 FP4/HBM roofline, M=1–2048"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP4_OVER_BF16 = 13.5 / 2.25       # nominal dense ratio (fp4 13.5 PF, bf16 2.25 PF per GPU)
L2_BYTES = 126 * 1024 * 1024

# Source page's microbenchmark (MI355X, median us; another machine: context,
# not a baseline): "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM",
# Kernel microbenchmark.
PAGES_US = {(7168, 4224, 1): 15.960, (7168, 4224, 8): 23.041, (7168, 4224, 32): 23.520,
            (1536, 7168, 1): 18.420, (1536, 7168, 8): 23.320, (1536, 7168, 32): 26.181,
            (7168, 768, 1): 12.580, (7168, 768, 8): 11.921, (7168, 768, 32): 12.120,
            (8448, 7168, 128): 60.121, (8448, 7168, 512): 89.480, (8448, 7168, 2048): 237.863,
            (7168, 4224, 128): 23.280, (7168, 4224, 512): 50.041, (7168, 4224, 2048): 107.041}
# "[gfx1250] Fuse A4W4 stage1 FP4 quantization", Performance (gfx1250, fused
# GEMM1 operator latency in us by token count; SiTUv2 there, SwiGLU here)
PAGES_MOE_US = {1: 47.39, 16: 201.41, 256: 676.86, 4096: 1351.28}
ALL_WORKLOADS = ["decode", "large", "stress", "moe", "moe2", "a16w4"]

WORKLOADS = {
    "decode": ("decode-size dense A4W4 sweep, M in {1,8,32} x (N,K) in {(7168,4224),(1536,7168),(7168,768)}",
               workloads.DECODE_SWEEP, "decode"),
    "small": ("dense A4W4 GEMM 16x256x256", workloads.SMALL, "small"),
    "large": ("large-M dense A4W4 sweep, M in {128,512,2048} x (N,K) in {(8448,7168),(7168,4224)}",
              workloads.LARGE_M_SWEEP, "large"),
    "stress": ("tail/scale-edge stress, M in {37,513,2047}, N=1536, K=4224", workloads.TAIL_STRESS, "stress"),
    "moe": ("grouped MoE GEMM1 A4W4 + SwiGLU + MXFP4 requant, T in {1,16,256,4096}, E=896, topk=16, D=3584, I=768",
            [], "moe"),
    "a16w4": ("A16WFP4 decode-size sweep (BF16 activations x MXFP4 weights), M in {1,8,32} x (N,K) in "
              "{(7168,4224),(1536,7168),(7168,768)}", workloads.DECODE_SWEEP, "decode"),
    "moe2": ("grouped MoE GEMM2 A4W4 (down projection of GEMM1's MXFP4 tiles, top-k weighted per-token sum), "
             "T in {1,16,256,4096}, E=896, topk=16, D=3584, I=768", [], "moe2"),
}


def gemm_bytes(M, N, K):
    return N * K // 2 + N * K // 32 + 2 * M * K + 2 * M * N


def gemm_flops(M, N, K):
    return 2 * M * N * K


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x, device):
    """The largest of every rank's value of `x` (one all_reduce), or `x`
    itself without a multi-rank process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, bytes_per_step, ms_per_step):
    """Whole-job TB/s: every rank streams `bytes_per_step` per step (weak
    scaling, independent replicas), timed by the slowest rank."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e12


# ---------------------------------------------------------------------------
# clocks sampled during the timed region

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax = float(f[1])
            except ValueError:
                continue
            for name, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# dense workloads on the GPU

class DenseSweep:
    def __init__(self, shapes, family, dev, a16w4=False):
        self.a16w4 = a16w4
        import torch
        import mxfp4_a4w4_gemm_gb300 as a4w4
        self.torch, self.a4w4, self.dev = torch, a4w4, dev
        self.shapes = list(shapes)
        self.family = family
        nk = sorted({(N, K) for _, N, K in self.shapes})
        wbytes = sum(a4w4.a4w4_weight_codes_bytes(N, K) + a4w4.a4w4_weight_scales_bytes(N, K) for N, K in nk)
        self.copies = max(2, -(-2 * L2_BYTES // wbytes))
        self.wq, self.ws = {}, {}
        for N, K in nk:
            W = workloads.bits_to_torch(workloads.weight_bits(N, K)).to(dev)
            q = torch.empty(a4w4.a4w4_weight_codes_bytes(N, K), dtype=torch.uint8, device=dev)
            s = torch.empty(a4w4.a4w4_weight_scales_bytes(N, K), dtype=torch.uint8, device=dev)
            a4w4.a4w4_prepare_gemm_weight(W, N, K, q, s)
            self.wq[(N, K)] = [q] + [q.clone() for _ in range(self.copies - 1)]
            self.ws[(N, K)] = [s] + [s.clone() for _ in range(self.copies - 1)]
            del W
        # A step's activations (and outputs) are views into one device buffer
        # with one pinned host mirror, so the end-to-end step moves them with
        # one copy each way (every view starts on a 256-byte boundary: K % 128 == 0,
        # N % 256 == 0).  Two such I/O slots let one step's copies overlap
        # another step's kernels; `slot` selects the one that calls use.
        a_elems = sum(M * K for M, _, K in self.shapes)
        c_elems = sum(M * N for M, N, _ in self.shapes)
        a_host = torch.empty(a_elems, dtype=torch.bfloat16)
        ao = 0
        for M, N, K in self.shapes:
            A_bits, _ = workloads.dense_problem(M, N, K, family) if family != "decode" else (
                workloads.decode_activation_bits(M, K), None)
            a_host[ao:ao + M * K].copy_(workloads.bits_to_torch(A_bits).reshape(-1))
            ao += M * K
        self.slot = 0
        self.A_host = [a_host.pin_memory() for _ in range(2)]
        self.C_host = [torch.empty(c_elems, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        self.A_dev = [torch.empty(a_elems, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.C_dev = [torch.empty(c_elems, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.A, self.C = [[], []], [[], []]
        for b in range(2):
            ao = co = 0
            for M, N, K in self.shapes:
                self.A[b].append(self.A_dev[b][ao:ao + M * K].view(M, K))
                self.C[b].append(self.C_dev[b][co:co + M * N].view(M, N))
                ao += M * K
                co += M * N
            self.A_dev[b].copy_(self.A_host[b])
        self.ws_bytes = max(a4w4.a4w4_gemm_workspace_bytes(M, N, K) for M, N, K in self.shapes)
        self.work = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=dev)
        a4w4.a4w4_workspace_init(self.work, self.ws_bytes)
        self.bytes_per_step = sum(gemm_bytes(*s) for s in self.shapes)
        self.flops_per_step = sum(gemm_flops(*s) for s in self.shapes)
        # the quantise-once plans launch the activation pre-pass too
        self.launches_per_step = sum(self.launches_of(i) for i in range(len(self.shapes)))
        self.flags = 0
        torch.cuda.synchronize()

    def call(self, i, r):
        M, N, K = self.shapes[i]
        c = (r * len(self.shapes) + i) % self.copies
        if self.a16w4:
            self.a4w4.a4w4_gemm_a16w4(self.A[self.slot][i], M, K, self.wq[(N, K)][c], self.ws[(N, K)][c], N,
                                      self.C[self.slot][i], self.flags)
            return
        self.a4w4.a4w4_gemm_ex(self.A[self.slot][i], M, K, self.wq[(N, K)][c], self.ws[(N, K)][c], N,
                               self.C[self.slot][i], self.work, self.ws_bytes, self.flags)

    def step(self, r):
        for i in range(len(self.shapes)):
            self.call(i, r)

    def h2d(self, b):
        self.A_dev[b].copy_(self.A_host[b], non_blocking=True)

    def d2h(self, b):
        self.C_host[b].copy_(self.C_dev[b], non_blocking=True)

    @property
    def h2d_bytes(self):
        return sum(2 * M * K for M, _, K in self.shapes)

    @property
    def d2h_bytes(self):
        return sum(2 * M * N for M, N, _ in self.shapes)

    def kernel_name(self, i):
        M, N, K = self.shapes[i]
        if self.a16w4:
            return f"a4w4_a16w4_kernel<{16 if M <= 16 else 32}>"
        return self.a4w4.a4w4_gemm_kernel_name(M, N, K)   # the library's own plan

    def launches_of(self, i):
        """Kernel launches of one call of GEMM i (the quantise-once plans add the pre-pass)."""
        return 2 if "prequant" in self.kernel_name(i) else 1

    def label(self, i):
        M, N, K = self.shapes[i]
        return {"M": M, "N": N, "K": K}


def sort_buffers(a4w4, torch, dev, ids, E, maxb):
    """Device buffers of one routing for the single-launch sort (its
    workspace zeroed once, as the library asks)."""
    T, topk = ids.shape
    wsb = a4w4.a4w4_moe_sort_aux_workspace_bytes(T, topk, E)
    ro = dict(ids=torch.from_numpy(ids).to(dev), hits=int(np.unique(ids).size),
              rows=torch.empty(maxb * 128, dtype=torch.int32, device=dev),
              toks=torch.empty(maxb * 128, dtype=torch.int32, device=dev),
              slot=torch.empty(T * topk, dtype=torch.int32, device=dev),
              bexp=torch.empty(maxb, dtype=torch.int32, device=dev),
              nb=torch.empty(1, dtype=torch.int32, device=dev),
              ws=torch.empty(wsb, dtype=torch.uint8, device=dev), wsb=wsb)
    a4w4.a4w4_workspace_init(ro["ws"], wsb)
    return ro


class MoeSweep:
    """Grouped MoE GEMM1 workload: for each token count T, the routed-row sort
    (single launch, with the gather/scatter arrays) and GEMM1 + SwiGLU + MXFP4
    requant (E=896, topk=16, D=3584, I=768)."""

    def __init__(self, dev, tokens=None, inline=False):
        self.inline = inline
        import torch
        import mxfp4_a4w4_gemm_gb300 as a4w4
        from mxfp4_a4w4_gemm_gb300.host_prep import prepare_moe_w1_from_host
        self.torch, self.a4w4, self.dev = torch, a4w4, dev
        c = workloads.MOE
        self.E, self.topk, self.D, self.I = c["experts"], c["topk"], c["model_dim"], c["inter_dim"]
        self.tokens = list(tokens or c["tokens"])
        self.W1q, self.W1s = prepare_moe_w1_from_host(
            lambda e: workloads.moe_expert_weight_bits(e, 2 * self.I, self.D), self.E, 2 * self.I, self.D,
            threads=16, device=dev)
        # rotate routings so that the experts a small-T step touches are cold in L2
        self.copies = 8
        self.items = []
        for T in self.tokens:
            X = workloads.bits_to_torch(workloads.moe_tokens_bits(T, self.D))
            routes = []
            for v in range(self.copies):
                ids = workloads.moe_topk_ids(T, self.E, self.topk, seed=2 + 1000 * v)
                maxb = a4w4.a4w4_moe_max_blocks(T, self.topk, self.E, 128)
                routes.append(sort_buffers(a4w4, torch, dev, ids, self.E, maxb))
            # quantise tokens once (workspace) unless T = 1 or inline quant is forced
            xwsb = 0 if (T == 1 or self.inline) else a4w4.a4w4_moe_gemm1_workspace_bytes(T, self.D)
            # tokens and outputs in two I/O slots (see DenseSweep); sort and
            # quantisation workspaces are used by the kernels alone
            R = T * self.topk
            self.items.append(dict(
                T=T, X=[X.to(dev) for _ in range(2)], X_host=[X.pin_memory() for _ in range(2)],
                routes=routes, xwsb=xwsb,
                xws=torch.empty(max(xwsb, 16), dtype=torch.uint8, device=dev) if xwsb else None,
                q=[torch.empty((R, self.I // 2), dtype=torch.uint8, device=dev) for _ in range(2)],
                s=[torch.empty((R, self.I // 32), dtype=torch.uint8, device=dev) for _ in range(2)],
                q_host=[torch.empty((R, self.I // 2), dtype=torch.uint8).pin_memory() for _ in range(2)],
                s_host=[torch.empty((R, self.I // 32), dtype=torch.uint8).pin_memory() for _ in range(2)]))
        self.slot = 0
        self.flags = 0
        self.shapes = [(it["T"], 2 * self.I, self.D) for it in self.items]
        # the sort + GEMM1 per T, + the token quantisation when GEMM1 has a workspace
        self.launches_per_step = sum(2 + (1 if it["xws"] is not None else 0) for it in self.items)
        self.bytes_per_step = sum(self.item_bytes(i, 0) for i in range(len(self.items)))
        self.flops_per_step = sum(2 * it["T"] * self.topk * 2 * self.I * self.D for it in self.items)
        torch.cuda.synchronize()

    def item_bytes(self, i, r):
        it = self.items[i]
        T, hits = it["T"], it["routes"][r % self.copies]["hits"]
        return int(hits * 2 * self.I * self.D * (1 / 2 + 1 / 32) + 2 * T * self.D + self.topk * T * (self.I // 2 + self.I // 32))

    def call(self, i, r, sort=True, gemm=True):
        it = self.items[i]
        ro = it["routes"][(r * len(self.items) + i) % self.copies]
        T = it["T"]
        if sort:
            self.a4w4.a4w4_moe_sort_aux(ro["ids"], T, self.topk, self.E, 128, ro["rows"], ro["bexp"], ro["nb"],
                                        ro["toks"], ro["slot"], ro["ws"], ro["wsb"])
        if gemm:
            b = self.slot
            self.a4w4.a4w4_moe_gemm1(it["X"][b], T, self.D, ro["rows"], ro["bexp"], ro["nb"], self.topk,
                                     self.W1q, self.W1s, self.E, self.I, it["q"][b], it["s"][b], it["xws"],
                                     it["xwsb"])

    def step(self, r):
        for i in range(len(self.items)):
            self.call(i, r)

    def h2d(self, b):
        for it in self.items:
            it["X"][b].copy_(it["X_host"][b], non_blocking=True)

    def d2h(self, b):
        for it in self.items:
            it["q_host"][b].copy_(it["q"][b], non_blocking=True)
            it["s_host"][b].copy_(it["s"][b], non_blocking=True)

    @property
    def h2d_bytes(self):
        return sum(2 * it["T"] * self.D for it in self.items)

    @property
    def d2h_bytes(self):
        return sum(it["T"] * self.topk * (self.I // 2 + self.I // 32) for it in self.items)

    def kernel_name(self, i):
        return "a4w4_gemm_kernel<moe,128>" if self.items[i]["xws"] is None else "a4w4_gemm_kernel<moe-prequant,128>"

    def launches_of(self, i):
        """Kernel launches of GEMM1 alone for token count i (+ the token quantisation)."""
        return 1 if self.items[i]["xws"] is None else 2

    def label(self, i):
        return {"T": self.items[i]["T"], "E": self.E, "topk": self.topk, "D": self.D, "I": self.I}


class Moe2Sweep:
    """Grouped MoE GEMM2 workload: for each token count T, the routed-row
    sort, then GEMM2 (down projection of GEMM1's sorted-slot MXFP4 tiles
    against W2[e] [D, I], top-k weighted fp32 rows) and the per-token sum to
    BF16 Y [T, D] (E=896, topk=16, D=3584, I=768).  The input tiles are
    random MXFP4 codes with E8M0 scales near 2^-7 (values do not change the
    work); W2 ~ N(0, 0.02) as in the recipe."""

    def __init__(self, dev, tokens=None):
        import torch
        import mxfp4_a4w4_gemm_gb300 as a4w4
        from mxfp4_a4w4_gemm_gb300.host_prep import prepare_dense_experts_from_host
        self.torch, self.a4w4, self.dev = torch, a4w4, dev
        c = workloads.MOE
        self.E, self.topk, self.D, self.I = c["experts"], c["topk"], c["model_dim"], c["inter_dim"]
        self.tokens = list(tokens or c["tokens"])
        self.W2q, self.W2s = prepare_dense_experts_from_host(
            lambda e: workloads.moe_expert_w2_bits(e, self.D, self.I), self.E, self.D, self.I, threads=16, device=dev)
        self.copies = 8
        self.items = []
        g = torch.Generator(device=dev)
        g.manual_seed(6)
        for T in self.tokens:
            routes = []
            maxb = a4w4.a4w4_moe_max_blocks(T, self.topk, self.E, 128)
            for v in range(self.copies):
                ids = workloads.moe_topk_ids(T, self.E, self.topk, seed=2 + 1000 * v)
                routes.append(sort_buffers(a4w4, torch, dev, ids, self.E, maxb))
            cb = a4w4.a4w4_moe_tiles_codes_bytes(T, self.topk, self.E, self.I)
            sb = a4w4.a4w4_moe_tiles_scales_bytes(T, self.topk, self.E, self.I)
            aq = torch.randint(0, 256, (cb,), dtype=torch.uint8, device=dev, generator=g)
            as_ = torch.randint(118, 124, (sb,), dtype=torch.uint8, device=dev, generator=g)
            wts = torch.from_numpy(workloads.moe_topk_weights(T, self.topk))
            # inputs (tiles + routing weights) in one buffer per I/O slot
            inp_host = torch.cat([aq.cpu(), as_.cpu(), wts.view(torch.uint8).reshape(-1)])
            wsb2 = a4w4.a4w4_moe_gemm2_workspace_bytes(T, self.topk, self.D)
            self.items.append(dict(
                T=T, routes=routes, cb=cb, sb=sb,
                inp=[inp_host.to(dev) for _ in range(2)], inp_host=[inp_host.pin_memory() for _ in range(2)],
                ws=torch.empty(wsb2, dtype=torch.uint8, device=dev), wsb=wsb2,
                Y=[torch.empty((T, self.D), dtype=torch.bfloat16, device=dev) for _ in range(2)],
                Y_host=[torch.empty((T, self.D), dtype=torch.bfloat16).pin_memory() for _ in range(2)]))
            del aq, as_
        self.slot = 0
        self.flags = 0
        self.shapes = [(it["T"], self.D, self.I) for it in self.items]
        # the sort + GEMM2 + the per-token sum per T
        self.launches_per_step = 3 * len(self.items)
        self.bytes_per_step = sum(self.item_bytes(i, 0) for i in range(len(self.items)))
        self.flops_per_step = sum(2 * it["T"] * self.topk * self.D * self.I for it in self.items)
        torch.cuda.synchronize()

    def item_bytes(self, i, r):
        it = self.items[i]
        T, hits = it["T"], it["routes"][r % self.copies]["hits"]
        return int(hits * self.D * self.I * (1 / 2 + 1 / 32) + T * self.topk * self.I * (1 / 2 + 1 / 32)
                   + 2 * T * self.D + 4 * T * self.topk)

    def call(self, i, r, sort=True, gemm=True):
        it = self.items[i]
        ro = it["routes"][(r * len(self.items) + i) % self.copies]
        T = it["T"]
        if sort:
            self.a4w4.a4w4_moe_sort_aux(ro["ids"], T, self.topk, self.E, 128, ro["rows"], ro["bexp"], ro["nb"],
                                        ro["toks"], ro["slot"], ro["ws"], ro["wsb"])
        if gemm:
            b = self.slot
            base = it["inp"][b].data_ptr()
            self.a4w4.a4w4_moe_gemm2(base, base + it["cb"], T, self.I, ro["rows"], ro["bexp"], ro["nb"], self.topk,
                                     base + it["cb"] + it["sb"], self.W2q, self.W2s, self.E, self.D, it["Y"][b],
                                     it["ws"], it["wsb"])

    def step(self, r):
        for i in range(len(self.items)):
            self.call(i, r)

    def h2d(self, b):
        for it in self.items:
            it["inp"][b].copy_(it["inp_host"][b], non_blocking=True)

    def d2h(self, b):
        for it in self.items:
            it["Y_host"][b].copy_(it["Y"][b], non_blocking=True)

    @property
    def h2d_bytes(self):
        return sum(it["inp"][0].numel() for it in self.items)

    @property
    def d2h_bytes(self):
        return sum(2 * it["T"] * self.D for it in self.items)

    def kernel_name(self, i):
        return "a4w4_moe2_kernel"      # the persistent GEMM2 walk, every token count

    def launches_of(self, i):
        """GEMM2 and the per-token sum."""
        return 2

    def label(self, i):
        return {"T": self.items[i]["T"], "E": self.E, "topk": self.topk, "D": self.D, "I": self.I}


def capture_graphs(torch, n, fn):
    graphs = []
    for r in range(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(r)
        graphs.append(g)
    torch.cuda.synchronize()
    return graphs


def fp4_peak_tflops(peaks):
    """Dense FP4 peak: the measured bf16 burst x the nominal fp4/bf16 ratio."""
    return peaks["bf16_tflops"] * FP4_OVER_BF16


def make_workload(name, args, dev):
    desc, shapes, family = WORKLOADS[name]
    tokens = [int(t) for t in args.tokens.split(",")] if args.tokens else None
    if name == "moe":
        return desc, MoeSweep(dev, tokens=tokens, inline=args.moe_inline)
    if name == "moe2":
        return desc, Moe2Sweep(dev, tokens=tokens)
    if args.shape and args.workload not in ("all", "moe", "moe2"):
        shapes = [tuple(int(v) for v in args.shape.split(","))]
        desc = f"one dense A4W4 GEMM {shapes[0][0]}x{shapes[0][1]}x{shapes[0][2]} ({name} inputs)"
    return desc, DenseSweep(shapes, family, dev, a16w4=(name == "a16w4"))


def time_step_graphs(torch, stream, graphs, steps, barrier, min_region_s=0.5):
    """Median, over repeated timed regions of `steps` graph replays (at least
    `min_region_s` of GPU time in all), of a region's milliseconds."""
    n = len(graphs)
    barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    regions = []
    t0 = time.time()
    while True:
        start.record(stream)
        for i in range(steps):
            graphs[i % n].replay()
        end.record(stream)
        torch.cuda.synchronize()
        regions.append(start.elapsed_time(end))
        if time.time() - t0 > min_region_s or len(regions) >= 50:
            break
    barrier()
    return statistics.median(regions), len(regions)


def measure(name, args, wl, desc, torch, stream, dev, world, barrier, peaks, peak_src):
    """Time one workload: graphs of whole steps (the value), per-GEMM launch
    durations (roofline), end-to-end with host buffers (graph-pipelined and
    eager).  Returns the workload's result block."""
    nrot = wl.copies
    is_moe = isinstance(wl, (MoeSweep, Moe2Sweep))
    # warm the library's per-device set-up before any capture, then capture
    for r in range(2):
        wl.step(r)
    torch.cuda.synchronize()
    step_graphs = capture_graphs(torch, nrot, wl.step)
    # spin-up (>= 1 s untimed, brings clocks up) + W warm-up steps
    t0 = time.time()
    r = 0
    while time.time() - t0 < 1.0:
        step_graphs[r % nrot].replay()
        r += 1
        if r % 64 == 0:
            torch.cuda.synchronize()
    for i in range(args.warmup):
        step_graphs[i % nrot].replay()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        time.sleep(0.25)
        region_ms, nregions = time_step_graphs(torch, stream, step_graphs, args.steps, barrier)
    region_ms = max_over_ranks(region_ms, dev)
    ms_per_step = region_ms / args.steps
    value = job_throughput(world, wl.bytes_per_step, ms_per_step)
    launches = args.steps * wl.launches_per_step * nregions
    del step_graphs

    # per-GEMM launch durations: one graph per shape of `nrot` back-to-back
    # launches on rotating weight copies, timed with events on this stream
    per = []
    for i in range(len(wl.shapes)):
        # MoE: time GEMM1 alone (the sort's outputs for every routing are in place)
        g = capture_graphs(torch, 1, lambda _r, i=i: [
            (wl.call(i, rr, sort=False) if is_moe else wl.call(i, rr)) for rr in range(nrot)])[0]
        g.replay()
        reps = max(3, int(2000 // nrot))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s0.record(stream)
        for _ in range(reps):
            g.replay()
        s1.record(stream)
        torch.cuda.synchronize()
        launches += reps * nrot * wl.launches_of(i)
        del g
        us = s0.elapsed_time(s1) * 1e3 / (reps * nrot)
        M, N, K = wl.shapes[i]
        if is_moe:
            nbytes = sum(wl.item_bytes(i, rr) for rr in range(nrot)) / nrot
            nflops = 2 * M * wl.topk * N * K
            pages = PAGES_MOE_US.get(M) if name == "moe" else None
        else:
            nbytes, nflops = gemm_bytes(M, N, K), gemm_flops(M, N, K)
            pages = PAGES_US.get((N, K, M))
        extra = {}
        if is_moe:
            # the single-launch sort of the same routings, timed alone
            g = capture_graphs(torch, 1, lambda _r, i=i: [wl.call(i, rr, gemm=False) for rr in range(nrot)])[0]
            g.replay()
            torch.cuda.synchronize()
            s0.record(stream)
            for _ in range(reps):
                g.replay()
            s1.record(stream)
            torch.cuda.synchronize()
            launches += reps * nrot
            extra["sort_us"] = round(s0.elapsed_time(s1) * 1e3 / (reps * nrot), 3)
            del g
        per.append(dict(wl.label(i), **extra, us=round(us, 3), tbs=round(nbytes / us / 1e6, 3),
                        tflops=round(nflops / us / 1e6, 2), kernel=wl.kernel_name(i), bytes=int(nbytes),
                        flops=int(nflops), hbm_frac=round(nbytes / us / 1e3 / peaks["hbm_gbs"], 4),
                        fp4_frac=round(nflops / us / 1e6 / fp4_peak_tflops(peaks), 4),
                        pages_mi355x_us=pages))

    # dominant kernel: the instantiation with the largest share of the step
    share = {}
    for p in per:
        e = share.setdefault(p["kernel"], [0.0, 0, 0, 0])
        e[0] += p["us"]
        e[1] += p["bytes"]
        e[2] += p["flops"]
        e[3] += 1
    dom = max(share, key=lambda k: share[k][0])
    dom_us, dom_bytes, dom_flops, dom_n = share[dom]
    achieved_gbs = dom_bytes / (dom_us * 1e-6) / 1e9
    roof_hbm = {"bound": "hbm", "kernel": dom, "achieved": round(achieved_gbs, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved_gbs / peaks["hbm_gbs"], 4),
                "traffic": traffic_from_profiles(name, dom), "peak_source": f"{peak_src} hbm_gbs (of {peak_src})",
                "bytes_per_launch": round(dom_bytes / dom_n), "avg_launch_us": round(dom_us / dom_n, 3)}
    block = {"workload": desc, "value": round(value, 4), "unit": "TB/s", "ms_per_step": round(ms_per_step, 5),
             "tflops": round(world * wl.flops_per_step / (ms_per_step * 1e-3) / 1e12, 2),
             "gemms_per_step": len(wl.shapes), "per_gemm": per, "roofline": roof_hbm,
             "timed_regions": nregions, "clocks": clk.summary()}
    big = [p for p in per if p["M"] >= 512] if name == "large" else []
    if big:
        # the compute-bound end of the metric: FP4 tensor roofline over the
        # GEMMs with M >= 512, the dominant kernel's launches (a --shape run
        # below 512 rows keeps the HBM roofline)
        us = sum(p["us"] for p in big)
        fl = sum(p["flops"] for p in big)
        tf = fl / (us * 1e-6) / 1e12
        pk = fp4_peak_tflops(peaks)
        block["roofline"] = {
            "bound": "tensor", "kernel": dom, "achieved": round(tf, 1), "peak": round(pk, 1), "unit": "TFLOP/s",
            "frac": round(tf / pk, 4), "traffic": traffic_from_profiles(name, dom),
            "peak_source": f"{peak_src} bf16_tflops x 13.5/2.25 (nominal dense fp4/bf16 ratio; of {peak_src})",
            "gemms": "M >= 512", "avg_launch_us": round(us / len(big), 3)}
        block["roofline_hbm"] = roof_hbm

    # end to end, graphs: step r's inputs go up on one copy stream and its
    # outputs come back on another, in I/O slot r % 2, so step r+1's upload and
    # step r-1's download overlap step r's kernels.  A slot is refilled only
    # after the kernels of step r-2 stopped reading it and its outputs were
    # read back; every step's copies lie inside the timed region.
    e2e_graphs = []
    for r in range(2 * nrot):
        wl.slot = r % 2
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            wl.step(r)
        e2e_graphs.append(g)
    wl.slot = 0
    torch.cuda.synchronize()
    block["e2e"], n1 = e2e_pipelined(torch, stream, dev, wl, args.steps, barrier, world,
                                     lambda r: e2e_graphs[r % len(e2e_graphs)].replay())
    block["e2e"]["pipeline"] = "CUDA graphs of the C ABI calls; pinned host buffers, two I/O slots; H2D, kernels and D2H on three streams"
    del e2e_graphs
    # end to end, eager: every C ABI call issued from Python on every step
    # (argument checks, planning, launch), same copies and pipelining
    def eager(r):
        wl.slot = r % 2
        wl.step(r)
    block["e2e_eager"], n2 = e2e_pipelined(torch, stream, dev, wl, args.steps, barrier, world, eager)
    block["e2e_eager"]["pipeline"] = "every C ABI call issued from Python (ctypes) per step; pinned host buffers, two I/O slots, three streams"
    wl.slot = 0
    block["gpu_launches"] = launches + (n1 + n2) * wl.launches_per_step
    status = wl.a4w4.a4w4_get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}: {wl.a4w4.a4w4_strerror(status)}")
    return block


def e2e_pipelined(torch, stream, dev, wl, steps, barrier, world, run_step):
    """Time `steps` end-to-end steps (H2D of the step's inputs, the step,
    D2H of its outputs), pipelined over two I/O slots on three streams."""
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    up = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    down = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def one(r):
        b = r % 2
        with torch.cuda.stream(s_up):
            if used[b]:
                s_up.wait_event(done[b])
            wl.h2d(b)
            up[b].record(s_up)
        stream.wait_event(up[b])
        if used[b]:
            stream.wait_event(down[b])
        run_step(r)
        done[b].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(done[b])
            wl.d2h(b)
            down[b].record(s_down)
        used[b] = True

    for r in range(4):
        one(r)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_up.wait_event(e0)
    s_down.wait_event(e0)
    for r in range(steps):
        one(r)
    for b in range(2):
        if used[b]:
            stream.wait_event(down[b])
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, dev)
    return ({"value": round(job_throughput(world, wl.bytes_per_step, ms), 4), "unit": "TB/s",
             "ms_per_step": round(ms, 5), "h2d_bytes_per_step": wl.h2d_bytes,
             "d2h_bytes_per_step": wl.d2h_bytes}, steps + 4)


def run_profile(args):
    """A short eager run for profilers: the workload's set-up, then
    args.steps steps of plain C ABI calls (no graphs, no spin-up, no
    end-to-end or CPU legs), so that a profiler sees few, predictable
    launches.  Prints one JSON line with the launches issued; not a bench
    value."""
    import torch
    import mxfp4_a4w4_gemm_gb300 as a4w4
    from mxfp4_a4w4_gemm_gb300 import build
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    a4w4.lib()
    desc, wl = make_workload(args.workload, args, dev)
    wl.flags = a4w4.A4W4_GEMM_WEIGHT_PREFETCH if args.weight_prefetch else 0
    torch.cuda.synchronize()
    for r in range(args.steps):
        wl.step(r)
    torch.cuda.synchronize()
    status = a4w4.a4w4_get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}: {a4w4.a4w4_strerror(status)}")
    print(json.dumps({"profile": True, "workload": desc, "steps": args.steps,
                      "launches": args.steps * wl.launches_per_step,
                      "kernels": [wl.kernel_name(i) for i in range(len(wl.shapes))]}), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch
    import mxfp4_a4w4_gemm_gb300 as a4w4
    from mxfp4_a4w4_gemm_gb300 import build

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)
    build.build()
    a4w4.lib()
    flags = a4w4.A4W4_GEMM_WEIGHT_PREFETCH if args.weight_prefetch else 0
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    names = ALL_WORKLOADS if args.workload == "all" else [args.workload]
    blocks = {}
    headline = names[0]
    for name in names:
        desc, wl = make_workload(name, args, dev)
        wl.flags = flags
        blocks[name] = measure(name, args, wl, desc, torch, stream, dev, world, barrier, peaks, peak_src)
        if name == "decode" and args.weight_prefetch:
            # the same step without weight prefetch (each GEMM streams its
            # weights only after the previous kernel completes)
            wl.flags = 0
            g = capture_graphs(torch, wl.copies, wl.step)
            for i in range(args.warmup):
                g[i % len(g)].replay()
            ms, _ = time_step_graphs(torch, stream, g, args.steps, barrier, min_region_s=0.3)
            ms = max_over_ranks(ms, dev) / args.steps
            blocks[name]["no_weight_prefetch"] = {"value": round(job_throughput(world, wl.bytes_per_step, ms), 4),
                                                  "unit": "TB/s", "ms_per_step": round(ms, 5)}
            blocks[name]["gpu_launches"] += (args.warmup + args.steps) * wl.launches_per_step
            del g
        if name == "decode" and world == 1:
            pages_us = sum(PAGES_US[(N, K, M)] for M, N, K in wl.shapes)
            blocks[name]["vs_pages_mi355x"] = round(
                blocks[name]["value"] / (wl.bytes_per_step / (pages_us * 1e-6) / 1e12), 3)
        if rank == 0 and not args.no_cpu_baseline:
            blocks[name]["cpu_baseline"] = cpu_baseline(name, budget_s=args.cpu_seconds)
        del wl
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    h = blocks[headline]
    line = {
        "metric": METRIC, "value": h["value"], "unit": "TB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": h["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e2m1 x e2m1 -> fp32 (bf16 in/out)",
        "data": "synthetic (seeded; no checkpoints or datasets)",
        "config": {"workload": h["workload"], "gemms_per_step": h["gemms_per_step"],
                   "graphs": "CUDA graphs, one per step",
                   "weight_prefetch": bool(args.weight_prefetch),
                   "l2": "inputs larger than L2: weights rotate over copies > 2x L2 (MoE: 2.6 GB of experts)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "per_gemm": h["per_gemm"], "timed_regions": h["timed_regions"]},
        "roofline": h["roofline"],
        "e2e": h["e2e"],
        "e2e_eager": h["e2e_eager"],
        "gpu_launches": sum(b["gpu_launches"] for b in blocks.values()),
        "clocks": h["clocks"],
    }
    for k in ("no_weight_prefetch", "vs_pages_mi355x", "cpu_baseline"):
        if k in h:
            line[k] = h[k]
    if len(blocks) > 1:
        line["configs"] = {k: {kk: vv for kk, vv in b.items()} for k, b in blocks.items() if k != headline}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def traffic_from_profiles(workload, kernel):
    """dram read+write bytes per launch of `kernel` in `workload`, derived from
    an ncu capture of the current kernel, if profiles/traffic.json holds one
    ("workload:kernel" keys); else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        v = d.get(f"{workload}:{kernel}")
        return v["bytes_per_launch"] if isinstance(v, dict) else v
    except (OSError, ValueError, KeyError, TypeError):
        return None


# ---------------------------------------------------------------------------
# CPU oracle timing

def oracle_sample_step(shapes, family, r, cols=16, a16=False):
    """One bounded oracle step: for every GEMM of the workload, the oracle's
    full path (quantise A and a 16-row slice of W, float64 products, BF16
    rounding) on the output columns n0..n0+15, n0 rotating with r.  Returns
    the algorithmic bytes of that sample."""
    from oracle import gemm
    done = 0
    for i, (M, N, K) in enumerate(shapes):
        A_bits, W_bits = _cached_problem(M, N, K, family)
        n0 = ((r * 7 + i) * cols) % N
        (gemm.gemm_a16w4 if a16 else gemm.gemm_a4w4)(A_bits, W_bits[n0:n0 + cols])
        done += cols * K // 2 + cols * K // 32 + 2 * M * K + 2 * M * cols
    return done


def oracle_quant_only(shapes, family, r, cols=16):
    """The quantisation part of oracle_sample_step alone (A and the W slice)."""
    from oracle import mxfp4
    for i, (M, N, K) in enumerate(shapes):
        A_bits, W_bits = _cached_problem(M, N, K, family)
        n0 = ((r * 7 + i) * cols) % N
        mxfp4.mxfp4_quant(A_bits)
        mxfp4.mxfp4_quant(W_bits[n0:n0 + cols])


_MOE_CACHE = {}


def oracle_moe_sample(r, rows_per_t=1):
    """One bounded oracle step of the MoE GEMM1 workload: for every token
    count T, `rows_per_t` routed rows (rotating with r) through the oracle's
    GEMM1 + SwiGLU + requant.  Returns the algorithmic bytes of the sample
    (each row's expert weights, token and output)."""
    from oracle import moe
    c = workloads.MOE
    E, topk, D, I = c["experts"], c["topk"], c["model_dim"], c["inter_dim"]
    done = 0
    for T in c["tokens"]:
        if T not in _MOE_CACHE:
            _MOE_CACHE[T] = (workloads.moe_tokens_bits(T, D), workloads.moe_topk_ids(T, E, topk))
        X, ids = _MOE_CACHE[T]
        rows = [(r * rows_per_t + j) * 7919 % (T * topk) for j in range(rows_per_t)]
        moe.gemm1_rows(X, ids, lambda e: workloads.moe_expert_weight_bits(e, 2 * I, D), rows, I)
        done += len(rows) * int(2 * I * D * (1 / 2 + 1 / 32) + 2 * D + I // 2 + I // 32)
    return done


def oracle_moe2_sample(r):
    """One bounded oracle step of the MoE GEMM2 workload: one token of token
    count T (T and the token rotate with r) through the oracle's GEMM2: its
    topk routed rows, each expert's W2 quantised in full.  Returns the
    algorithmic bytes of the sample."""
    from oracle import moe, mxfp4
    c = workloads.MOE
    E, topk, D, I = c["experts"], c["topk"], c["model_dim"], c["inter_dim"]
    T = c["tokens"][r % len(c["tokens"])]
    key = ("moe2", T)
    if key not in _MOE_CACHE:
        _MOE_CACHE[key] = (workloads.moe_hidden_bits(T * topk, I), workloads.moe_topk_ids(T, E, topk),
                           workloads.moe_topk_weights(T, topk))
    H, ids, wts = _MOE_CACHE[key]
    t = (r * 7919) % T
    q, s = mxfp4.mxfp4_quant(H[t * topk:(t + 1) * topk])
    moe.gemm2_tokens(q, s, ids[t:t + 1], wts[t:t + 1], lambda e: workloads.moe_expert_w2_bits(e, D, I), [0])
    return int(topk * (D * I * (1 / 2 + 1 / 32) + I * (1 / 2 + 1 / 32) + 4) + 2 * D)


_PROBLEMS = {}


def _cached_problem(M, N, K, family):
    key = (M, N, K, family)
    if key not in _PROBLEMS:
        if family == "decode":
            _PROBLEMS[key] = (workloads.decode_activation_bits(M, K), workloads.weight_bits(N, K))
        else:
            _PROBLEMS[key] = workloads.dense_problem(M, N, K, family)
    return _PROBLEMS[key]


def _threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def cpu_baseline(workload, budget_s=15.0):
    """The oracle as it stands, timed on this host's cores on a bounded sample
    of `workload`: repeated sample steps for about `budget_s` seconds (the
    value), plus quantisation and GEMM timed apart on one sample step (median
    of 3 each)."""
    if workload == "a16w4":
        desc, shapes, family = WORKLOADS[workload]
        for M, N, K in shapes:
            _cached_problem(M, N, K, family)
        step, quant = (lambda r: oracle_sample_step(shapes, family, r, a16=True)), None
        sample = ("every GEMM of the workload on 16 output columns per step (quantisation of those W rows, "
                  "float64 sums of the BF16 activations, BF16 rounding)")
    elif workload == "moe":
        step, quant = oracle_moe_sample, None
        sample = ("every token count's routed row per step through GEMM1 + SwiGLU + requant "
                  "(each row's expert quantised in full)")
    elif workload == "moe2":
        step, quant = oracle_moe2_sample, None
        sample = ("one token per step (token counts 1, 16, 256, 4096 in turn) through GEMM2: its 16 routed "
                  "rows, each expert's W2 quantised in full")
    else:
        desc, shapes, family = WORKLOADS[workload]
        for M, N, K in shapes:
            _cached_problem(M, N, K, family)
        step = lambda r: oracle_sample_step(shapes, family, r)        # noqa: E731
        quant = lambda r: oracle_quant_only(shapes, family, r)        # noqa: E731
        sample = ("every GEMM of the workload on 16 output columns per step (full quantisation of A and of "
                  "those W rows, float64 sums, BF16 rounding)")
    step(0)
    t0 = time.time()
    done, r = 0, 0
    while time.time() - t0 < budget_s or r == 0:
        done += step(r)
        r += 1
    dt = time.time() - t0
    out = {"value": round(done / dt / 1e12, 9), "unit": "TB/s", "cores": _threads(), "kind": "oracle",
           "cpu": cpu_model(), "nproc": os.cpu_count(),
           "sample": f"{r} oracle steps over {dt:.1f} s; {sample}"}
    if quant is not None:
        full = []
        qt = []
        for _ in range(3):
            t = time.perf_counter()
            step(0)
            full.append(time.perf_counter() - t)
            t = time.perf_counter()
            quant(0)
            qt.append(time.perf_counter() - t)
        out["quant_s"] = round(statistics.median(qt), 4)
        out["gemm_s"] = round(max(0.0, statistics.median(full) - statistics.median(qt)), 4)
        out["split"] = "one sample step, median of 3: quantisation of A and the W slice; the rest (products, sums, rounding)"
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return
    name = ALL_WORKLOADS[0] if args.workload == "all" else args.workload
    desc, shapes, family = WORKLOADS[name]
    if name == "moe":
        step = oracle_moe_sample
        sample = "every token count's routed row per step through the oracle's GEMM1 + SwiGLU + requant"
    elif name == "moe2":
        step = oracle_moe2_sample
        sample = "one token per step (token counts in turn) through the oracle's GEMM2"
    else:
        for M, N, K in shapes:
            _cached_problem(M, N, K, family)
        step = lambda r: oracle_sample_step(shapes, family, r)        # noqa: E731
        sample = "every GEMM of the workload on 16 output columns per step"
    for r in range(args.warmup):
        step(r)
    t0 = time.time()
    done = 0
    for r in range(args.steps):
        done += step(r)
    dt = time.time() - t0
    value = done / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 9), "unit": "TB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": desc, "sample": sample},
            "cpu_baseline": {"value": round(value, 9), "unit": "TB/s", "cores": _threads(), "kind": "oracle",
                             "cpu": cpu_model(), "nproc": os.cpu_count(),
                             "sample": f"{args.steps} oracle steps; {sample}"},
            "e2e": {"value": round(value, 9), "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["all"] + sorted(WORKLOADS), default="all")
    ap.add_argument("--cpu-seconds", type=float, default=6.0, help="oracle baseline budget per workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shape", default="", help="M,N,K: time one GEMM of the workload's input family "
                                                "(with a single --workload)")
    ap.add_argument("--moe-inline", action="store_true", help="MoE: quantise gathered rows inline in every tile")
    ap.add_argument("--tokens", default="", help="MoE workloads: comma-separated token counts (default all)")
    ap.add_argument("--profile", action="store_true",
                    help="a few eager steps for a profiler (no graphs, spin-up, e2e or CPU legs); not a bench value")
    ap.add_argument("--no-weight-prefetch", dest="weight_prefetch", action="store_false",
                    help="do not let a GEMM stream its weights before the previous kernel finishes (default: "
                         "it may, since the weights are prepared before the timed region and never written in it)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = dist_env()
    if args.profile:
        if args.workload == "all":
            ap.error("--profile needs a single --workload")
        run_profile(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
