"""Benchmark of the MXFP4 A4W4 GEMM path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|small|large|stress|moe]

Prints ONE JSON line (rank 0).  A step is one pass of the path over the
workload: for the default ``decode`` workload, the nine decode-size GEMMs
M in {1, 8, 32} x (N, K) in {(7168, 4224), (1536, 7168), (7168, 768)} (BF16
activations N(0,1) with 1% x20 outlier channels, MXFP4 weights from N(0,0.02)),
each one launch of the fused quant + tcgen05 block-scaled GEMM + BF16
epilogue.  Weights are prepared once, outside timing, as on the source page.

Timing: W warm-up steps, then K steps replayed from CUDA graphs, bracketed by
a barrier and torch.cuda.synchronize(), CUDA events on the launching stream.
Each GEMM call in a step reads a different copy of its weights, rotating over
copies totalling more than twice the L2 size, so weights stream from HBM.

value  = sum of algorithmic bytes (N*K/2 + N*K/32 + 2*M*K + 2*M*N per GEMM)
         over the step / step time, in TB/s (whole job: all ranks' bytes over
         the slowest rank's time).
e2e    = the same metric with each step's activations copied from pinned host
         memory and its outputs copied back inside the timed region.
N > 1: replicas only (the GEMMs of different ranks are independent; no
collective on the data path).

``--impl reference`` times the CPU oracle (oracle/) on a bounded sample of the
same workload on the host cores and prints the same line with "impl":
"reference".
"""

import argparse
import json
import os
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

# Source page's microbenchmark (MI355X, median us) for the decode-size points:
# "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM", Kernel microbenchmark.
PAGES_US = {(7168, 4224, 1): 15.960, (7168, 4224, 8): 23.041, (7168, 4224, 32): 23.520,
            (1536, 7168, 1): 18.420, (1536, 7168, 8): 23.320, (1536, 7168, 32): 26.181,
            (7168, 768, 1): 12.580, (7168, 768, 8): 11.921, (7168, 768, 32): 12.120}

WORKLOADS = {
    "decode": ("decode-size dense A4W4 sweep, M in {1,8,32} x (N,K) in {(7168,4224),(1536,7168),(7168,768)}",
               workloads.DECODE_SWEEP, "decode"),
    "small": ("dense A4W4 GEMM 16x256x256", workloads.SMALL, "small"),
    "large": ("large-M dense A4W4 sweep, M in {128,512,2048} x (N,K) in {(8448,7168),(7168,4224)}",
              workloads.LARGE_M_SWEEP, "large"),
    "stress": ("tail/scale-edge stress, M in {37,513,2047}, N=1536, K=4224", workloads.TAIL_STRESS, "stress"),
    "moe": ("grouped MoE GEMM1 A4W4 + SwiGLU + MXFP4 requant, T in {1,16,256,4096}, E=896, topk=16, D=3584, I=768",
            [], "moe"),
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
    def __init__(self, shapes, family, dev):
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
        self.launches_per_step = len(self.shapes)
        torch.cuda.synchronize()

    def call(self, i, r):
        M, N, K = self.shapes[i]
        c = (r * len(self.shapes) + i) % self.copies
        self.a4w4.a4w4_gemm(self.A[self.slot][i], M, K, self.wq[(N, K)][c], self.ws[(N, K)][c], N,
                            self.C[self.slot][i], self.work, self.ws_bytes)

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
        return self.a4w4.a4w4_gemm_kernel_name(M, N, K)   # the library's own plan

    def label(self, i):
        M, N, K = self.shapes[i]
        return {"M": M, "N": N, "K": K}


class MoeSweep:
    """Grouped MoE GEMM1 workload: for each token count T, the routed-row sort
    and GEMM1 + SwiGLU + MXFP4 requant (E=896, topk=16, D=3584, I=768)."""

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
                wsb = a4w4.a4w4_moe_sort_workspace_bytes(T, self.topk, self.E)
                routes.append(dict(
                    ids=torch.from_numpy(ids).to(dev), hits=int(np.unique(ids).size),
                    rows=torch.empty(maxb * 128, dtype=torch.int32, device=dev),
                    bexp=torch.empty(maxb, dtype=torch.int32, device=dev),
                    nb=torch.empty(1, dtype=torch.int32, device=dev),
                    ws=torch.empty(wsb, dtype=torch.uint8, device=dev), wsb=wsb))
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
        self.shapes = [(it["T"], 2 * self.I, self.D) for it in self.items]
        self.launches_per_step = 4 * len(self.items)      # 3 sort kernels + GEMM1 per T
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
            self.a4w4.a4w4_moe_sort(ro["ids"], T, self.topk, self.E, 128, ro["rows"], ro["bexp"], ro["nb"],
                                    ro["ws"], ro["wsb"])
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
    if args.weight_prefetch:
        a4w4.a4w4_set_weight_prefetch(1)
    desc, shapes, family = WORKLOADS[args.workload]
    if args.workload == "moe":
        wl = MoeSweep(dev, inline=args.moe_inline)
    else:
        if args.shape:
            shapes = [tuple(int(v) for v in args.shape.split(","))]
            desc = f"one dense A4W4 GEMM {shapes[0][0]}x{shapes[0][1]}x{shapes[0][2]} ({args.workload} inputs)"
        wl = DenseSweep(shapes, family, dev)
    nrot = wl.copies

    def barrier():
        if world > 1:
            torch.distributed.barrier()

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

    stream = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        time.sleep(0.25)
        barrier()
        torch.cuda.synchronize()
        # keep the timed region >= 0.5 s for the clock samples: repeat whole timed
        # regions of K steps and report the median region
        regions = []
        t_region = time.time()
        while True:
            start.record(stream)
            for i in range(args.steps):
                step_graphs[i % nrot].replay()
            end.record(stream)
            torch.cuda.synchronize()
            regions.append(start.elapsed_time(end))
            if time.time() - t_region > 0.5 or len(regions) >= 50:
                break
        barrier()
    region_ms = max_over_ranks(statistics.median(regions), dev)
    ms_per_step = region_ms / args.steps
    value = job_throughput(world, wl.bytes_per_step, ms_per_step)

    # per-GEMM launch durations: one graph per shape of `nrot` back-to-back
    # launches on rotating weight copies, timed with events on this stream
    per = []
    is_moe = isinstance(wl, MoeSweep)
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
        us = s0.elapsed_time(s1) * 1e3 / (reps * nrot)
        M, N, K = wl.shapes[i]
        if is_moe:
            nbytes = sum(wl.item_bytes(i, rr) for rr in range(nrot)) / nrot
            nflops = 2 * M * wl.topk * N * K
        else:
            nbytes, nflops = gemm_bytes(M, N, K), gemm_flops(M, N, K)
        per.append(dict(wl.label(i), us=round(us, 3), tbs=round(nbytes / us / 1e6, 3),
                        tflops=round(nflops / us / 1e6, 2), kernel=wl.kernel_name(i), bytes=int(nbytes)))

    peaks, peak_src = load_peaks()
    # dominant kernel: the instantiation with the largest share of the step
    share = {}
    for p in per:
        share.setdefault(p["kernel"], [0.0, 0, 0])
        share[p["kernel"]][0] += p["us"]
        share[p["kernel"]][1] += p["bytes"]
        share[p["kernel"]][2] += 1
    dom = max(share, key=lambda k: share[k][0])
    dom_us, dom_bytes, dom_n = share[dom]
    achieved_gbs = dom_bytes / (dom_us * 1e-6) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved_gbs, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved_gbs / peaks["hbm_gbs"], 4),
                "traffic": traffic_from_profiles(args.workload, dom), "peak_source": f"{peak_src} hbm_gbs",
                "bytes_per_launch": round(dom_bytes / dom_n), "avg_launch_us": round(dom_us / dom_n, 3)}

    # End to end through the C ABI with host buffers, pipelined as a serving
    # loop would run it: step r's inputs go up on one copy stream and its
    # outputs come back on another, in I/O slot r % 2, so step r+1's upload
    # and step r-1's download overlap step r's kernels.  A slot is refilled
    # only after the kernels of step r-2 stopped reading it and its outputs
    # were read back; every step's copies lie inside the timed region.
    e2e_graphs = []
    for r in range(2 * nrot):
        wl.slot = r % 2
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            wl.step(r)
        e2e_graphs.append(g)
    wl.slot = 0
    torch.cuda.synchronize()
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    up = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    down = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(r):
        b = r % 2
        with torch.cuda.stream(s_up):
            if used[b]:
                s_up.wait_event(done[b])
            wl.h2d(b)
            up[b].record(s_up)
        stream.wait_event(up[b])
        if used[b]:
            stream.wait_event(down[b])
        e2e_graphs[r % len(e2e_graphs)].replay()
        done[b].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(done[b])
            wl.d2h(b)
            down[b].record(s_down)
        used[b] = True

    for r in range(4):
        e2e_step(r)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_up.wait_event(e0)
    s_down.wait_event(e0)
    for r in range(args.steps):
        e2e_step(r)
    for b in range(2):
        if used[b]:
            stream.wait_event(down[b])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
    e2e_value = job_throughput(world, wl.bytes_per_step, e2e_ms)

    status = a4w4.a4w4_get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}: {a4w4.a4w4_strerror(status)}")

    pages_us = sum(PAGES_US.get((N, K, M), float("nan")) for M, N, K in wl.shapes)
    vs = None
    if args.workload == "decode" and world == 1:
        vs = round(value / (wl.bytes_per_step / (pages_us * 1e-6) / 1e12), 3)

    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "TB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": vs, "dtype": "e2m1 x e2m1 -> fp32 (bf16 in/out)",
        "data": "synthetic (seeded; no checkpoints or datasets)",
        "config": {"workload": desc, "gemms_per_step": len(wl.shapes), "graphs": "CUDA graphs, one per step",
                   "weight_prefetch": bool(args.weight_prefetch),
                   "l2": (f"{nrot} routings rotate (experts touched per step differ); W1 is 2.6 GB" if is_moe else
                          f"weights rotate over {nrot} copies ({nrot * sum(gemm_bytes(0, N, K) for N, K in wl.wq) / 1e6:.0f} MB > 2x L2)"),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "per_gemm": per, "timed_regions": len(regions)},
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 4), "unit": "TB/s", "ms_per_step": round(e2e_ms, 5),
                "pipeline": "pinned host buffers, two I/O slots; H2D, kernels and D2H on three streams",
                "h2d_bytes_per_step": wl.h2d_bytes, "d2h_bytes_per_step": wl.d2h_bytes},
        "gpu_launches": args.steps * wl.launches_per_step * len(regions),
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline and not is_moe:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_seconds)
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

def oracle_sample_step(shapes, family, r, cols=16):
    """One bounded oracle step: for every GEMM of the workload, the oracle's
    full path (quantise A and a 16-row slice of W, float64 products, BF16
    rounding) on the output columns n0..n0+15, n0 rotating with r."""
    from oracle import gemm
    done = 0
    for i, (M, N, K) in enumerate(shapes):
        A_bits, W_bits = _cached_problem(M, N, K, family)
        n0 = ((r * 7 + i) * cols) % N
        gemm.gemm_a4w4(A_bits, W_bits[n0:n0 + cols])
        done += cols * K // 2 + cols * K // 32 + 2 * M * K + 2 * M * cols
    return done


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


def cpu_baseline(workload, budget_s=15.0):
    desc, shapes, family = WORKLOADS[workload]
    for M, N, K in shapes:
        _cached_problem(M, N, K, family)
    oracle_sample_step(shapes, family, 0)
    t0 = time.time()
    done, r = 0, 0
    while time.time() - t0 < budget_s or r == 0:
        done += oracle_sample_step(shapes, family, r)
        r += 1
    dt = time.time() - t0
    return {"value": round(done / dt / 1e12, 9), "unit": "TB/s", "cores": _threads(), "kind": "oracle",
            "sample": f"{r} oracle steps over {dt:.1f} s; each step: every GEMM of the workload on 16 output "
                      f"columns (full quantisation of A and of those W rows, float64 sums, BF16 rounding)"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    desc, shapes, family = WORKLOADS[args.workload]
    for M, N, K in shapes:
        _cached_problem(M, N, K, family)
    for r in range(args.warmup):
        oracle_sample_step(shapes, family, r)
    t0 = time.time()
    done = 0
    for r in range(args.steps):
        done += oracle_sample_step(shapes, family, r)
    dt = time.time() - t0
    value = done / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 9), "unit": "TB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": desc, "sample": "every GEMM of the workload on 16 output columns per step"},
            "cpu_baseline": {"value": round(value, 9), "unit": "TB/s", "cores": _threads(), "kind": "oracle",
                             "sample": f"{args.steps} oracle steps, 16 output columns of every GEMM per step"},
            "e2e": {"value": round(value, 9), "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shape", default="", help="M,N,K: time one GEMM of the workload's input family")
    ap.add_argument("--moe-inline", action="store_true", help="MoE: quantise gathered rows inline in every tile")
    ap.add_argument("--no-weight-prefetch", dest="weight_prefetch", action="store_false",
                    help="do not let a GEMM stream its weights before the previous kernel finishes (default: "
                         "it may, since the weights are prepared before the timed region and never written in it)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
