"""GPU parity of the MoE stage-1 variants and stage 2 against the oracle:

* GEMM1 with the ungated SiLU epilogue (rows layout), and with SwiGLU or SiLU
  writing the sorted-slot operand tiles that GEMM2 reads (codes and scales
  bit-exact, except 32-blocks whose oracle value lies within the fp32 error
  bound of a rounding decision point; padding slots zero);
* GEMM2 (down projection + top-k weighted per-token sum) fed with tiles that
  the test builds from oracle-quantised activations, within the GEMM
  tolerance |Y - y| <= 2^-8 |y| + 2^-20 sum_k |w| sum_i |a_i w2_i|, at a small
  shape in full and at the MoE workload shape (E=896, topk=16, D=3584, I=768)
  for every token count, on sampled tokens;
* the two stages chained on the GPU against the two oracle stages chained.
"""

import numpy as np
import pytest
import torch

import mxfp4_a4w4_gemm_gb300 as a4w4
import workloads
from gpu_util import dev_bits, gemm_violations, host_bits, shuffle_tiles, unshuffle_tiles
from mxfp4_a4w4_gemm_gb300.host_prep import prepare_dense_experts_from_host
from oracle import moe, mxfp4
from test_gpu_moe import h_error_bound

pytestmark = pytest.mark.gpu

CFG = workloads.MOE
E_FULL, TOPK_FULL, D_FULL, I_FULL = CFG["experts"], CFG["topk"], CFG["model_dim"], CFG["inter_dim"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mxfp4_a4w4_gemm_gb300 import build
    build.build()
    a4w4.lib()


def h_error_bound_silu(out):
    """|h_gpu - h| for h = silu(g): fp32 accumulation (< 2^-18 of sum|x w|),
    silu's slope (< 1.1) and a few fp32 ulps."""
    g = out["gate"]
    dg = 2.0 ** -18 * out["gate_abs"] + 2.0 ** -22 * np.abs(g)
    return 1.1 * dg + 2.0 ** -19 * np.abs(moe.silu(g)) + 1e-30


def run_sort(ids, n_exp):
    T, topk = ids.shape
    maxb = a4w4.a4w4_moe_max_blocks(T, topk, n_exp, 128)
    rows = torch.empty(maxb * 128, dtype=torch.int32, device="cuda")
    bexp = torch.empty(maxb, dtype=torch.int32, device="cuda")
    nb = torch.empty(1, dtype=torch.int32, device="cuda")
    wsb = a4w4.a4w4_moe_sort_workspace_bytes(T, topk, n_exp)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    a4w4.a4w4_moe_sort(torch.from_numpy(ids).cuda(), T, topk, n_exp, 128, rows, bexp, nb, ws, wsb)
    return rows, bexp, nb


class Small:
    """A small routed problem: T tokens, n_exp experts, topk, D, I."""

    def __init__(self, act, T=19, n_exp=6, topk=2, D=512, I=256):
        self.act, self.T, self.E, self.topk, self.D, self.I = act, T, n_exp, topk, D, I
        self.X = workloads.moe_tokens_bits(T, D)
        self.ids = workloads.moe_topk_ids(T, n_exp, topk)
        rows = 2 * I if act == "swiglu" else I
        self.W1 = [workloads.moe_expert_weight_bits(e, rows, D) for e in range(n_exp)]
        if act == "swiglu":
            self.W1q = torch.empty(a4w4.a4w4_moe_w1_codes_bytes(n_exp, rows, D), dtype=torch.uint8, device="cuda")
            self.W1s = torch.empty(a4w4.a4w4_moe_w1_scales_bytes(n_exp, rows, D), dtype=torch.uint8, device="cuda")
            a4w4.a4w4_moe_prepare_w1(dev_bits(np.stack(self.W1)), n_exp, rows, D, self.W1q, self.W1s)
        else:
            self.W1q = torch.empty(n_exp * a4w4.a4w4_weight_codes_bytes(rows, D), dtype=torch.uint8, device="cuda")
            self.W1s = torch.empty(n_exp * a4w4.a4w4_weight_scales_bytes(rows, D), dtype=torch.uint8, device="cuda")
            a4w4.a4w4_prepare_gemm_weight(dev_bits(np.concatenate(self.W1)), n_exp * rows, D, self.W1q, self.W1s)
        self.rows, self.bexp, self.nb = run_sort(self.ids, n_exp)
        self.er, _, self.enb = moe.sort_routed_rows(self.ids, n_exp, 128)
        self.code = a4w4.A4W4_MOE_ACT_SWIGLU if act == "swiglu" else a4w4.A4W4_MOE_ACT_SILU

    def gemm1(self, layout, prequant):
        T, D, I = self.T, self.D, self.I
        ws, wsb = None, 0
        if prequant:
            wsb = a4w4.a4w4_moe_gemm1_workspace_bytes(T, D)
            ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        if layout == a4w4.A4W4_MOE_OUT_ROWS:
            q = torch.full((T * self.topk, I // 2), 0xEE, dtype=torch.uint8, device="cuda")
            s = torch.full((T * self.topk, I // 32), 0xEE, dtype=torch.uint8, device="cuda")
        else:
            q = torch.full((a4w4.a4w4_moe_tiles_codes_bytes(T, self.topk, self.E, I),), 0xEE, dtype=torch.uint8,
                           device="cuda")
            s = torch.full((a4w4.a4w4_moe_tiles_scales_bytes(T, self.topk, self.E, I),), 0xEE, dtype=torch.uint8,
                           device="cuda")
        a4w4.a4w4_moe_gemm1_ex(dev_bits(self.X), T, D, self.rows, self.bexp, self.nb, self.topk, self.W1q, self.W1s,
                               self.E, I, self.code, layout, q, s, ws, wsb)
        assert a4w4.a4w4_get_device_status() == 0
        return q, s

    def oracle1(self, rows):
        return moe.gemm1_rows(self.X, self.ids, lambda e: self.W1[e], rows, self.I, activation=self.act)

    def bound(self, out):
        return h_error_bound(out) if self.act == "swiglu" else h_error_bound_silu(out)


def compare_requant(gq, gs, out, bound):
    """Blocks of GPU codes/scales [R, I/2], [R, I/32] against the oracle's,
    excusing only fragile blocks.  Returns a bool per row: all blocks equal."""
    R, I2 = gq.shape
    fragile = moe.requant_fragile_blocks(out["h"], bound)
    same = np.all(gq.reshape(R, I2 // 16, 16) == out["codes"].reshape(R, I2 // 16, 16), axis=-1) & (gs == out["scales"])
    bad = ~same & ~fragile
    assert not bad.any(), f"{int(bad.sum())} non-fragile blocks differ, first {np.argwhere(bad)[:5].tolist()}"
    assert (~same).mean() < 0.02
    return np.all(same, axis=1)


@pytest.mark.parametrize("prequant", [False, True])
def test_gemm1_silu_rows(prequant):
    p = Small("silu")
    q, s = p.gemm1(a4w4.A4W4_MOE_OUT_ROWS, prequant)
    out = p.oracle1(np.arange(p.T * p.topk))
    compare_requant(q.cpu().numpy(), s.cpu().numpy(), out, p.bound(out))


def tiles_by_slot(p, q, s):
    KT = p.I // 256
    codes, scales = unshuffle_tiles(q.cpu().numpy(), s.cpu().numpy(), 128, p.enb, KT)
    return codes, scales      # [enb*128, I/2], [enb*128, I/32], row = sorted slot


@pytest.mark.parametrize("act", ["swiglu", "silu"])
@pytest.mark.parametrize("prequant", [False, True])
def test_gemm1_tiles_layout(act, prequant):
    p = Small(act)
    q, s = p.gemm1(a4w4.A4W4_MOE_OUT_TILES, prequant)
    codes, scales = tiles_by_slot(p, q, s)
    valid = p.er < p.T * p.topk
    assert np.all(codes[~valid] == 0) and np.all(scales[~valid] == 0), "padding slots must be zero"
    out = p.oracle1(p.er[valid])
    compare_requant(codes[valid], scales[valid], out, p.bound(out))


def gemm2_tiles(q_rows, s_rows, er, nb, R, I):
    """Oracle-quantised routed rows -> sorted-slot operand tiles (test code,
    the header's layout)."""
    valid = er < R
    cs = np.zeros((nb * 128, I // 2), np.uint8)
    ss = np.zeros((nb * 128, I // 32), np.uint8)
    cs[valid] = q_rows[er[valid]]
    ss[valid] = s_rows[er[valid]]
    return shuffle_tiles(cs, ss, 128, nb, I // 256)


def run_gemm2(tq, ts, T, I, rows, bexp, nb, topk, wts, W2q, W2s, E, D, maxb):
    Aq = torch.zeros(maxb * (I // 256) * 16384, dtype=torch.uint8, device="cuda")
    As = torch.zeros(maxb * (I // 256) * 1024, dtype=torch.uint8, device="cuda")
    Aq[:tq.size].copy_(torch.from_numpy(tq))
    As[:ts.size].copy_(torch.from_numpy(ts))
    wsb = a4w4.a4w4_moe_gemm2_workspace_bytes(T, topk, D)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    Y = torch.full((T, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    a4w4.a4w4_moe_gemm2(Aq, As, T, I, rows, bexp, nb, topk, torch.from_numpy(wts).cuda(), W2q, W2s, E, D, Y, ws,
                        wsb)
    assert a4w4.a4w4_get_device_status() == 0
    return host_bits(Y)


@pytest.mark.parametrize("T,E,topk,D,I", [
    (21, 6, 3, 512, 256),       # few rows per expert, one CTA per unit
    (200, 4, 2, 512, 256),      # experts with more than one 128-row block
    (37, 5, 2, 256, 1024),      # one column tile per block; I = 1024, the largest K (4 tiles resident)
    (600, 8, 4, 3584, 256),     # 378 units over 152 CTAs: runs that cross block boundaries
], ids=lambda v: str(v))
def test_gemm2_small_every_output(T, E, topk, D, I):
    ids = workloads.moe_topk_ids(T, E, topk)
    wts = workloads.moe_topk_weights(T, topk)
    H = workloads.moe_hidden_bits(T * topk, I)
    q, s = mxfp4.mxfp4_quant(H)
    W2 = [workloads.moe_expert_w2_bits(e, D, I) for e in range(E)]
    W2q = torch.empty(E * a4w4.a4w4_weight_codes_bytes(D, I), dtype=torch.uint8, device="cuda")
    W2s = torch.empty(E * a4w4.a4w4_weight_scales_bytes(D, I), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_prepare_gemm_weight(dev_bits(np.concatenate(W2)), E * D, I, W2q, W2s)
    rows, bexp, nb = run_sort(ids, E)
    er, _, enb = moe.sort_routed_rows(ids, E, 128)
    tq, ts = gemm2_tiles(q, s, er, enb, T * topk, I)
    y_gpu = run_gemm2(tq, ts, T, I, rows, bexp, nb, topk, wts, W2q, W2s, E, D, a4w4.a4w4_moe_max_blocks(T, topk, E, 128))
    y, abs_sum, yb = moe.gemm2_tokens(q, s, ids, wts, lambda e: W2[e], np.arange(T))
    bad = gemm_violations(y_gpu, y, abs_sum)[0]
    assert bad.size == 0, f"{bad.size} of {y_gpu.size} outside tolerance"
    assert np.mean(y_gpu == yb) > 0.9


@pytest.fixture(scope="module")
def full_w2():
    return prepare_dense_experts_from_host(lambda e: workloads.moe_expert_w2_bits(e, D_FULL, I_FULL), E_FULL, D_FULL,
                                           I_FULL)


@pytest.mark.parametrize("T", CFG["tokens"])
def test_gemm2_workload(T, full_w2):
    """The MoE workload shape at full size for every token count; the oracle
    checks every output of up to 4 sampled tokens (all for T = 1), and a
    second run gives the same bits for every token."""
    W2q, W2s = full_w2
    E, topk, D, I = E_FULL, TOPK_FULL, D_FULL, I_FULL
    ids = workloads.moe_topk_ids(T, E, topk)
    wts = workloads.moe_topk_weights(T, topk)
    H = workloads.moe_hidden_bits(T * topk, I)
    q, s = mxfp4.mxfp4_quant(H)
    rows, bexp, nb = run_sort(ids, E)
    er, _, enb = moe.sort_routed_rows(ids, E, 128)
    tq, ts = gemm2_tiles(q, s, er, enb, T * topk, I)
    maxb = a4w4.a4w4_moe_max_blocks(T, topk, E, 128)
    y_gpu = run_gemm2(tq, ts, T, I, rows, bexp, nb, topk, wts, W2q, W2s, E, D, maxb)
    assert np.all((y_gpu & 0x7F80) != 0x7F80), "NaN or Inf in the output"
    assert np.array_equal(y_gpu, run_gemm2(tq, ts, T, I, rows, bexp, nb, topk, wts, W2q, W2s, E, D, maxb))
    tokens = np.arange(T) if T == 1 else np.random.default_rng(T).choice(T, 4, replace=False)
    y, abs_sum, _ = moe.gemm2_tokens(q, s, ids, wts, lambda e: workloads.moe_expert_w2_bits(e, D, I), tokens)
    bad = gemm_violations(y_gpu[tokens], y, abs_sum)[0]
    assert bad.size == 0, f"{bad.size} of {y.size} sampled outputs outside tolerance"


@pytest.mark.parametrize("act", ["swiglu", "silu"])
def test_two_stages_chained(act):
    """GPU GEMM1 (tiles) -> GPU GEMM2 against oracle GEMM1 -> oracle GEMM2.
    Tokens whose routed rows all requantised to the oracle's codes (nearly
    all: a block differs only next to a rounding decision point) must match
    within the GEMM tolerance."""
    p = Small(act, T=33, n_exp=5, topk=3, D=512, I=256)
    q1, s1 = p.gemm1(a4w4.A4W4_MOE_OUT_TILES, prequant=True)
    D2 = 512
    W2 = [workloads.moe_expert_w2_bits(e, D2, p.I) for e in range(p.E)]
    W2q = torch.empty(p.E * a4w4.a4w4_weight_codes_bytes(D2, p.I), dtype=torch.uint8, device="cuda")
    W2s = torch.empty(p.E * a4w4.a4w4_weight_scales_bytes(D2, p.I), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_prepare_gemm_weight(dev_bits(np.concatenate(W2)), p.E * D2, p.I, W2q, W2s)
    wts = workloads.moe_topk_weights(p.T, p.topk)
    wsb = a4w4.a4w4_moe_gemm2_workspace_bytes(p.T, p.topk, D2)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    Y = torch.empty((p.T, D2), dtype=torch.bfloat16, device="cuda")
    a4w4.a4w4_moe_gemm2(q1, s1, p.T, p.I, p.rows, p.bexp, p.nb, p.topk, torch.from_numpy(wts).cuda(), W2q, W2s,
                        p.E, D2, Y, ws, wsb)
    assert a4w4.a4w4_get_device_status() == 0
    y_gpu = host_bits(Y)
    out = p.oracle1(np.arange(p.T * p.topk))
    # which routed rows did GPU GEMM1 requantise exactly as the oracle?
    codes, scales = tiles_by_slot(p, q1, s1)
    valid = p.er < p.T * p.topk
    row_ok = np.zeros(p.T * p.topk, bool)
    row_ok[p.er[valid]] = compare_requant(codes[valid], scales[valid], moe.gemm1_rows(
        p.X, p.ids, lambda e: p.W1[e], p.er[valid], p.I, activation=act), p.bound(out))
    tok_ok = np.all(row_ok.reshape(p.T, p.topk), axis=1)
    assert tok_ok.mean() >= 0.8, tok_ok.mean()
    y, abs_sum, _ = moe.gemm2_tokens(out["codes"], out["scales"], p.ids, wts, lambda e: W2[e], np.nonzero(tok_ok)[0])
    bad = gemm_violations(y_gpu[tok_ok], y, abs_sum)[0]
    assert bad.size == 0, f"{bad.size} of {y.size} outputs outside tolerance"


@pytest.mark.parametrize("T,E,topk", [(21, 6, 3), (200, 4, 2)])
def test_gemm2_bitwise_deterministic(T, E, topk):
    """Each routed row is written by one CTA and a token's rows are summed in k
    order: repeated runs agree bit for bit."""
    D, I = 512, 256
    ids = workloads.moe_topk_ids(T, E, topk)
    wts = workloads.moe_topk_weights(T, topk)
    q, s = mxfp4.mxfp4_quant(workloads.moe_hidden_bits(T * topk, I))
    W2 = np.concatenate([workloads.moe_expert_w2_bits(e, D, I) for e in range(E)])
    W2q = torch.empty(E * a4w4.a4w4_weight_codes_bytes(D, I), dtype=torch.uint8, device="cuda")
    W2s = torch.empty(E * a4w4.a4w4_weight_scales_bytes(D, I), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_prepare_gemm_weight(dev_bits(W2), E * D, I, W2q, W2s)
    rows, bexp, nb = run_sort(ids, E)
    er, _, enb = moe.sort_routed_rows(ids, E, 128)
    tq, ts = gemm2_tiles(q, s, er, enb, T * topk, I)
    maxb = a4w4.a4w4_moe_max_blocks(T, topk, E, 128)
    y1 = run_gemm2(tq, ts, T, I, rows, bexp, nb, topk, wts, W2q, W2s, E, D, maxb)
    y2 = run_gemm2(tq, ts, T, I, rows, bexp, nb, topk, wts, W2q, W2s, E, D, maxb)
    assert np.array_equal(y1, y2)


def test_gemm2_expired_wait_is_reported_and_context_survives():
    """With a 1 ns wait limit the persistent walk's waits expire: it reports
    A4W4_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and returns; the
    next call with the default limit gives the same bits as a normal run."""
    T, E, topk, D, I = 600, 8, 4, 3584, 256
    ids = workloads.moe_topk_ids(T, E, topk)
    wts = workloads.moe_topk_weights(T, topk)
    q, s = mxfp4.mxfp4_quant(workloads.moe_hidden_bits(T * topk, I))
    W2 = np.concatenate([workloads.moe_expert_w2_bits(e, D, I) for e in range(E)])
    W2q = torch.empty(E * a4w4.a4w4_weight_codes_bytes(D, I), dtype=torch.uint8, device="cuda")
    W2s = torch.empty(E * a4w4.a4w4_weight_scales_bytes(D, I), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_prepare_gemm_weight(dev_bits(W2), E * D, I, W2q, W2s)
    rows, bexp, nb = run_sort(ids, E)
    er, _, enb = moe.sort_routed_rows(ids, E, 128)
    tq, ts = gemm2_tiles(q, s, er, enb, T * topk, I)
    maxb = a4w4.a4w4_moe_max_blocks(T, topk, E, 128)
    want = run_gemm2(tq, ts, T, I, rows, bexp, nb, topk, wts, W2q, W2s, E, D, maxb)
    Aq = torch.zeros(maxb * (I // 256) * 16384, dtype=torch.uint8, device="cuda")
    As = torch.zeros(maxb * (I // 256) * 1024, dtype=torch.uint8, device="cuda")
    Aq[:tq.size].copy_(torch.from_numpy(tq))
    As[:ts.size].copy_(torch.from_numpy(ts))
    wsb = a4w4.a4w4_moe_gemm2_workspace_bytes(T, topk, D)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    Y = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    w_dev = torch.from_numpy(wts).cuda()
    assert a4w4.a4w4_get_device_status() == 0
    a4w4.a4w4_set_wait_limit_ns(1)
    try:
        a4w4.a4w4_moe_gemm2(Aq, As, T, I, rows, bexp, nb, topk, w_dev, W2q, W2s, E, D, Y, ws, wsb)
        status = a4w4.a4w4_get_device_status()
    finally:
        a4w4.a4w4_set_wait_limit_ns(0)
    assert status == a4w4.A4W4_ERR_TIMEOUT
    assert a4w4.a4w4_get_device_status() == 0
    a4w4.a4w4_moe_gemm2(Aq, As, T, I, rows, bexp, nb, topk, w_dev, W2q, W2s, E, D, Y, ws, wsb)
    assert a4w4.a4w4_get_device_status() == 0
    assert np.array_equal(host_bits(Y), want)
