"""GPU parity: the routed-row sort (bit-exact) and the grouped MoE GEMM1 with
SwiGLU + MXFP4 requant (codes and scales bit-exact, except 32-blocks whose
oracle value lies within the fp32 error bound of a rounding decision point)."""

import numpy as np
import pytest
import torch

import mxfp4_a4w4_gemm_gb300 as a4w4
import workloads
from gpu_util import dev_bits
from mxfp4_a4w4_gemm_gb300.host_prep import prepare_moe_w1_from_host
from oracle import moe

pytestmark = pytest.mark.gpu

CFG = workloads.MOE
E, TOPK, D, I = CFG["experts"], CFG["topk"], CFG["model_dim"], CFG["inter_dim"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mxfp4_a4w4_gemm_gb300 import build
    build.build()
    a4w4.lib()


def run_sort(ids, n_exp, bm):
    T, topk = ids.shape
    maxb = a4w4.a4w4_moe_max_blocks(T, topk, n_exp, bm)
    rows = torch.full((maxb * bm,), -7, dtype=torch.int32, device="cuda")
    bexp = torch.full((maxb,), -7, dtype=torch.int32, device="cuda")
    nb = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsb = a4w4.a4w4_moe_sort_workspace_bytes(T, topk, n_exp)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    a4w4.a4w4_moe_sort(torch.from_numpy(ids).cuda(), T, topk, n_exp, bm, rows, bexp, nb, ws, wsb)
    assert a4w4.a4w4_get_device_status() == 0
    return rows, bexp, nb


def test_sort_by_hand():
    ids = np.array([[2, 0], [0, 3], [2, 1]], dtype=np.int32)
    rows, bexp, nb = run_sort(ids, 4, 16)
    assert int(nb.item()) == 4
    r = rows.cpu().numpy()
    assert list(r[:16][:2]) == [1, 2] and list(r[16:18]) == [5, 6] and list(r[32:34]) == [0, 4]
    assert list(bexp.cpu().numpy()[:4]) == [0, 1, 2, 3]


@pytest.mark.parametrize("T", CFG["tokens"])
@pytest.mark.parametrize("bm", [16, 128])
def test_sort_bit_exact(T, bm):
    ids = workloads.moe_topk_ids(T, E, TOPK)
    rows, bexp, nb = run_sort(ids, E, bm)
    er, ee, enb = moe.sort_routed_rows(ids, E, bm)
    assert int(nb.item()) == enb
    assert np.array_equal(rows.cpu().numpy()[:enb * bm], er)
    assert np.array_equal(bexp.cpu().numpy()[:enb], ee)


def run_sort_aux(ids, n_exp, bm, ws=None):
    T, topk = ids.shape
    maxb = a4w4.a4w4_moe_max_blocks(T, topk, n_exp, bm)
    rows = torch.full((maxb * bm,), -7, dtype=torch.int32, device="cuda")
    toks = torch.full((maxb * bm,), -7, dtype=torch.int32, device="cuda")
    slot = torch.full((T * topk,), -7, dtype=torch.int32, device="cuda")
    bexp = torch.full((maxb,), -7, dtype=torch.int32, device="cuda")
    nb = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsb = a4w4.a4w4_moe_sort_aux_workspace_bytes(T, topk, n_exp)
    if ws is None:
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        a4w4.a4w4_workspace_init(ws, wsb)
    a4w4.a4w4_moe_sort_aux(torch.from_numpy(ids).cuda(), T, topk, n_exp, bm, rows, bexp, nb, toks, slot, ws, wsb)
    assert a4w4.a4w4_get_device_status() == 0
    return rows, bexp, nb, toks, slot, ws


@pytest.mark.parametrize("T,n_exp,topk", [(1, E, TOPK), (2, E, TOPK), (3, E, TOPK), (16, E, TOPK), (256, E, TOPK),
                                          (4096, E, TOPK), (37, 5, 3), (3000, 64, 8), (1, 4096, 1)])
@pytest.mark.parametrize("bm", [16, 128])
def test_sort_aux_bit_exact(T, n_exp, topk, bm):
    """The single-launch sort: sorted rows, block experts and block count equal
    the oracle's, and the gather/scatter arrays equal the oracle's; twice in a
    row on one workspace (the grid barrier resets itself)."""
    ids = workloads.moe_topk_ids(T, n_exp, topk)
    er, ee, enb = moe.sort_routed_rows(ids, n_exp, bm)
    et, es = moe.sort_aux_arrays(er, T, topk)
    ws = None
    for _ in range(2):
        rows, bexp, nb, toks, slot, ws = run_sort_aux(ids, n_exp, bm, ws)
        assert int(nb.item()) == enb
        assert np.array_equal(rows.cpu().numpy()[:enb * bm], er)
        assert np.array_equal(bexp.cpu().numpy()[:enb], ee)
        assert np.array_equal(toks.cpu().numpy()[:enb * bm], et)
        assert np.array_equal(slot.cpu().numpy(), es)


@pytest.mark.parametrize("bm", [16, 32])
def test_sort_aux_repeated_experts(bm):
    """Rows that repeat an expert (more than a block's worth in the one-warp
    path for up to 32 rows, and in the one-CTA path), and an expert id outside
    [0, E) that is not routed."""
    cases = [np.array([[3] * 20 + [1] * 5 + [3] * 7], dtype=np.int32),          # 32 rows, one token
             np.array([[2, 2, 0], [2, 9, 1], [0, 2, 2]] * 13, dtype=np.int32)]   # 117 rows, id 9 >= E
    for ids in cases:
        T, topk = ids.shape
        n_exp = 4 if ids.max() > 3 else 8
        er, ee, enb = moe.sort_routed_rows(np.where(ids < n_exp, ids, -1), n_exp, bm)
        rows, bexp, nb, toks, slot, _ = run_sort_aux(ids, n_exp, bm)
        et, es = moe.sort_aux_arrays(er, T, topk)
        assert int(nb.item()) == enb
        assert np.array_equal(rows.cpu().numpy()[:enb * bm], er)
        assert np.array_equal(bexp.cpu().numpy()[:enb], ee)
        assert np.array_equal(toks.cpu().numpy()[:enb * bm], et)
        assert np.array_equal(slot.cpu().numpy(), es)


def h_error_bound(out):
    """Per-element bound on |h_gpu - h|: fp32 accumulation of 3584/64 = 56 MMA
    partial sums (at most 56 * 2^-24 < 2^-18 of sum|x w|), then silu and the
    product in fp32 (a few ulps)."""
    g, u = out["gate"], out["up"]
    dg = 2.0 ** -18 * out["gate_abs"] + 2.0 ** -22 * np.abs(g)
    du = 2.0 ** -18 * out["up_abs"] + 2.0 ** -22 * np.abs(u)
    s = moe.silu(g)
    return 1.1 * np.abs(u) * dg + np.abs(s) * du + 2.0 ** -19 * np.abs(s * u) + 1e-30


def run_gemm1(X_bits, ids, W1q, W1s, n_exp, inter, prequant=False):
    """prequant: tokens quantised once into a workspace, else inline per tile."""
    T = X_bits.shape[0]
    topk = ids.shape[1]
    Dm = X_bits.shape[1]
    rows, bexp, nb = run_sort(ids, n_exp, 128)
    out_q = torch.full((T * topk, inter // 2), 0xEE, dtype=torch.uint8, device="cuda")
    out_s = torch.full((T * topk, inter // 32), 0xEE, dtype=torch.uint8, device="cuda")
    ws, wsb = None, 0
    if prequant:
        wsb = a4w4.a4w4_moe_gemm1_workspace_bytes(T, Dm)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    a4w4.a4w4_moe_gemm1(dev_bits(X_bits), T, Dm, rows, bexp, nb, topk, W1q, W1s, n_exp, inter, out_q, out_s,
                        ws, wsb)
    assert a4w4.a4w4_get_device_status() == 0
    return out_q.cpu().numpy(), out_s.cpu().numpy()


def check_rows(q, s, X_bits, ids, expert_bits, rows, inter):
    out = moe.gemm1_rows(X_bits, ids, expert_bits, rows, inter)
    fragile = moe.requant_fragile_blocks(out["h"], h_error_bound(out))
    gq = q[rows].reshape(len(rows), inter // 32, 16)
    eq = out["codes"].reshape(len(rows), inter // 32, 16)
    same = np.all(gq == eq, axis=-1) & (s[rows] == out["scales"])
    bad = ~same & ~fragile
    assert not bad.any(), f"{int(bad.sum())} non-fragile blocks differ, first {np.argwhere(bad)[:5].tolist()}"
    # the excuse must stay narrow: few blocks near a decision point, fewer differing
    differ = float((~same).mean())
    print(f"requant blocks: {same.size} checked, {differ:.4%} differ, {fragile.mean():.4%} within the error bound")
    assert fragile.mean() < 0.15 and differ < 0.02, (fragile.mean(), differ)
    return int((~same).sum()), int(fragile.sum())


@pytest.mark.parametrize("prequant", [False, True])
def test_gemm1_small(prequant):
    T, n_exp, topk, Dm, inter = 5, 6, 2, 256, 128
    X = workloads.moe_tokens_bits(T, Dm)
    ids = workloads.moe_topk_ids(T, n_exp, topk)
    W1 = [workloads.moe_expert_weight_bits(e, 2 * inter, Dm) for e in range(n_exp)]
    W1q = torch.empty(a4w4.a4w4_moe_w1_codes_bytes(n_exp, 2 * inter, Dm), dtype=torch.uint8, device="cuda")
    W1s = torch.empty(a4w4.a4w4_moe_w1_scales_bytes(n_exp, 2 * inter, Dm), dtype=torch.uint8, device="cuda")
    a4w4.a4w4_moe_prepare_w1(dev_bits(np.stack(W1)), n_exp, 2 * inter, Dm, W1q, W1s)
    q, s = run_gemm1(X, ids, W1q, W1s, n_exp, inter, prequant)
    check_rows(q, s, X, ids, lambda e: W1[e], np.arange(T * topk), inter)


@pytest.fixture(scope="module")
def full_w1():
    return prepare_moe_w1_from_host(lambda e: workloads.moe_expert_weight_bits(e, 2 * I, D), E, 2 * I, D)


@pytest.mark.parametrize("prequant", [False, True])
@pytest.mark.parametrize("T", CFG["tokens"])
def test_gemm1_workload(T, prequant, full_w1):
    """The MoE workload at full size; all routed rows for T = 1, else every
    routed row of 12 seeded-random experts."""
    W1q, W1s = full_w1
    X = workloads.moe_tokens_bits(T, D)
    ids = workloads.moe_topk_ids(T, E, TOPK)
    q, s = run_gemm1(X, ids, W1q, W1s, E, I, prequant)
    flat = ids.reshape(-1)
    if T == 1:
        rows = np.arange(T * TOPK)
    else:
        experts = np.random.default_rng(T).choice(np.unique(flat), 12, replace=False)
        rows = np.nonzero(np.isin(flat, experts))[0]
    assert not np.any(np.all(q == 0xEE, axis=1)), "a routed row was never written"
    check_rows(q, s, X, ids, lambda e: workloads.moe_expert_weight_bits(e, 2 * I, D), rows, I)
