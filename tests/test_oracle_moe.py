"""Pins for oracle.moe (CPU only): sort by hand and by invariants, SwiGLU
closed forms, GEMM1 by an independent scalar computation, and the fragility
test used to excuse requant mismatches that sit on a rounding boundary."""

import math

import numpy as np

import workloads
from oracle import moe, mxfp4
from test_oracle_gemm import brute_quant_row, bf16_value


def test_sort_by_hand():
    ids = np.array([[2, 0], [0, 3], [2, 1]])        # rows r = t*2 + k: 0->2 1->0 2->0 3->3 4->2 5->1
    rows, experts, nb = moe.sort_routed_rows(ids, 4, 2)
    S = 6
    assert nb == 4
    assert list(experts) == [0, 1, 2, 3]
    assert list(rows) == [1, 2, 5, S, 0, 4, 3, S]


def test_sort_invariants():
    for T in (1, 16, 256):
        ids = workloads.moe_topk_ids(T, 896, 16)
        for bm in (16, 128):
            rows, experts, nb = moe.sort_routed_rows(ids, 896, bm)
            S = T * 16
            assert rows.size == nb * bm
            real = rows[rows != S]
            assert np.array_equal(np.sort(real), np.arange(T * 16))          # a permutation
            counts = np.bincount(ids.reshape(-1), minlength=896)
            assert nb == int(np.sum(-(-counts // bm)))
            flat = ids.reshape(-1)
            for b in range(nb):
                blk = rows[b * bm:(b + 1) * bm]
                r = blk[blk != S]
                assert np.all(flat[r] == experts[b])                         # single expert
                assert np.all(np.diff(r) > 0)
            assert np.all(np.diff(experts) >= 0)


def test_topk_ids_distinct():
    ids = workloads.moe_topk_ids(64, 896, 16)
    assert all(len(set(r)) == 16 for r in ids.tolist())


def test_silu_closed_forms():
    l3 = math.log(3.0)
    got = moe.silu(np.array([0.0, l3, -l3, 60.0, -800.0]))
    assert got[0] == 0.0
    assert abs(got[1] - 0.75 * l3) < 1e-15 and abs(got[2] + 0.25 * l3) < 1e-15
    assert abs(got[3] - 60.0) < 1e-12
    assert got[4] == 0.0


def test_gemm1_matches_scalar_brute_force():
    T, E, topk, D, I = 3, 3, 2, 64, 64
    rng = np.random.default_rng(1)
    X = workloads.to_bf16_bits(rng.standard_normal((T, D)).astype(np.float32))
    W1 = [workloads.to_bf16_bits((rng.standard_normal((2 * I, D)) * 0.3).astype(np.float32)) for _ in range(E)]
    ids = np.array([[0, 2], [1, 0], [2, 1]])
    rows = np.arange(T * topk)
    out = moe.gemm1_rows(X, ids, lambda e: W1[e], rows, I)
    for r in rows:
        t, k = divmod(int(r), topk)
        e = ids[t, k]
        x = brute_quant_row([bf16_value(v) for v in X[t]])
        h = []
        for j in range(I):
            wg = brute_quant_row([bf16_value(v) for v in W1[e][j]])
            wu = brute_quant_row([bf16_value(v) for v in W1[e][I + j]])
            g = float(sum(a * b for a, b in zip(x, wg)))
            u = float(sum(a * b for a, b in zip(x, wu)))
            h.append(g / (1.0 + math.exp(-g)) * u)
        assert np.allclose(out["h"][r], h, rtol=1e-13, atol=1e-300)
        codes, e8 = mxfp4.quantize_blocks(np.array(h)[None, :])
        assert np.array_equal(out["codes"][r], mxfp4.pack_codes(codes)[0])
        assert np.array_equal(out["scales"][r], e8[0])


def test_gate_rows_come_first():
    T, E, topk, D, I = 1, 1, 1, 32, 32
    X = workloads.to_bf16_bits(np.ones((1, D), np.float32))
    W = np.zeros((2 * I, D), np.float32)
    W[:I] = 0.5                   # gate = 16 * ... large positive -> silu(g) ~ g
    W[I:] = 0.0                   # up = 0 -> h = 0
    out = moe.gemm1_rows(X, np.zeros((1, 1), int), lambda e: workloads.to_bf16_bits(W), [0], I)
    assert np.all(out["h"] == 0) and np.all(out["gate"] > 0)
    W[:I], W[I:] = 0.0, 0.5       # gate = 0 -> silu = 0 -> h = 0, up > 0
    out = moe.gemm1_rows(X, np.zeros((1, 1), int), lambda e: workloads.to_bf16_bits(W), [0], I)
    assert np.all(out["h"] == 0) and np.all(out["up"] > 0)


def test_fragile_blocks():
    h = np.zeros((1, 64))
    h[0, :32] = np.linspace(0.1, 1.0, 32) * 4.0         # amax 4.0 exactly: a power of two
    h[0, 32] = 6.0
    h[0, 33] = 2.5                                        # y = 2.5: a rounding midpoint at e = 0
    h[0, 34:] = 0.3
    f0 = moe.requant_fragile_blocks(h, np.zeros_like(h))
    assert not f0.any()
    f1 = moe.requant_fragile_blocks(h, np.full_like(h, 1e-9))
    assert f1[0, 0] and f1[0, 1]
    h[0, :32] = 3.0
    h[0, 33] = 2.2
    f2 = moe.requant_fragile_blocks(h, np.full_like(h, 1e-9))
    assert not f2.any()
