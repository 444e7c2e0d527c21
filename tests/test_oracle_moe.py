"""Pins for oracle.moe (CPU only): sort by hand and by invariants, SwiGLU
closed forms, GEMM1 (SwiGLU and SiLU) by an independent scalar computation,
GEMM2 by exact rationals with an independent MXFP4 decoder, its reduction to
the dense GEMM, its linearity in the top-k weights and its per-token sum, and
the fragility test used to excuse requant mismatches that sit on a rounding
boundary."""

import math
from fractions import Fraction

import numpy as np

import workloads
from oracle import gemm, moe, mxfp4
from test_oracle_gemm import brute_quant_row, bf16_value, exact_bf16_bits


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


E2M1_FRACTION = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]


def decode_row_exact(packed, scales):
    """Independent MXFP4 decoder (exact rationals): element 2j in the low
    nibble of byte j, sign bit 3, magnitude index bits 0-2; scale 2^(e8m0-127)."""
    out = []
    for j, byte in enumerate(packed):
        for code in (int(byte) & 0xF, int(byte) >> 4):
            i = len(out)
            v = E2M1_FRACTION[code & 7] * Fraction(2) ** (int(scales[i // 32]) - 127)
            out.append(-v if code & 8 else v)
    return out


def test_gemm1_silu_matches_scalar_brute_force():
    """Ungated SiLU epilogue: W1[e] is [I, D] and h = silu(x . w)."""
    T, E, topk, D, I = 2, 2, 2, 64, 64
    rng = np.random.default_rng(7)
    X = workloads.to_bf16_bits(rng.standard_normal((T, D)).astype(np.float32))
    W1 = [workloads.to_bf16_bits((rng.standard_normal((I, D)) * 0.3).astype(np.float32)) for _ in range(E)]
    ids = np.array([[0, 1], [1, 0]])
    rows = np.arange(T * topk)
    out = moe.gemm1_rows(X, ids, lambda e: W1[e], rows, I, activation="silu")
    assert "up" not in out
    for r in rows:
        t, k = divmod(int(r), topk)
        x = brute_quant_row([bf16_value(v) for v in X[t]])
        h = []
        for j in range(I):
            w = brute_quant_row([bf16_value(v) for v in W1[ids[t, k]][j]])
            g = float(sum(a * b for a, b in zip(x, w)))
            h.append(g / (1.0 + math.exp(-g)))
        assert np.allclose(out["h"][r], h, rtol=1e-13, atol=1e-300)
        codes, e8 = mxfp4.quantize_blocks(np.array(h)[None, :])
        assert np.array_equal(out["codes"][r], mxfp4.pack_codes(codes)[0])
        assert np.array_equal(out["scales"][r], e8[0])


def _gemm2_problem(T, topk, E, D, I, seed=3):
    rng = np.random.default_rng(seed)
    H = workloads.to_bf16_bits((rng.standard_normal((T * topk, I)) * 2.0).astype(np.float32))
    q, s = mxfp4.mxfp4_quant(H)
    W2 = [workloads.to_bf16_bits((rng.standard_normal((D, I)) * 0.3).astype(np.float32)) for _ in range(E)]
    ids = np.stack([rng.choice(E, topk, replace=False) for _ in range(T)])
    # signed weights (some negative) so that |w| in the magnitude sum is pinned too
    sign = np.where((np.arange(T)[:, None] + np.arange(topk)[None, :]) % 2 == 0, 1.0, -1.0)
    wts = ((rng.random((T, topk)) + 0.25) * sign).astype(np.float32)
    return H, q, s, W2, ids, wts


def test_gemm2_matches_exact_rational_brute_force():
    T, topk, E, D, I = 3, 2, 3, 16, 64
    _, q, s, W2, ids, wts = _gemm2_problem(T, topk, E, D, I)
    y, abs_sum, bits = moe.gemm2_tokens(q, s, ids, wts, lambda e: W2[e], np.arange(T))
    for t in range(T):
        for n in range(D):
            exact, absx = Fraction(0), Fraction(0)
            for k in range(topk):
                r = t * topk + k
                a = decode_row_exact(q[r], s[r])
                w = brute_quant_row([bf16_value(v) for v in W2[ids[t, k]][n]])
                dot = sum(x * z for x, z in zip(a, w))
                exact += Fraction(float(wts[t, k])) * dot
                absx += abs(Fraction(float(wts[t, k]))) * sum(abs(x * z) for x, z in zip(a, w))
            assert abs(Fraction(y[t, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)
            assert abs(Fraction(abs_sum[t, n]) - absx) <= absx * Fraction(1, 2 ** 50)
            assert bits[t, n] == exact_bf16_bits(exact)


def test_gemm2_with_one_unit_weight_is_the_dense_gemm():
    """topk = 1, weight 1: the down projection of each routed row is the dense
    A4W4 GEMM of GEMM1's activations against W2 (fixes the contraction axis)."""
    T, topk, E, D, I = 5, 1, 1, 256, 128
    H, q, s, W2, ids, _ = _gemm2_problem(T, topk, E, D, I, seed=4)
    y, abs_sum, bits = moe.gemm2_tokens(q, s, np.zeros((T, 1), int), np.ones((T, 1), np.float32),
                                        lambda e: W2[0], np.arange(T))
    ref, ref_abs, cref = gemm.gemm_a4w4(H, W2[0])
    assert np.allclose(y, ref, rtol=1e-12, atol=0) and np.allclose(abs_sum, ref_abs, rtol=1e-12, atol=0)
    assert np.array_equal(bits, cref)


def test_gemm2_weights_scale_and_rows_sum_per_token():
    T, topk, E, D, I = 4, 3, 5, 32, 64
    _, q, s, W2, ids, wts = _gemm2_problem(T, topk, E, D, I, seed=5)
    f = lambda e: W2[e]      # noqa: E731
    y, _, _ = moe.gemm2_tokens(q, s, ids, wts, f, np.arange(T))
    # doubling every weight doubles y exactly (powers of two scale exactly)
    y2, _, _ = moe.gemm2_tokens(q, s, ids, 2 * wts, f, np.arange(T))
    assert np.array_equal(y2, 2 * y)
    # y is the sum over k of the single-route contributions of the same token
    parts = []
    for k in range(topk):
        w1 = np.zeros_like(wts)
        w1[:, k] = wts[:, k]
        parts.append(moe.gemm2_tokens(q, s, ids, w1, f, np.arange(T))[0])
    assert np.allclose(y, sum(parts), rtol=1e-12, atol=1e-300)
    # reordering a token's k slots (rows, ids and weights together) changes nothing
    perm = [2, 0, 1]
    q3 = q.reshape(T, topk, -1)[:, perm].reshape(T * topk, -1)
    s3 = s.reshape(T, topk, -1)[:, perm].reshape(T * topk, -1)
    yp, _, _ = moe.gemm2_tokens(q3, s3, ids[:, perm], wts[:, perm], f, np.arange(T))
    assert np.allclose(yp, y, rtol=1e-12, atol=1e-300)
    # a subset of tokens gives those rows of the full result
    ys, _, _ = moe.gemm2_tokens(q, s, ids, wts, f, [3, 1])
    assert np.array_equal(ys, y[[3, 1]])


def test_sort_aux_arrays_by_hand_and_invariants():
    ids = np.array([[2, 0], [0, 3], [2, 1]])
    rows, experts, nb = moe.sort_routed_rows(ids, 4, 2)          # [1, 2, 5, S, 0, 4, 3, S]
    tok, slot = moe.sort_aux_arrays(rows, 3, 2)
    assert list(tok) == [0, 1, 2, 3, 0, 2, 1, 3]                 # token of each slot, T for padding
    assert list(slot) == [4, 0, 1, 6, 5, 2]                      # slot of each routed row
    for T in (1, 37, 256):
        ids = workloads.moe_topk_ids(T, 896, 16)
        for bm in (16, 128):
            rows, experts, nb = moe.sort_routed_rows(ids, 896, bm)
            tok, slot = moe.sort_aux_arrays(rows, T, 16)
            assert np.array_equal(rows[slot], np.arange(T * 16))       # inverse permutation
            real = rows < T * 16
            assert np.array_equal(tok[real], rows[real] // 16) and np.all(tok[~real] == T)
            # a block's tokens are distinct (topk experts per token are distinct)
            for b in range(nb):
                t = tok[b * bm:(b + 1) * bm]
                t = t[t < T]
                assert np.unique(t).size == t.size
