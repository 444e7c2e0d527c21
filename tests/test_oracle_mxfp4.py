"""Pins for oracle.mxfp4 against the MXFP4 definition (CPU only).

Each test ties the oracle to something other than itself: the E2M1 bit-field
definition, an independent brute-force nearest-value rounding, hand-derived
worked values, closed forms of the scale rule, invariants, and torch's BF16
conversion (a library routine).
"""

import json
import os

import numpy as np
import pytest
import torch

from oracle import mxfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def e2m1_value_from_bits(code):
    """E2M1 per the OCP MX v1.0 element format: 1 sign, 2 exponent (bias 1), 1 mantissa."""
    s, E, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = (m * 0.5) if E == 0 else (2.0 ** (E - 1)) * (1.0 + m / 2.0)
    return -mag if s else mag


def brute_force_index(y):
    """Nearest E2M1 magnitude index to y >= 0; on equal distance the even index."""
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    return min(range(8), key=lambda i: (abs(y - grid[i]), i % 2))


def test_e2m1_table_matches_bit_field_definition():
    codes = np.arange(16, dtype=np.uint8)
    block = np.tile(codes, 2)                        # 32 codes, scale 2^0
    vals = mxfp4.decode(block[None, :], np.array([[127]], dtype=np.uint8))[0]
    for c in range(16):
        want = e2m1_value_from_bits(c)
        assert vals[c] == want
        assert np.signbit(vals[c]) == bool(c & 8)               # sign bit, including -0


@pytest.mark.parametrize("y,idx", [
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),    # ties -> even
    (0.2499, 0), (0.2501, 1), (6.0, 7), (6.5, 7), (7.9375, 7), (1e30, 7),        # near ties, saturation
])
def test_rounding_ties_and_saturation(y, idx):
    assert mxfp4.e2m1_round_index(np.array([y]))[0] == idx


def test_rounding_matches_brute_force_on_all_bf16_magnitudes():
    bits = np.arange(0, 0x7F80, dtype=np.uint16)             # every finite non-negative BF16
    y = mxfp4.bf16_bits_to_f64(bits)
    got = mxfp4.e2m1_round_index(y)
    # brute force over the values that can land anywhere but index 0 or 7
    sel = (y >= 0.125) & (y <= 8.0)
    want = np.array([brute_force_index(v) for v in y[sel]])
    assert np.array_equal(got[sel], want)
    assert np.all(got[y < 0.25] == 0) and np.all(got[y > 5.0] == 7)
    rng = np.random.default_rng(5)
    r = rng.uniform(0, 8, 20000)
    assert np.array_equal(mxfp4.e2m1_round_index(r), [brute_force_index(v) for v in r])


def test_scale_rule_closed_form():
    for p in range(-125, 126):
        for f in (1.0, 1.5, 1.9921875):
            assert mxfp4.e8m0_exponent(np.array([f * 2.0 ** p]))[0] == p - 2
    assert mxfp4.e8m0_exponent(np.array([0.0]))[0] == -127
    assert mxfp4.e8m0_exponent(np.array([2.0 ** -130]))[0] == -127       # clamped
    assert mxfp4.e8m0_exponent(np.array([2.0 ** -125]))[0] == -127
    assert mxfp4.e8m0_exponent(np.array([2.0 ** 127 * 1.99]))[0] == 125


def test_scale_invariants_on_random_blocks():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((4000, 32)) * np.ldexp(1.0, rng.integers(-110, 110, (4000, 1)))
    x[::17] = 0.0
    codes, e8 = mxfp4.quantize_blocks(x)
    e = e8.astype(np.int64)[:, 0] - 127
    amax = np.abs(x).max(axis=1)
    nz = amax > 0
    r = amax[nz] / np.ldexp(1.0, e[nz])
    assert np.all((r >= 4.0) & (r < 8.0))                 # amax / 2^e in [4, 8)
    assert np.all(e[~nz] == -127)
    dec = mxfp4.decode(codes, e8)
    assert np.all(np.abs(dec) <= 6.0 * np.ldexp(1.0, e)[:, None])
    # each element's error is at most half the E2M1 spacing around it, or the saturation gap
    err = np.abs(dec - x) / np.ldexp(1.0, e)[:, None]
    assert np.all(err <= np.maximum(1.0, np.abs(x) / np.ldexp(1.0, e)[:, None] - 6.0) + 1e-12)


def test_lossless_roundtrip_on_grid_values():
    rng = np.random.default_rng(11)
    mags = mxfp4.E2M1_MAGNITUDE
    for e in (-127, -100, -3, 0, 5, 90):
        v = mags[rng.integers(0, 8, (64, 32))] * np.where(rng.random((64, 32)) < 0.5, -1, 1)
        v[:, 0] = np.where(rng.random(64) < 0.5, 4.0, 6.0)          # amax in [4, 8)
        x = np.ldexp(v, e)
        if e == -127:
            continue  # 4 * 2^-127 has floor(log2) = -125 -> e = -127: still lossless, checked below
        assert np.array_equal(mxfp4.quant_dequant(x), x)
    x = np.ldexp(np.array([[4.0, 0.5, -1.5] + [0.0] * 29]), -125)       # e = -127 exactly
    assert np.array_equal(mxfp4.quant_dequant(x), x)


def test_sign_of_zero_results():
    x = np.zeros((1, 32))
    x[0, 0] = -0.0
    x[0, 1] = -1e-3
    x[0, 2] = 1.0
    codes, _ = mxfp4.quantize_blocks(x)
    assert codes[0, 0] == 8 and codes[0, 1] == 8 and codes[0, 3] == 0


def test_nibble_order_and_roundtrip():
    c = np.array([2, 15, 0, 8], dtype=np.uint8)
    assert list(mxfp4.pack_codes(c)) == [0xF2, 0x80]
    rng = np.random.default_rng(3)
    c = rng.integers(0, 16, (5, 64)).astype(np.uint8)
    assert np.array_equal(mxfp4.unpack_codes(mxfp4.pack_codes(c)), c)


def test_worked_example_golden():
    d = json.load(open(os.path.join(GOLDEN, "mxfp4_worked_example.json")))
    row = np.zeros(32 * len(d["blocks"]))
    for b, blk in enumerate(d["blocks"]):
        for i, h in enumerate(blk["x"]):
            row[32 * b + i] = float.fromhex(h)
    bits = mxfp4.round_to_bf16_bits(row)
    assert np.array_equal(mxfp4.bf16_bits_to_f64(bits), row)         # inputs are BF16-exact
    assert np.array_equal(np.signbit(mxfp4.bf16_bits_to_f64(bits)), np.signbit(row))
    packed, scales = mxfp4.mxfp4_quant(bits[None, :])
    assert packed[0].tobytes().hex() == d["packed_hex"]
    assert list(scales[0]) == d["scales"]


def test_bf16_rounding_matches_torch_for_float32_inputs():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(200000) * np.ldexp(1.0, rng.integers(-140, 126, 200000))).astype(np.float32)
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = mxfp4.round_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_rounding_float64_nearest_neighbour():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(3000) * np.ldexp(1.0, rng.integers(-135, 126, 3000))
    got = mxfp4.round_to_bf16_bits(x)
    for v, g in zip(x, got):
        # the two BF16 neighbours of v from float32 truncation, chosen by exact distance
        f = np.float32(v)
        lo_bits = int(np.array([f], np.float32).view(np.uint32)[0] >> 16)
        cands = {lo_bits, lo_bits + 1, lo_bits - 1}
        vals = {c: float(np.array([c << 16], np.uint32).view(np.float32)[0]) for c in cands if 0 <= c < 0x10000}
        best = min(vals, key=lambda c: (abs(vals[c] - v), c & 1))
        assert int(g) == best


def test_mxfp4_quant_shapes():
    bits = np.zeros((3, 128), dtype=np.uint16)
    q, s = mxfp4.mxfp4_quant(bits)
    assert q.shape == (3, 64) and s.shape == (3, 4)
    assert np.all(q == 0) and np.all(s == 0)
