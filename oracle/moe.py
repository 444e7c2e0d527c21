"""Grouped-MoE GEMM1 oracle: routed-row sort, GEMM1, SwiGLU, MXFP4 requant.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

"[gfx1250] Fuse A4W4 stage1 FP4 quantization", Summary and Performance: the
grouped MoE GEMM1 multiplies each routed token by its expert's gate+up weight
(E experts, topk experts per token, model_dim D, inter_dim I, 2I outputs per
expert), applies the activation and emits packed MXFP4 codes plus E8M0 scales
directly, the scale computed from the FP32 activation.  "[HIP] [CK] [FlyDSL]
[Kernel] Extend MXFP4 GEMM1 replacement to A4W4", Summary: rows are grouped
per expert by an auxiliary sort into blocks of block_m rows.

Readings (the pages leave these open):
* routed row r = t * topk + k carries token t to expert topk_ids[t, k];
* the sort lists, for e = 0..E-1 in order, the rows routed to e in increasing
  r, padded with the sentinel T * topk up to a multiple of block_m; block b
  holds block_m consecutive entries and belongs to one expert;
* W1[e] is [2I, D]: rows 0..I-1 are the gate projection, rows I..2I-1 the up
  projection; SwiGLU h = silu(gate) * up with silu(g) = g / (1 + exp(-g)), no
  clamp, no bias, top-k weights not applied in GEMM1;
* the gfx1250 page's Summary lists SiLU beside SwiGLU as a separate epilogue
  activation: read as the ungated form, W1[e] is [I, D] (one projection) and
  h = silu(x . w);
* h is requantised with the same MXFP4 rule as the inputs (oracle.mxfp4),
  once, from the float64 value (the gfx1250 page rounds to BF16 first; this
  library rounds once, from fp32);
* output row r of the codes [T*topk, I/2] and scales [T*topk, I/32] (plain
  row-major) belongs to routed row r.

GEMM2 (the down projection; "[HIP] [CK] [FlyDSL] [Kernel] Extend MXFP4 GEMM1
replacement to A4W4", Summary: the stage-2 paths consume stage 1's layout;
GEMM2 scope; the pages print no formula for it).  Reading: routed row r =
t*topk + k holds GEMM1's MXFP4 output a~_r (I values); W2[e] is [D, I]; the
top-k weight w[t, k] that GEMM1 did not apply is applied here, and the rows
of a token are summed:

    y[t] = sum_k  w[t, k] * (W2q[topk_ids[t, k]] @ a~_{t*topk+k})      (float64)

with W2q the MXFP4 quantisation of W2 (same rule), output BF16 [T, D].
"""

import numpy as np

from . import mxfp4


def sort_routed_rows(topk_ids, num_experts, block_m):
    """Expected (sorted_rows int32 [nb*block_m], block_expert int32 [nb], nb)."""
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, topk = ids.shape
    flat = ids.reshape(-1)
    sentinel = T * topk
    rows, experts = [], []
    for e in range(num_experts):
        r = np.nonzero(flat == e)[0]
        if r.size == 0:
            continue
        nb = -(-r.size // block_m)
        padded = np.full(nb * block_m, sentinel, dtype=np.int64)
        padded[: r.size] = r
        rows.append(padded)
        experts.extend([e] * nb)
    if not rows:
        return np.zeros(0, np.int32), np.zeros(0, np.int32), 0
    return (np.concatenate(rows).astype(np.int32), np.asarray(experts, np.int32),
            len(experts))


def sort_aux_arrays(sorted_rows, num_tokens, topk):
    """Gather and scatter indices that accompany the sort ("[HIP] [CK]
    [FlyDSL] [Kernel] Extend MXFP4 GEMM1 replacement to A4W4", Summary: the
    adaptive MoE auxiliary sort; the review names the aux arrays that the sort
    emits for A4W4).  Reading: for every sorted slot s, the token whose row
    it holds (sorted_tokens[s] = sorted_rows[s] // topk, or num_tokens for a
    padding slot), and for every routed row r the slot that holds it
    (row_slot[sorted_rows[s]] = s).  Returns (sorted_tokens, row_slot), int32."""
    rows = np.asarray(sorted_rows, dtype=np.int64)
    sentinel = num_tokens * topk
    tokens = np.where(rows < sentinel, rows // topk, num_tokens)
    row_slot = np.full(sentinel, -1, dtype=np.int64)
    for s, r in enumerate(rows):
        if r < sentinel:
            row_slot[r] = s
    return tokens.astype(np.int32), row_slot.astype(np.int32)


def silu(g):
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def gemm1_rows(X_bits, topk_ids, expert_weight_bits, rows, inter_dim, activation="swiglu"):
    """Oracle GEMM1 + activation + requant for the routed rows ``rows``.

    X_bits [T, D] BF16 bits; expert_weight_bits(e) -> BF16 bits of W1[e]:
    [2I, D] for activation "swiglu" (h = silu(gate) * up), [I, D] for "silu"
    (h = silu(gate)).  Returns a dict of float64 gate (and up) and their |.|
    sums [R, I], h [R, I], the expected packed codes uint8 [R, I/2] and E8M0
    scales uint8 [R, I/32].
    """
    assert activation in ("swiglu", "silu")
    ids = np.asarray(topk_ids, dtype=np.int64)
    topk = ids.shape[1]
    rows = np.asarray(rows, dtype=np.int64)
    I = inter_dim
    x = {}
    wq = {}
    keys = ("gate", "up", "gate_abs", "up_abs") if activation == "swiglu" else ("gate", "gate_abs")
    out = {k: np.empty((rows.size, I)) for k in keys}
    for i, r in enumerate(rows):
        t, k = divmod(int(r), topk)
        e = int(ids[t, k])
        if t not in x:
            x[t] = mxfp4.quant_dequant(mxfp4.bf16_bits_to_f64(X_bits[t]))
        if e not in wq:
            wq[e] = mxfp4.quant_dequant(mxfp4.bf16_bits_to_f64(expert_weight_bits(e)))
        w = wq[e]
        out["gate"][i] = w[:I] @ x[t]
        out["gate_abs"][i] = np.abs(w[:I]) @ np.abs(x[t])
        if activation == "swiglu":
            out["up"][i] = w[I:] @ x[t]
            out["up_abs"][i] = np.abs(w[I:]) @ np.abs(x[t])
    h = silu(out["gate"]) * out["up"] if activation == "swiglu" else silu(out["gate"])
    codes, e8m0 = mxfp4.quantize_blocks(h)
    out.update(h=h, codes=mxfp4.pack_codes(codes), scales=e8m0)
    return out


def gemm2_tokens(a_codes, a_scales, topk_ids, topk_weights, expert_weight_bits, tokens):
    """Oracle MoE GEMM2 (down projection + top-k weighted sum) for ``tokens``.

    a_codes uint8 [T*topk, I/2] packed MXFP4 codes and a_scales uint8
    [T*topk, I/32] E8M0 scales of every routed row (GEMM1's output, plain
    row-major); topk_weights float32 [T, topk]; expert_weight_bits(e) -> BF16
    bits [D, I] of W2[e].  Returns (y float64 [n, D], abs_sum float64 [n, D]
    = sum_k |w| * sum_i |a~_i w2_i|, y rounded to BF16 bits uint16 [n, D]).
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    topk = ids.shape[1]
    wts = np.asarray(topk_weights, dtype=np.float32).astype(np.float64)
    tokens = np.asarray(tokens, dtype=np.int64)
    w2 = {}
    y = None
    for i, t in enumerate(tokens):
        for k in range(topk):
            r = int(t) * topk + k
            e = int(ids[t, k])
            if e not in w2:
                w2[e] = mxfp4.quant_dequant(mxfp4.bf16_bits_to_f64(expert_weight_bits(e)))
            a = mxfp4.decode(mxfp4.unpack_codes(a_codes[r]), a_scales[r])
            if y is None:
                D = w2[e].shape[0]
                y = np.zeros((tokens.size, D))
                abs_sum = np.zeros((tokens.size, D))
            y[i] += wts[t, k] * (w2[e] @ a)
            abs_sum[i] += abs(wts[t, k]) * (np.abs(w2[e]) @ np.abs(a))
    return y, abs_sum, mxfp4.round_to_bf16_bits(y)


def requant_fragile_blocks(h, delta):
    """Blocks whose MXFP4 result could change under a perturbation <= delta.

    h [R, I] float64 oracle values, delta [R, I] per-element error bound of a
    GPU computing h in fp32.  A 32-block is fragile when its absolute maximum
    lies within the bound of a power of two (the shared exponent could flip)
    or any element's scaled magnitude lies within the scaled bound of an E2M1
    rounding midpoint (its code could flip).  Returns bool [R, I/32].
    """
    R, I = h.shape
    hb = np.abs(h).reshape(R, I // 32, 32)
    db = np.asarray(delta, dtype=np.float64).reshape(R, I // 32, 32)
    amax = hb.max(axis=-1)
    dmax = db.max(axis=-1)
    e = mxfp4.e8m0_exponent(amax)
    # exponent flip: floor(log2 a) changes inside [amax - d, amax + d]
    lo = mxfp4.e8m0_exponent(np.maximum(amax - dmax, 0.0))
    hi = mxfp4.e8m0_exponent(amax + dmax)
    fragile = (lo != e) | (hi != e)
    y = np.ldexp(hb, -e[..., None])
    dy = np.ldexp(db, -e[..., None])
    mids = 0.5 * (mxfp4.E2M1_MAGNITUDE[:-1] + mxfp4.E2M1_MAGNITUDE[1:])
    near = np.zeros(y.shape, dtype=bool)
    for m in mids:
        near |= (np.abs(y - m) <= dy) & (dy > 0)
    fragile |= near.any(axis=-1)
    return fragile
