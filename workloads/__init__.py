"""Seeded synthetic inputs for the A4W4 GEMM workloads.

Shared by the tests, ``bench.py`` and ``__graft_entry__.smoke()``, on both
sides of the parity check (oracle and CUDA library).  This module holds none
of the method's arithmetic: it draws random numbers (numpy PCG64) and stores
them as BF16 with torch's float32 -> bfloat16 conversion (round to nearest
even), nothing else.

The workloads follow the shapes and value mixes of the dense A4W4 and grouped
MoE GEMM1 measurements on "[gfx950][FlyDSL] Add direct dense A4W4 MXFP4 GEMM"
(Kernel microbenchmark: N x K in {8448x7168, 7168x4224, 1536x7168, 7168x768},
M from 1 to 2048) and "[gfx1250] Fuse A4W4 stage1 FP4 quantization"
(Performance: E=896, topk=16, model_dim=3584, inter_dim=768, tokens 1..4096).
No public dataset is involved; all values are synthetic.
"""

import numpy as np
import torch

# Dense shapes (M, N, K) per workload family.
SMALL = [(16, 256, 256)]
DECODE_SWEEP = [(M, N, K) for (N, K) in ((7168, 4224), (1536, 7168), (7168, 768)) for M in (1, 8, 32)]
LARGE_M_SWEEP = [(M, N, K) for (N, K) in ((8448, 7168), (7168, 4224)) for M in (128, 512, 2048)]
TAIL_STRESS = [(M, 1536, 4224) for M in (37, 513, 2047)]
MOE = dict(tokens=(1, 16, 256, 4096), experts=896, topk=16, model_dim=3584, inter_dim=768)

W_STD = 0.02
OUTLIER_FRACTION = 0.01
OUTLIER_GAIN = 20.0

_TAG_A, _TAG_W, _TAG_X, _TAG_W1, _TAG_STRESS, _TAG_W2, _TAG_GATE, _TAG_H, _TAG_WIDE = 11, 12, 13, 14, 15, 16, 17, 18, 19


def rng(*key):
    """Independent PCG64 stream for an integer key tuple."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def to_bf16_bits(x):
    """float32 array -> BF16 bit patterns (uint16), torch's RNE conversion."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_torch(bits):
    """uint16 BF16 bit patterns -> torch.bfloat16 tensor (CPU, same storage)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def normal_bits(shape, std, *key):
    return to_bf16_bits(rng(*key).standard_normal(shape, dtype=np.float32) * np.float32(std))


def weight_bits(N, K, seed=0):
    """W [N, K] ~ N(0, 0.02) as BF16."""
    return normal_bits((N, K), W_STD, seed, _TAG_W, N, K)


def activation_bits(M, K, seed=0):
    """A [M, K] ~ N(0, 1) as BF16."""
    return normal_bits((M, K), 1.0, seed, _TAG_A, M, K)


def outlier_channels(K, seed=1):
    """floor(1% of K) K-channels, uniform without replacement."""
    n = int(np.floor(OUTLIER_FRACTION * K))
    return np.sort(rng(seed, K).choice(K, size=n, replace=False))


def decode_activation_bits(M, K, seed=0, outlier_seed=1):
    """A [M, K] ~ N(0, 1) with the same 1% of K-channels scaled by 20 in every row."""
    a = rng(seed, _TAG_A, M, K).standard_normal((M, K), dtype=np.float32)
    a[:, outlier_channels(K, outlier_seed)] *= np.float32(OUTLIER_GAIN)
    return to_bf16_bits(a)


_TIES = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
_SATURATING = np.array([6.5, 7.0, 7.5, 7.9375], dtype=np.float32)


def stress_activation_bits(M, K, seed=3):
    """Scale-edge stress rows: every 32-block of A is drawn independently as

    * 10% all zero;
    * 40% N(0,1) * 2**u, u a uniform integer in [-100, 100];
    * 25% exact-tie blocks: elements 2**u * (+-{0.25,0.75,1.25,1.75,2.5,3.5,5}),
      one element +-4 * 2**u so that the block maximum is in [4, 8) * 2**u;
    * 25% saturating blocks: 2**u * N(0,1) with about a quarter of the
      elements (at least one) replaced by 2**u * (+-{6.5, 7, 7.5, 7.9375}).

    Every value is exactly representable in BF16.
    """
    g = rng(seed, _TAG_STRESS, M, K)
    nb = K // 32
    kind = g.choice(4, size=(M, nb), p=[0.10, 0.40, 0.25, 0.25])
    u = g.integers(-100, 101, size=(M, nb)).astype(np.float64)
    scale = np.ldexp(1.0, u.astype(np.int64))[..., None]
    normal = g.standard_normal((M, nb, 32))
    signs = np.where(g.random((M, nb, 32)) < 0.5, -1.0, 1.0)
    ties = _TIES[g.integers(0, len(_TIES), size=(M, nb, 32))] * signs
    pos = g.integers(0, 32, size=(M, nb))
    np.put_along_axis(ties, pos[..., None], 4.0 * signs[..., :1], axis=-1)
    sat_pick = g.random((M, nb, 32)) < 0.25
    np.put_along_axis(sat_pick, pos[..., None], True, axis=-1)
    sat = np.where(sat_pick, _SATURATING[g.integers(0, len(_SATURATING), size=(M, nb, 32))] * signs, normal)
    blocks = np.select([kind[..., None] == 0, kind[..., None] == 1, kind[..., None] == 2],
                       [np.zeros_like(normal), normal, ties], default=sat) * scale
    # float64 -> float32 is exact here for the tie/saturating values; the
    # N(0,1)*2**u values are rounded by the BF16 conversion like any input.
    return to_bf16_bits(blocks.reshape(M, K).astype(np.float32))


def dense_problem(M, N, K, family, seed=0):
    """(A_bits [M, K], W_bits [N, K]) for one dense GEMM of a workload family."""
    if family == "decode":
        A = decode_activation_bits(M, K, seed)
    elif family == "stress":
        A = stress_activation_bits(M, K)
    else:
        A = activation_bits(M, K, seed)
    return A, weight_bits(N, K, seed)


# K-block exponents of wide_scale_problem: both ends of the E8M0 range the
# BF16-decoding paths cover, and points between.
WIDE_EXPONENTS = (-126, -125, -124, -64, 0, 64, 124, 125)


def wide_scale_problem(M, N, K, seed=6):
    """(A_bits [M, K], W_bits [N, K]) whose 32-blocks of K span the weight
    scale range: K-block b has weights +-U(0.5, 3) * 2**x and activations
    +-U(0.5, 1.5) * 2**-x with x = WIDE_EXPONENTS[b % 8], so every product is
    of order 1 while the weight blocks' E8M0 scales run from 2^-127 to about
    2^124.  Activations stay BF16 normal numbers; the smallest weights are
    BF16 subnormals."""
    g = rng(seed, _TAG_WIDE, M, N, K)
    nb = K // 32
    x = np.array(WIDE_EXPONENTS, dtype=np.int64)[np.arange(nb) % len(WIDE_EXPONENTS)]
    x = np.repeat(x, 32)
    ws = np.where(g.random((N, K)) < 0.5, -1.0, 1.0)
    as_ = np.where(g.random((M, K)) < 0.5, -1.0, 1.0)
    w = ws * g.uniform(0.5, 3.0, (N, K)) * np.ldexp(1.0, x)[None, :]
    a = as_ * g.uniform(0.5, 1.5, (M, K)) * np.ldexp(1.0, -x)[None, :]
    return to_bf16_bits(a.astype(np.float32)), to_bf16_bits(w.astype(np.float32))


def moe_topk_ids(T, E, topk, seed=2):
    """topk distinct experts per token, uniform without replacement: int32 [T, topk]."""
    keys = rng(seed, T, E, topk).random((T, E))
    return np.argsort(keys, axis=1, kind="stable")[:, :topk].astype(np.int32)


def moe_tokens_bits(T, D, seed=0):
    """X [T, D] ~ N(0, 1) as BF16."""
    return normal_bits((T, D), 1.0, seed, _TAG_X, T, D)


def moe_expert_weight_bits(e, two_I, D, seed=0):
    """W1[e] [2I, D] ~ N(0, 0.02) as BF16; each expert has its own stream."""
    return normal_bits((two_I, D), W_STD, seed, _TAG_W1, e, two_I, D)


def moe_expert_w2_bits(e, D, I, seed=0):
    """W2[e] [D, I] (down projection) ~ N(0, 0.02) as BF16; one stream per expert."""
    return normal_bits((D, I), W_STD, seed, _TAG_W2, e, D, I)


def moe_topk_weights(T, topk, seed=4):
    """Routing weights float32 [T, topk]: a softmax over each token's topk
    N(0, 1) logits (positive, each row sums to about 1)."""
    z = rng(seed, _TAG_GATE, T, topk).standard_normal((T, topk))
    p = np.exp(z - z.max(axis=1, keepdims=True))
    return (p / p.sum(axis=1, keepdims=True)).astype(np.float32)


def moe_hidden_bits(R, I, seed=5):
    """Stand-in GEMM1 activations [R, I] as BF16: products of two N(0, 1)
    draws (the shape of silu(gate) * up), for feeding GEMM2 on its own."""
    g = rng(seed, _TAG_H, R, I)
    return to_bf16_bits((g.standard_normal((R, I)) * g.standard_normal((R, I))).astype(np.float32))
