"""Seeded synthetic inputs for the skinny MUL_MAT workloads.

This module only draws random numbers and lays out shapes; it holds none of the
method's arithmetic (no quantization, no products).  The same generators feed
the CUDA path and the CPU oracle in the tests and the benchmark.

Workload recipe (7B-class decode, synthetic stand-ins for real model weights):
  * weights  ~ N(0, 0.02^2), f32 [N, K], then quantized to Q4_0 or rounded to F16;
  * activations ~ N(0, 1), f32 [M, K]; the prefill workloads additionally scale
    round(0.01 * K) distinct positions per row by 20 (outliers);
  * one numpy PCG64 generator per problem, seeded with the problem's seed, draws
    the weights first and the activations second;
  * the 32-layer stack uses seed 1000 + 7 * layer + p for matrix p of a layer.
"""
from __future__ import annotations

import numpy as np

WEIGHT_SIGMA = 0.02
OUTLIER_FRACTION = 0.01
OUTLIER_SCALE = 20.0

# Matrix shapes [N, K] of one 7B-class decoder layer, in the order p = 0..6.
LAYER_SHAPES = (
    ("attn_q", 4096, 4096),
    ("attn_k", 4096, 4096),
    ("attn_v", 4096, 4096),
    ("attn_o", 4096, 4096),
    ("ffn_gate", 11008, 4096),
    ("ffn_up", 11008, 4096),
    ("ffn_down", 4096, 11008),
)
N_LAYERS = 32

# The distinct single-matrix decode shapes [N, K].
DECODE_SHAPES = ((4096, 4096), (11008, 4096), (4096, 11008))


def stack_seed(layer: int, p: int) -> int:
    return 1000 + 7 * layer + p


def _outliers(gen: np.random.Generator, x: np.ndarray) -> None:
    M, K = x.shape
    n_out = int(round(OUTLIER_FRACTION * K))
    for m in range(M):
        idx = gen.choice(K, size=n_out, replace=False)
        x[m, idx] *= np.float32(OUTLIER_SCALE)


def problem(seed: int, M: int, N: int, K: int, outliers: bool = False):
    """(weights f32 [N, K], activations f32 [M, K]) for one seeded problem."""
    gen = np.random.default_rng(seed)
    w = gen.standard_normal((N, K), dtype=np.float32) * np.float32(WEIGHT_SIGMA)
    x = gen.standard_normal((M, K), dtype=np.float32)
    if outliers:
        _outliers(gen, x)
    return w, x


def weights(seed: int, N: int, K: int) -> np.ndarray:
    gen = np.random.default_rng(seed)
    return gen.standard_normal((N, K), dtype=np.float32) * np.float32(WEIGHT_SIGMA)


def activations(seed: int, M: int, K: int, outliers: bool = False) -> np.ndarray:
    gen = np.random.default_rng(seed)
    x = gen.standard_normal((M, K), dtype=np.float32)
    if outliers:
        _outliers(gen, x)
    return x


def f16_bits(w: np.ndarray) -> np.ndarray:
    """Round f32 weights to IEEE binary16 (numpy, nearest-even) and return the bit patterns."""
    return np.ascontiguousarray(w, dtype=np.float32).astype(np.float16).view(np.uint16)


def edge_weights(seed: int, N: int, K: int) -> np.ndarray:
    """Weights that exercise the quantizer's corner cases, block by block.

    Blocks cycle through: all zero; tiny magnitudes (subnormal fp16 scales);
    a positive signed maximum (the clamp case, d < 0); a tie in magnitude with
    opposite signs; exact half-way codes; large magnitudes; plain Gaussian.
    """
    gen = np.random.default_rng(seed)
    w = gen.standard_normal((N, K), dtype=np.float32) * np.float32(WEIGHT_SIGMA)
    nb = K // 32
    blocks = w.reshape(N, nb, 32)
    for n in range(N):
        for b in range(nb):
            kind = (n * nb + b) % 7
            blk = blocks[n, b]
            if kind == 0:
                blk[:] = 0.0
            elif kind == 1:
                blk *= np.float32(1e-4)
            elif kind == 2:
                j = gen.integers(32)
                blk[j] = np.abs(blk).max() * np.float32(1.5)
            elif kind == 3:
                j0, j1 = gen.choice(32, size=2, replace=False)
                a = np.abs(blk).max() * np.float32(1.25)
                blk[j0], blk[j1] = a, -a
            elif kind == 4:
                # codes (q - 8) * d with d a power of two, plus half-way points
                c = gen.integers(-8, 8, size=32).astype(np.float32)
                c[gen.integers(32)] = -8.0
                half = gen.random(32) < 0.3
                c[half & (c > -8) & (c < 7)] += np.float32(0.5)
                blk[:] = c * np.float32(2.0 ** -6)
            elif kind == 5:
                blk *= np.float32(1e3)
    return w


def edge_activations(seed: int, M: int, K: int) -> np.ndarray:
    """Activations with zero blocks, exact ties of the Q8_0 codes and wide ranges."""
    gen = np.random.default_rng(seed)
    x = gen.standard_normal((M, K), dtype=np.float32)
    nb = K // 32
    blocks = x.reshape(M, nb, 32)
    for m in range(M):
        for b in range(nb):
            kind = (m * nb + b) % 5
            blk = blocks[m, b]
            if kind == 0:
                blk[:] = 0.0
            elif kind == 1:
                # amax = 127 so d = 1 and the codes land on .5 ties
                c = gen.integers(-126, 126, size=32).astype(np.float32) + np.float32(0.5)
                c[gen.integers(32)] = 127.0
                blk[:] = c
            elif kind == 2:
                blk *= np.float32(1e-3)
            elif kind == 3:
                blk *= np.float32(50.0)
    return x


# ---------------------------------------------------------------------------
# INT8 KV-cache decode attention (xFasterTransformer, "2.2 Effective KV cache
# Optimization": Llama2-7B with 32 heads of 128, batch 256, 1024 input and 1024
# output tokens).  Keys and values ~ N(0, 1), keys with a per-channel spread
# exp(0.5 N(0, 1)) drawn once per head (a few wide channels, as keys have);
# queries ~ N(0, 1).  Lengths: "full" = Tcap for every sequence; "mix" = uniform
# in [1, Tcap]; the tests add their own edge lengths.
# ---------------------------------------------------------------------------
KV_LLAMA2_7B = {"B": 256, "Hq": 32, "Hkv": 32, "Tcap": 2048, "D": 128}


def kv_lengths(seed: int, B: int, Tcap: int, mode: str = "full") -> np.ndarray:
    if mode == "full":
        return np.full(B, Tcap, np.int32)
    gen = np.random.default_rng(seed)
    return gen.integers(1, Tcap + 1, size=B).astype(np.int32)


def kv_problem(seed: int, B: int, Hq: int, Hkv: int, Tcap: int, D: int):
    """(q f32 [B, Hq, D], k f32 [B, Hkv, Tcap, D], v f32 [B, Hkv, Tcap, D])."""
    gen = np.random.default_rng(seed)
    chan = np.exp(np.float32(0.5) * gen.standard_normal((1, Hkv, 1, D), dtype=np.float32))
    k = gen.standard_normal((B, Hkv, Tcap, D), dtype=np.float32) * chan
    v = gen.standard_normal((B, Hkv, Tcap, D), dtype=np.float32)
    q = gen.standard_normal((B, Hq, D), dtype=np.float32)
    return q, k, v


def kv_codes_device(seed: int, B: int, Hkv: int, Tcap: int, D: int, device):
    """Random INT8 cache contents drawn on the device (for sizes the host should not
    generate): codes uniform in [-127, 127] and scales exp(0.3 N(0, 1)) / 42, for K and V.
    Returns (k, k_scale, v, v_scale) torch tensors."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    shape = (B, Hkv, Tcap, D)
    k = torch.randint(-127, 128, shape, generator=g, device=device, dtype=torch.int8)
    v = torch.randint(-127, 128, shape, generator=g, device=device, dtype=torch.int8)
    ks = torch.exp(0.3 * torch.randn(shape[:3], generator=g, device=device)) / 42.0
    vs = torch.exp(0.3 * torch.randn(shape[:3], generator=g, device=device)) / 42.0
    return k, ks.float().contiguous(), v, vs.float().contiguous()
