"""Seeded synthetic inputs for the W12 decode-GEMM workloads.

This module only draws random numbers and rounds them to BF16 (torch's
round-to-nearest-even); it holds none of the W12 arithmetic, so both the
product path and the test oracle may use it.

Workloads (the weight shapes are those of a dense 27B-class decoder layer,
hidden size 5120; there are no real checkpoints here, so every tensor is
synthetic):

  single    1024 x 1024, weights ~N(0, 0.02), x[1, 1024] ~N(0, 1), one
            PCG64 stream seeded with 0 (W drawn first, then x)
  layer     q 6144x5120, k/v 1024x5120, o 5120x6144, gate/up 17408x5120,
            down 5120x17408; weights ~N(0, 0.02), activations ~N(0, 1)
  heavy     the layer shapes with Student-t(3) * 0.02 weights and 0.5 % of
            entries (Bernoulli) multiplied by 100 before rounding
  lmhead    the LM head, 151936 x 5120, weights ~N(0, 0.02)
  model64   64 layers of the layer shapes, weights ~N(0, 0.02) drawn on the
            GPU (21.8 G weights: 43.6 GB BF16, 32.7 GB W12), one activation
            per shape shared by all layers

Seeds: weights use numpy PCG64 seeded with 100 * workload_id + matrix_index
(q0 k1 v2 o3 gate4 up5 down6); activations use 10000 + 100 * workload_id + M.
model64 weights use torch's CUDA generator seeded with
50000 + 7 * layer + matrix_index, its activations PCG64 seeded with
(10000 + 100 * 5 + M, K): one x per K, shared by the matrices of that K.
"""
from __future__ import annotations

import numpy as np
import torch

WEIGHT_STD = 0.02

# (name, N = out_features, K = in_features); y = x . W^T
LAYER_SHAPES = (
    ("q", 6144, 5120),
    ("k", 1024, 5120),
    ("v", 1024, 5120),
    ("o", 5120, 6144),
    ("gate", 17408, 5120),
    ("up", 17408, 5120),
    ("down", 5120, 17408),
)

# LM head of the same model: hidden 5120 and a ~152K-token vocabulary (the
# pages give no vocabulary size; this one is assumed)
LMHEAD_SHAPE = ("lm_head", 151936, 5120)

WORKLOAD_IDS = {"single": 1, "layer": 2, "layer_sweep": 3, "heavy": 4, "model64": 5, "lmhead": 6}
SWEEP_M = (2, 4, 8, 16, 32)
HEAVY_M = (1, 16)
MODEL64_M = (16, 32)
MODEL64_LAYERS = 64


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest even) and return the bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 values (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def gaussian_weights(n: int, k: int, seed: int, std: float = WEIGHT_STD) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return to_bf16_bits(rng.standard_normal((n, k), dtype=np.float32) * np.float32(std))


def heavy_tail_weights(n: int, k: int, seed: int, outlier_p: float = 0.005,
                       outlier_scale: float = 100.0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    w = rng.standard_t(3.0, size=(n, k)).astype(np.float32) * np.float32(WEIGHT_STD)
    out = rng.random((n, k), dtype=np.float32) < outlier_p
    w[out] *= np.float32(outlier_scale)
    return to_bf16_bits(w)


def activations(m: int, k: int, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return to_bf16_bits(rng.standard_normal((m, k), dtype=np.float32))


def forced_escape_weights(n: int, k: int, frac: float, seed: int) -> np.ndarray:
    """Gaussian weights where a fraction `frac` of entries get an exponent drawn
    uniformly from 0..255 (sign and mantissa kept), so that many fall outside
    any 15-entry table."""
    w = gaussian_weights(n, k, seed)
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    pick = rng.random((n, k)) < frac
    expo = rng.integers(0, 256, size=(n, k), dtype=np.uint16)
    forced = (w & np.uint16(0x807F)) | (expo << np.uint16(7))
    return np.where(pick, forced, w).astype(np.uint16)


def all_bf16_patterns(shuffle_seed: int | None = None) -> np.ndarray:
    """All 65536 BF16 bit patterns as a 256 x 256 matrix (optionally shuffled)."""
    v = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    if shuffle_seed is not None:
        v = np.random.Generator(np.random.PCG64(shuffle_seed)).permutation(v)
    return v.reshape(256, 256)


def table_rule_weights(seed: int) -> np.ndarray:
    """2048 x 4096 BF16 patterns: the 128 x 256 block at (tile t, segment s)
    draws its exponents from t distinct values below 128 and s distinct values
    from 128 up, so the blocks cover every split of the table between the two
    halves, more than 15 distinct exponents, and (every other block) exactly
    equal counts, where the ranking falls to the smaller exponent.  Signs and
    mantissas are uniform."""
    rng = np.random.Generator(np.random.PCG64(seed))
    w = np.empty((2048, 4096), dtype=np.uint16)
    cells = 128 * 256
    for t in range(16):
        for s in range(16):
            low = rng.choice(np.arange(0, 128), size=t, replace=False)
            high = rng.choice(np.arange(128, 256), size=s, replace=False)
            exps = np.concatenate([low, high]).astype(np.uint16)
            if exps.size == 0:
                exps = np.array([0], dtype=np.uint16)
            if (t + s) % 2 == 0:
                counts = np.full(exps.size, cells // exps.size)
                counts[: cells % exps.size] += 1
            else:
                counts = rng.multinomial(cells, rng.dirichlet(np.ones(exps.size)))
            e = rng.permutation(np.repeat(exps, counts)).reshape(128, 256)
            sm = rng.integers(0, 1 << 16, size=(128, 256), dtype=np.uint32).astype(np.uint16) & np.uint16(0x807F)
            w[128 * t:128 * (t + 1), 256 * s:256 * (s + 1)] = sm | (e << np.uint16(7))
    return w


def weight_seed(workload: str, index: int) -> int:
    wid = WORKLOAD_IDS[workload]
    if workload == "layer_sweep":
        wid = WORKLOAD_IDS["layer"]
    return 100 * wid + index


def activation_seed(workload: str, m: int) -> int:
    return 10000 + 100 * WORKLOAD_IDS[workload] + m


def layer_weights(workload: str = "layer"):
    """Yield (name, W bits[N, K]) for the seven layer matrices of a workload."""
    gen = heavy_tail_weights if workload == "heavy" else gaussian_weights
    for idx, (name, n, k) in enumerate(LAYER_SHAPES):
        yield name, gen(n, k, weight_seed(workload, idx))


def model64_weight_dev(layer: int, index: int) -> torch.Tensor:
    """Weight `index` (q0 .. down6) of layer `layer` of the 64-layer stream,
    drawn on the current CUDA device as BF16 [N, K]."""
    _, n, k = LAYER_SHAPES[index]
    g = torch.Generator(device="cuda")
    g.manual_seed(50000 + 7 * layer + index)
    w = torch.randn((n, k), generator=g, device="cuda", dtype=torch.float32)
    return (w * WEIGHT_STD).to(torch.bfloat16)


def model64_activation(m: int, index: int) -> np.ndarray:
    """The x [m, K] fed to matrix `index` of every layer of the 64-layer
    stream: one activation per K (N(0, 1), PCG64 seeded with
    (activation_seed, K)), so q, k, v, gate and up (K = 5120) share it as in a
    decoder layer, and o and down get their own."""
    k = LAYER_SHAPES[index][2]
    rng = np.random.Generator(np.random.PCG64([activation_seed("model64", m), k]))
    return to_bf16_bits(rng.standard_normal((m, k), dtype=np.float32))


def single_case():
    """The 1024 x 1024 single-layer case: (W bits, x bits[1, 1024]); one PCG64
    stream seeded with 0 draws W first, then x."""
    rng = np.random.Generator(np.random.PCG64(0))
    w = rng.standard_normal((1024, 1024), dtype=np.float32) * np.float32(WEIGHT_STD)
    x = rng.standard_normal((1, 1024), dtype=np.float32)
    return to_bf16_bits(w), to_bf16_bits(x)
