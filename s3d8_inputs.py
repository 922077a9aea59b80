"""Seeded synthetic inputs for the S3D8 W2.7A8 linear layer.

This module is shared by the CUDA-path tests, the benchmark and the oracle
tests.  It holds input recipes only (random draws, the bf16 storage
conversion and the workload shapes) and none of the layer's arithmetic:
decoding, activation quantisation and the matrix product live in the CUDA
library and, independently, in the oracle.

Recipe (one independent numpy ``Generator`` per tensor, spawned in the fixed
order centroids, packed bytes, channel scales, activations):
  * centroid table C: int8 uniform in [1, 127], shape 32 x 3, one per matrix;
  * packed bytes: uniform over 0..255, shape [ceil(N/3), K].  The byte layout
    is a bijection onto (Q, S0, S1, S2), so this is Q uniform on 0..31 with
    three independent fair signs;
  * channel scales: bf16(|N(0, 0.02)| / 127), shape [N];
  * activations: bf16(N(0, 1)), shape [M, K]; with ``outliers`` 1 % of the
    elements (uniform positions) are multiplied by 20.

The shapes are those of the Llama-3.2-11B text decoder that the pages
benchmark ("11 billion parameters on a phone", section "Fast? How fast?",
and the runtime table of the Llama-Mobile paper, section 4.3).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# (name, K, N) for one text decoder layer: Y[M, N] = X[M, K] W[N, K]^T.
LLAMA_11B_LAYER = (
    ("q", 4096, 4096),
    ("k", 4096, 1024),
    ("v", 4096, 1024),
    ("o", 4096, 4096),
    ("gate", 4096, 14336),
    ("up", 4096, 14336),
    ("down", 14336, 4096),
)
LLAMA_11B_HEAD = ("head", 4096, 128256)
LLAMA_11B_LAYERS = 40

# The activation each projection reads in a decoder layer: q/k/v share the
# attention input, gate/up share the MLP input, o and down read their own.
LLAMA_11B_INPUT_OF = {"q": "attn", "k": "attn", "v": "attn", "o": "o", "gate": "mlp",
                      "up": "mlp", "down": "down"}


def groups(N: int) -> int:
    """Packed rows for N output channels (3 channels per byte)."""
    return (N + 2) // 3


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bfloat16 (ties to even); uint16 bit patterns.

    Inputs here are finite; this is the storage conversion of the recipe.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class Matrix:
    """One S3D8 weight matrix with its seeded fields."""
    name: str
    K: int
    N: int
    C: np.ndarray          # int8 [32, 3]
    packed: np.ndarray     # uint8 [ceil(N/3), K]
    chan_scale: np.ndarray  # uint16 (bf16 bits) [N]


def _streams(seed, key):
    ss = np.random.SeedSequence([int(seed)] + [int(v) for v in key])
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(4)]


def centroids(rng: np.random.Generator) -> np.ndarray:
    return rng.integers(1, 128, size=(32, 3), dtype=np.int16).astype(np.int8)


def packed_bytes(rng: np.random.Generator, G: int, K: int) -> np.ndarray:
    return rng.integers(0, 256, size=(G, K), dtype=np.uint8)


def chan_scale(rng: np.random.Generator, N: int) -> np.ndarray:
    s = np.abs(rng.normal(0.0, 0.02, size=N)).astype(np.float32) / np.float32(127.0)
    return f32_to_bf16_bits(s)


def activations(rng: np.random.Generator, M: int, K: int, outliers: bool = False) -> np.ndarray:
    x = rng.standard_normal(size=(M, K), dtype=np.float32)
    if outliers:
        n_out = max(1, (M * K) // 100)
        pos = rng.choice(M * K, size=n_out, replace=False)
        x.reshape(-1)[pos] *= np.float32(20.0)
    return f32_to_bf16_bits(x)


def matrix(name: str, K: int, N: int, seed: int = 0, index: int = 0) -> Matrix:
    """Seeded S3D8 matrix fields; ``index`` separates matrices of one workload."""
    r_c, r_p, r_s, _ = _streams(seed, (1, index))
    return Matrix(name, K, N, centroids(r_c), packed_bytes(r_p, groups(N), K), chan_scale(r_s, N))


def acts(M: int, K: int, seed: int = 0, index: int = 0, outliers: bool = False) -> np.ndarray:
    """Seeded bf16 activation bits [M, K]."""
    _, _, _, r_x = _streams(seed, (2, index))
    return activations(r_x, M, K, outliers)


def tiny_case(seed: int = 0):
    """Tiny S3D8 linear: K=256, N=96, M=4 (matrix, activations)."""
    m = matrix("tiny", 256, 96, seed)
    return m, acts(4, 256, seed)


def layer_matrices(layer: int = 0, seed: int = 0):
    """The seven projections of one decoder layer, each with its own table."""
    return [matrix(n, K, N, seed, index=layer * 8 + i) for i, (n, K, N) in enumerate(LLAMA_11B_LAYER)]


def head_matrix(seed: int = 0) -> Matrix:
    n, K, N = LLAMA_11B_HEAD
    return matrix(n, K, N, seed, index=LLAMA_11B_LAYERS * 8)


# Batched-decode and prefill sweeps use these two projection shapes (K, N).
SWEEP_SHAPES = (("gate_up", 4096, 14336), ("down", 14336, 4096))
DECODE_SWEEP_M = (8, 16, 32, 64)
PREFILL_M = (512, 2048)
