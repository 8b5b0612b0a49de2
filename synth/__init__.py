"""Seeded synthetic inputs shared by the tests and the benchmark.

This module holds none of the layer's arithmetic. It produces:
  * expert blobs in the canonical block layout (per block: an fp16 scale as two
    little-endian bytes, then 16 bytes of codes). The codes are uniform random
    bytes, so every code value is uniform whatever the bit order; the scales are
    d ~ U[d_lo, d_hi] drawn in fp64 and rounded to nearest-even binary16;
  * activations and router weights ~ N(0, sigma^2) (Box-Muller in fp64, rounded to
    fp32, then to bf16 when asked);
  * a Zipf(s) per-expert router bias b_e = -s * ln(r_e), r a seeded permutation of
    1..E, so that expert popularity falls off as a power law.

All randomness comes from one counter-based generator, SplitMix64 (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014): output i of
the stream with seed s is mix64(s + (i + 1) * 0x9E3779B97F4A7C15) mod 2^64, with
the mix64 finaliser of that paper's reference code. ``synth_dev.cu`` is the CUDA
twin that fills the large expert arenas on the device; the test suite checks that
both produce the same bytes.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)
BLOCK_BYTES = 18
BLOCK_WEIGHTS = {0: 32, 1: 64}  # format kind -> weights per block (Q4, Q2_0)


def mix64(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * M1
        z = (z ^ (z >> np.uint64(27))) * M2
    return z ^ (z >> np.uint64(31))


def sm64(seed: int, idx) -> np.ndarray:
    """Output number idx (array) of the SplitMix64 stream seeded with seed."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(seed) + (idx + np.uint64(1)) * GOLDEN)


def sub_seed(seed: int, tag: int) -> int:
    """Seed of an independent stream for tensor `tag` under base seed `seed`."""
    return int(sm64(seed, np.array([tag], dtype=np.uint64))[0])


def uniform01(seed: int, n: int, offset: int = 0) -> np.ndarray:
    r = sm64(seed, np.arange(offset, offset + n, dtype=np.uint64))
    return (r >> np.uint64(11)).astype(np.float64) * 2.0 ** -53


def normal(seed: int, n: int, std: float = 1.0) -> np.ndarray:
    """n draws of N(0, std^2) in fp64 (cosine branch of Box-Muller, two words per draw)."""
    r = sm64(seed, np.arange(0, 2 * n, dtype=np.uint64))
    u1 = ((r[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53  # (0, 1]
    u2 = (r[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53  # [0, 1)
    return std * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the 16-bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    nan = (b & 0x7FFFFFFF) > 0x7F800000
    r = ((b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16))
    r = np.where(nan, (b >> np.uint32(16)) | np.uint32(0x40), r)
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_round(a: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 -> bf16 -> fp64, the values a bf16 tensor of `a` holds."""
    return bf16_bits_to_f64(f32_to_bf16_bits(np.asarray(a, dtype=np.float64).astype(np.float32)))


def expert_blobs(seed: int, tags, n_blocks: int, d_lo: float, d_hi: float) -> np.ndarray:
    """Canonical blobs [len(tags)][n_blocks*18] for experts with stream tags `tags`.

    Block b of the expert with tag g uses words 3b, 3b+1 (codes, little-endian) and
    3b+2 (scale) of the stream sub_seed(seed, g).
    """
    tags = list(tags)
    out = np.empty((len(tags), n_blocks * BLOCK_BYTES), dtype=np.uint8)
    b = np.arange(n_blocks, dtype=np.uint64)
    for i, g in enumerate(tags):
        s = sub_seed(seed, g)
        w0 = sm64(s, 3 * b)
        w1 = sm64(s, 3 * b + np.uint64(1))
        u = (sm64(s, 3 * b + np.uint64(2)) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        d = (d_lo + (d_hi - d_lo) * u).astype(np.float16)
        blk = out[i].reshape(n_blocks, BLOCK_BYTES)
        blk[:, 0:2] = d.view(np.uint16).astype("<u2").view(np.uint8).reshape(n_blocks, 2)
        blk[:, 2:10] = w0.astype("<u8").view(np.uint8).reshape(n_blocks, 8)
        blk[:, 10:18] = w1.astype("<u8").view(np.uint8).reshape(n_blocks, 8)
    return out


def permutation(seed: int, n: int) -> np.ndarray:
    """A seeded permutation of 0..n-1 (stable argsort of n random words)."""
    return np.argsort(sm64(seed, np.arange(n, dtype=np.uint64)), kind="stable")


def zipf_bias(seed: int, E: int, s: float) -> np.ndarray:
    """b_e = -s * ln(r_e) with r a seeded permutation of the ranks 1..E (fp32)."""
    rank = np.empty(E, dtype=np.float64)
    rank[permutation(seed, E)] = np.arange(1, E + 1, dtype=np.float64)
    return (-s * np.log(rank)).astype(np.float32)
