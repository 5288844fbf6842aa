"""Seeded synthetic inputs for the hyper-connection mix-statistics path.

This module only draws random numbers and encodes them as bf16 / fp32 host
arrays. It holds none of the method's arithmetic and is shared by the CPU
oracle's tests, the CUDA parity tests and the benchmark, so both sides see
identical inputs.

Generator (portable, counter based, identical on x86 and Arm):
  * splitmix64: value i of stream `seed` is mix64(seed + (i + 1) * 0x9E3779B97F4A7C15),
    with mix64 the published splitmix64 finaliser (Steele, Lea, Flood 2014).
  * uniform double in [0, 1): top 53 bits of a draw times 2**-53.
  * standard normal: Box-Muller on consecutive draw pairs (u1, u2):
    r = sqrt(-2 ln(1 - u1)); z_even = r cos(2 pi u2), z_odd = r sin(2 pi u2).
  * bf16: round-to-nearest-even of the double, applied once (no detour via fp32).
  * fp32: IEEE round-to-nearest of the double.

Workloads (the hc_fused page's shapes; the page measures on the DSV4.1 forward,
which these synthetic tensors stand in for):
  * x[M, K] bf16 ~ N(0, 1), stream seed 0, row-major element index m*K + k, so a
    smaller M is always a prefix of a larger one;
  * W[24, K] fp32 ~ N(0, 1) * K**-0.5 (std K**-1/2), seed 1;
  * hc_scale[3] fp32 ~ U(0.5, 1.5), seed 2;
  * hc_base[24] fp32 ~ N(0, 1) * 0.1, seed 3;
  * outlier channels: round(0.01 K) distinct columns chosen by a partial
    Fisher-Yates shuffle driven by seed 4; x there is the same normal draw times
    20, rounded once to bf16;
  * layer stack: call i uses seeds 1000+3i, 1001+3i, 1002+3i for W, hc_scale, hc_base.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

K_DEFAULT = 20480
MIX = 24
HC = 4

SEED_X, SEED_W, SEED_SCALE, SEED_BASE, SEED_OUTLIER = 0, 1, 2, 3, 4


def splitmix64(seed: int, start: int, n: int) -> np.ndarray:
    """Draws start .. start+n-1 of splitmix64 stream `seed` (uint64)."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(seed) + i * GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniform(seed: int, start: int, n: int) -> np.ndarray:
    """Doubles in [0, 1) from draws start .. start+n-1."""
    return (splitmix64(seed, start, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, start: int, n: int) -> np.ndarray:
    """Standard normals start .. start+n-1 of stream `seed` (Box-Muller on draw pairs).

    Normal i uses draws 2*(i//2) and 2*(i//2)+1, so any window of the stream is
    reproducible on its own.
    """
    if n <= 0:
        return np.zeros(0, np.float64)
    p0 = start // 2
    p1 = (start + n + 1) // 2
    u = uniform(seed, 2 * p0, 2 * (p1 - p0)).reshape(-1, 2)
    r = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
    t = 2.0 * math.pi * u[:, 1]
    z = np.empty((p1 - p0, 2), np.float64)
    z[:, 0] = r * np.cos(t)
    z[:, 1] = r * np.sin(t)
    z = z.reshape(-1)
    off = start - 2 * p0
    return z[off:off + n]


def bf16_bits_from_f64(a: np.ndarray) -> np.ndarray:
    """Round doubles once to bf16 (nearest, ties to even); returns uint16 bit patterns.

    Valid for finite values in the bf16 normal range (all inputs drawn here).
    """
    u = np.ascontiguousarray(a, dtype=np.float64).view(np.uint64)
    keep_shift = np.uint64(52 - 7)
    lsb = (u >> keep_shift) & np.uint64(1)
    bias = (np.uint64(1) << np.uint64(44)) - np.uint64(1) + lsb
    with np.errstate(over="ignore"):
        r = (u + bias) & ~((np.uint64(1) << keep_shift) - np.uint64(1))
    f32 = r.view(np.float64).astype(np.float32)  # exact: r has an 8-bit significand
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def outlier_channels(K: int, seed: int = SEED_OUTLIER, frac: float = 0.01) -> np.ndarray:
    """round(frac*K) distinct channel indices by a partial Fisher-Yates shuffle."""
    n = int(round(frac * K))
    perm = np.arange(K, dtype=np.int64)
    draws = splitmix64(seed, 0, n)
    for i in range(n):
        j = i + int(draws[i] % np.uint64(K - i))
        perm[i], perm[j] = perm[j], perm[i]
    return np.sort(perm[:n])


def make_x(M: int, K: int = K_DEFAULT, seed: int = SEED_X, outliers: bool = False,
           row_block: int = 64, threads: int | None = None, out: np.ndarray | None = None,
           row0: int = 0) -> np.ndarray:
    """Rows row0 .. row0+M-1 of x[., K] as uint16 bf16 bit patterns.

    Row-major and prefix-stable in M.  Row blocks are drawn on a thread pool;
    every element depends only on its index, so the result does not depend on
    the block size or thread count.
    """
    if out is None:
        out = np.empty((M, K), np.uint16)
    ch = outlier_channels(K) if outliers else None

    def block(r0):
        r1 = min(M, r0 + row_block)
        z = normal(seed, (row0 + r0) * K, (r1 - r0) * K).reshape(r1 - r0, K)
        if ch is not None:
            z[:, ch] *= 20.0
        out[r0:r1] = bf16_bits_from_f64(z).reshape(r1 - r0, K)

    starts = list(range(0, M, row_block))
    n = threads if threads is not None else min(len(starts), os.cpu_count() or 1, 16)
    if n <= 1:
        for r0 in starts:
            block(r0)
    else:
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(block, starts))
    return out


def make_w(K: int = K_DEFAULT, seed: int = SEED_W, mix: int = MIX) -> np.ndarray:
    """W[mix, K] fp32 with std K**-1/2."""
    return (normal(seed, 0, mix * K) * (K ** -0.5)).astype(np.float32).reshape(mix, K)


def make_scale(seed: int = SEED_SCALE) -> np.ndarray:
    return (0.5 + uniform(seed, 0, 3)).astype(np.float32)


def make_base(seed: int = SEED_BASE, mix: int = MIX) -> np.ndarray:
    return (0.1 * normal(seed, 0, mix)).astype(np.float32)


def layer_seeds(i: int) -> tuple[int, int, int]:
    """Seeds (W, hc_scale, hc_base) of call i in the 43-layer, 86-call stack."""
    return 1000 + 3 * i, 1001 + 3 * i, 1002 + 3 * i


CONFIGS = {
    "m16": dict(M=16, outliers=False),
    "m512_outliers": dict(M=512, outliers=True),
    "m4096": dict(M=4096, outliers=False),
    "decode_sweep": dict(Ms=(1, 4, 16, 64, 128, 256), outliers=False),
    "stack86_m16384": dict(M=16384, calls=86, outliers=False),
}

RMS_EPS = 1e-6
HC_EPS = 0.0
SINKHORN_ITERS = 20
