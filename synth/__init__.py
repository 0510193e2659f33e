"""Seeded synthetic inputs for the Purlin collectives (input generation only).

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It holds no collective arithmetic: it only draws numbers and
partition lengths.  Nothing here sums, rounds to an output type or places data.

Generators
----------
* ``u64_stream(seed, rank, n)`` -- SplitMix64 (Steele, Lea & Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014): the state advances
  by the golden-ratio increment and each output is the state passed through the
  published 64-bit finaliser.  Written counter-style, output ``i`` (0-based) is
  ``mix(key + (i + 1) * GAMMA)``; the per-(seed, rank) key is itself one mix of
  ``seed * GAMMA + rank``.
* ``uniform_pm1_f32``      -- U(-1, 1) on a 2^-23 grid (24 random bits).
* ``int_uniform_f32``      -- integers uniform in [lo, hi] (Lemire's
  multiply-shift range reduction of the top 32 bits), stored as fp32.
* ``normal_f32``           -- N(0, 1) by the Box-Muller transform in float64,
  then rounded to fp32.
* ``to_bf16``              -- fp32 -> bf16 conversion by PyTorch's CPU cast
  (library rounding; used only to prepare inputs).
* ``zipf_lengths``         -- partition lengths proportional to (i+1)^-s,
  largest-remainder rounding, then a seeded Fisher-Yates shuffle.
* ``host_normal_bf16_torch`` -- N(0,1) bf16 from PyTorch's seeded CPU generator,
  for large host-side samples.
* ``device_normal_bf16`` / ``device_uniform_pm1`` -- large inputs drawn on the
  GPU by PyTorch's seeded Philox generator (too large to draw on the host in
  reasonable time); used for the full-size benchmark and sampled parity checks,
  where the checker copies the sampled input slices back to the host.

The Purlin pages (Purlin: Separating Orchestration from the Datapath of
Collectives, Figure 16 caption) fix only the Zipf exponent s = 0.125 for the
variable-length collectives; the rest of the recipe is this module's choice.
"""
from __future__ import annotations

import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output finaliser on a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def stream_key(seed: int, rank: int) -> np.uint64:
    """Key of the SplitMix64 stream that feeds logical rank ``rank`` under ``seed``."""
    with np.errstate(over="ignore"):
        z = np.array([seed], dtype=np.uint64) * GAMMA + np.uint64(rank)
    return _mix(z)[0]


def u64_stream(seed: int, rank: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs ``start .. start+n-1`` of the SplitMix64 stream of (seed, rank)."""
    key = stream_key(seed, rank)
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + i * GAMMA)


def uniform_pm1_f32(seed: int, rank: int, n: int) -> np.ndarray:
    """U(-1, 1): k * 2^-23 - 1 for a uniform 24-bit k; exact in fp32."""
    k = (u64_stream(seed, rank, n) >> np.uint64(40)).astype(np.float64)
    return (k * 2.0 ** -23 - 1.0).astype(np.float32)


def int_uniform_f32(seed: int, rank: int, n: int, lo: int = -8, hi: int = 8) -> np.ndarray:
    """Integers uniform in [lo, hi] (inclusive), as fp32."""
    span = np.uint64(hi - lo + 1)
    top = u64_stream(seed, rank, n) >> np.uint64(32)
    with np.errstate(over="ignore"):
        k = (top * span) >> np.uint64(32)
    return (k.astype(np.int64) + lo).astype(np.float32)


def normal_f32(seed: int, rank: int, n: int) -> np.ndarray:
    """N(0, 1) by Box-Muller on consecutive output pairs, computed in float64."""
    m = (n + 1) // 2
    x = u64_stream(seed, rank, 2 * m)
    u1 = ((x[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53  # (0, 1]
    u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53          # [0, 1)
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * math.pi * u2)
    z[1::2] = r * np.sin(2.0 * math.pi * u2)
    return z[:n].astype(np.float32)


def to_bf16(a: np.ndarray):
    """fp32 numpy array -> bf16 torch CPU tensor (PyTorch's round-to-nearest-even cast)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def host_tensor(kind: str, dtype: str, seed: int, rank: int, n: int):
    """A 1-D torch CPU tensor of ``n`` elements for logical rank ``rank``.

    kind: "normal" (N(0,1)), "uniform" (U(-1,1)) or "int8range" (integers in [-8, 8]).
    dtype: "bf16", "fp16" (PyTorch's round-to-nearest-even casts of the fp32 draw),
    "fp32", or "fp8": one-byte elements, for which ``kind`` is ignored and every
    byte is drawn uniformly from the SplitMix64 stream (all 256 patterns occur).
    """
    import torch
    if dtype == "fp8":
        return torch.from_numpy(random_bytes(seed, rank, n))
    if kind == "normal":
        a = normal_f32(seed, rank, n)
    elif kind == "uniform":
        a = uniform_pm1_f32(seed, rank, n)
    elif kind == "int8range":
        a = int_uniform_f32(seed, rank, n)
    else:
        raise ValueError(f"unknown input kind {kind!r}")
    if dtype == "bf16":
        return to_bf16(a)
    if dtype == "fp16":
        return torch.from_numpy(a).to(torch.float16)
    if dtype == "fp32":
        return torch.from_numpy(a)
    raise ValueError(f"unknown dtype {dtype!r}")


def random_bytes(seed: int, rank: int, n: int) -> np.ndarray:
    """n bytes, the top byte of each SplitMix64 output of stream (seed, rank)."""
    return (u64_stream(seed, rank, n) >> np.uint64(56)).astype(np.uint8)


def zipf_lengths(total: int, R: int, s: float, seed: int, stream: int = 0) -> list[int]:
    """Split ``total`` elements over ``R`` partitions with Zipf weights (i+1)^-s.

    Largest-remainder rounding (leftover elements go to the largest fractional
    parts, ties to the lower index), then a Fisher-Yates shuffle driven by the
    SplitMix64 stream (seed, 1000 + stream).  The lengths always sum to ``total``.
    """
    if R < 1 or total < 0:
        raise ValueError("need R >= 1 and total >= 0")
    w = [(i + 1) ** (-s) for i in range(R)]
    sw = sum(w)
    exact = [total * wi / sw for wi in w]
    base = [int(math.floor(e)) for e in exact]
    left = total - sum(base)
    order = sorted(range(R), key=lambda i: (-(exact[i] - base[i]), i))
    for i in order[:left]:
        base[i] += 1
    rnd = u64_stream(seed, 1000 + stream, R)
    for i in range(R - 1, 0, -1):
        j = int((int(rnd[i] >> np.uint64(32)) * (i + 1)) >> 32)
        base[i], base[j] = base[j], base[i]
    return base


def zipf_matrix(total: int, R: int, s: float, seed: int) -> list[list[int]]:
    """R x R length matrix for AllToAllV: row r (source r) is its own Zipf split of ``total``."""
    return [zipf_lengths(total, R, s, seed, stream=r) for r in range(R)]


def equal_lengths(total: int, R: int) -> list[int]:
    """Equal split: the first R-1 partitions get total // R, the last gets the rest."""
    q = total // R
    return [q] * (R - 1) + [total - q * (R - 1)]


def host_normal_bf16_torch(seed: int, rank: int, n: int):
    """N(0,1) bf16 on the host from PyTorch's seeded CPU generator (fast; for large
    host-side samples where the SplitMix64 Box-Muller stream would take minutes)."""
    import torch
    g = torch.Generator()
    g.manual_seed(device_seed(seed, rank))
    return torch.randn(n, generator=g, dtype=torch.float32).to(torch.bfloat16)


def device_seed(seed: int, rank: int) -> int:
    """Seed of PyTorch's device generator for (seed, rank)."""
    return int(stream_key(seed, rank) & np.uint64(0x7FFFFFFFFFFFFFFF))


def device_normal_bf16(seed: int, rank: int, n: int, device):
    """N(0,1) bf16 drawn on ``device`` by PyTorch's seeded generator (large inputs)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(device_seed(seed, rank))
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    step = 1 << 28
    for s in range(0, n, step):
        e = min(n, s + step)
        out[s:e] = torch.randn(e - s, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def device_uniform_pm1(seed: int, rank: int, n: int, device, dtype):
    """U(-1,1) drawn on ``device`` by PyTorch's seeded generator (large inputs)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(device_seed(seed, rank))
    out = torch.empty(n, dtype=dtype, device=device)
    step = 1 << 28
    for s in range(0, n, step):
        e = min(n, s + step)
        out[s:e] = (torch.rand(e - s, generator=g, device=device, dtype=torch.float32) * 2 - 1).to(dtype)
    return out


def device_bytes(seed: int, rank: int, n: int, device):
    """Uniform bytes drawn on ``device`` by PyTorch's seeded generator (large one-byte inputs)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(device_seed(seed, rank))
    return torch.randint(0, 256, (n,), generator=g, device=device, dtype=torch.uint8)


def device_int_f32(seed: int, rank: int, n: int, device, lo: int = -8, hi: int = 8):
    """Integers uniform in [lo, hi] (inclusive) as fp32, drawn on ``device`` by
    PyTorch's seeded generator (large inputs whose sums stay exact)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(device_seed(seed, rank))
    return torch.randint(lo, hi + 1, (n,), generator=g, device=device, dtype=torch.int32).to(torch.float32)
