"""Helpers for the GPU parity tests: host <-> device transfers of bf16/fp32
buffers (bf16 kept as uint16 bit patterns on the host, as the oracle wants)."""
from __future__ import annotations

import numpy as np
import torch

import synth

TORCH = {"bf16": torch.bfloat16, "fp32": torch.float32}
NP = {"bf16": np.uint16, "fp32": np.float32}


def host(kind, dtype, seed, rank, n):
    """Seeded host input as the oracle's numpy representation."""
    t = synth.host_tensor(kind, dtype, seed, rank, n)
    return to_np(t, dtype)


def to_np(t, dtype):
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def to_dev(a, dtype, device="cuda"):
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def empty(n, dtype, device="cuda", fill=None):
    t = torch.empty(int(n), dtype=TORCH[dtype], device=device)
    if fill is not None:
        t.view(torch.int16 if dtype == "bf16" else torch.int32).fill_(fill)
    return t


def assert_equal(got, want, what=""):
    """Bit-exact comparison with the first differing index in the message."""
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    gb = got.view(np.uint16 if got.dtype == np.uint16 else np.uint32)
    wb = want.view(np.uint16 if want.dtype == np.uint16 else np.uint32)
    bad = np.nonzero(gb != wb)[0]
    assert bad.size == 0, (f"{what}: {bad.size} of {got.size} elements differ; first at {bad[0]}: "
                           f"got {got[bad[0]]!r} want {want[bad[0]]!r}")
