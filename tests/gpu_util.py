"""Helpers for the GPU parity tests: host <-> device transfers of buffers in
the oracle's representation (bf16 and fp16 as uint16 bit patterns, fp8 as
uint8 bytes, fp32 as float32)."""
from __future__ import annotations

import numpy as np
import torch

import synth

TORCH = {"bf16": torch.bfloat16, "fp32": torch.float32, "fp16": torch.float16, "fp8": torch.uint8}
NP = {"bf16": np.uint16, "fp32": np.float32, "fp16": np.uint16, "fp8": np.uint8}
# integer views of the same bytes (torch and numpy)
_TBITS = {"bf16": torch.int16, "fp16": torch.int16, "fp32": torch.int32, "fp8": torch.uint8}
_NBITS = {1: np.uint8, 2: np.uint16, 4: np.uint32}


def host(kind, dtype, seed, rank, n):
    """Seeded host input as the oracle's numpy representation."""
    t = synth.host_tensor(kind, dtype, seed, rank, n)
    return to_np(t, dtype)


def to_np(t, dtype):
    t = t.detach().cpu().contiguous()
    if dtype in ("bf16", "fp16"):
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def to_dev(a, dtype, device="cuda"):
    a = np.ascontiguousarray(a)
    if dtype in ("bf16", "fp16"):
        return torch.from_numpy(a.view(np.int16)).view(TORCH[dtype]).to(device)
    return torch.from_numpy(a).to(device)


def empty(n, dtype, device="cuda", fill=None):
    t = torch.empty(int(n), dtype=TORCH[dtype], device=device)
    if fill is not None:
        t.view(_TBITS[dtype]).fill_(fill)
    return t


def bits(a):
    """The raw bit patterns of a numpy array of 1-, 2- or 4-byte elements."""
    a = np.asarray(a)
    return a.view(_NBITS[a.dtype.itemsize])


def assert_equal(got, want, what=""):
    """Bit-exact comparison with the first differing index in the message."""
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    assert got.dtype.itemsize == want.dtype.itemsize, f"{what}: element sizes differ"
    bad = np.nonzero(bits(got) != bits(want))[0]
    assert bad.size == 0, (f"{what}: {bad.size} of {got.size} elements differ; first at {bad[0]}: "
                           f"got {got[bad[0]]!r} want {want[bad[0]]!r}")


# ------------------------------------------------- collectives under test

# Canary patterns around every output: NaNs no reduction or conversion here
# produces.  One-byte elements can take every pattern, so there a stray write
# of 0xA5 would go unseen (1 in 256 per guard element).
CANARY = {"bf16": 0x7FA5, "fp16": 0x7DA5, "fp32": 0x7FA5A5A5, "fp8": 0xA5}
GUARD = 37  # elements of canary before and after every output
SIZE = {"bf16": 2, "fp16": 2, "fp32": 4, "fp8": 1}


def aligned_guard(dtype):
    """Elements of a 64-byte canary: outputs after it keep the allocation's 16-byte alignment."""
    return 64 // SIZE[dtype]


def policies():
    from copy_reduce_datapath_gb300 import purlin as P
    return {
        "zs": P.pl_policy_default(),
        "zs_small_chunks": P.pl_policy_default(chunk_bytes=4096),
        "staged": P.pl_policy_default(path=P.PL_PATH_STAGED, chunk_bytes=8192),
    }


def ar_policies():
    from copy_reduce_datapath_gb300 import purlin as P
    return {
        "zs_fused": P.pl_policy_default(),
        "zs_composed": P.pl_policy_default(allreduce_form=P.PL_AR_COMPOSED, chunk_bytes=8192),
        "zs_notified": P.pl_policy_default(allreduce_form=P.PL_AR_NOTIFIED, chunk_bytes=8192),
        "staged_fused": P.pl_policy_default(path=P.PL_PATH_STAGED, chunk_bytes=8192),
        "staged_composed": P.pl_policy_default(path=P.PL_PATH_STAGED, allreduce_form=P.PL_AR_COMPOSED,
                                               chunk_bytes=8192),
    }


class Outs:
    """Output buffers with canary guard regions on both sides: `lead` elements
    before each (GUARD by default, which leaves outputs off 16-byte alignment
    for every element size) and GUARD after."""

    def __init__(self, sizes, dtype, lead=GUARD):
        self.dtype = dtype
        self.lead = int(lead)
        self.sizes = [int(s) for s in sizes]
        self.full = [empty(self.lead + s + GUARD, dtype, fill=CANARY[dtype]) for s in self.sizes]
        self.views = [f[self.lead:self.lead + s] for f, s in zip(self.full, self.sizes)]

    def ptrs(self):
        from copy_reduce_datapath_gb300 import purlin as P
        return P.ptrs(self.views)

    def counts(self):
        return self.sizes

    def host(self, r):
        return to_np(self.views[r], self.dtype)

    def check_guards(self):
        canary = CANARY[self.dtype] & 0xFFFFFFFF
        for r, f in enumerate(self.full):
            b = bits(to_np(f, self.dtype))
            assert np.all(b[:self.lead] == canary), f"rank {r}: write before its output"
            assert np.all(b[self.lead + self.sizes[r]:] == canary), f"rank {r}: write past its output"


def run(ctx, lin, lout, op, dtype, ins_host, out_sizes, pol):
    """pl_collective over host inputs copied to the device, twice: into outputs
    at 16-byte aligned addresses (the kernels for aligned plans, the inline
    form) and into outputs off that alignment (the realigning kernels).  Both
    must agree bit for bit; the outputs as host arrays."""
    from copy_reduce_datapath_gb300 import purlin as P
    R = len(ins_host)
    ins = [to_dev(a, dtype) for a in ins_host]
    s = P.stream_handle()
    got = None
    for lead in (aligned_guard(dtype), GUARD):
        outs = Outs(out_sizes, dtype, lead)
        P.pl_collective(ctx, lin, lout, op, dtype, R, P.ptrs(ins), P.counts(ins), outs.ptrs(), outs.counts(), pol, s)
        assert P.pl_ctx_status(ctx, s) == P.PL_OK
        outs.check_guards()
        res = [outs.host(r) for r in range(R)]
        if got is None:
            got = res
        else:
            for r in range(R):
                assert_equal(res[r], got[r], f"misaligned outputs, rank {r}")
    return got
