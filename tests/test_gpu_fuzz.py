"""Random layout pairs (tests/fuzz_layouts.py) on the GPU through the C ABI,
against the oracle bit for bit: copies, sums and maxima of bf16, fp16, fp32
and one-byte elements over 1 to 8 ranks, regions at every alignment (some
strided, some empty), buffers whose bases sit off 16-byte alignment, and
every policy form (automatic, vector, bulk ring, inline parameters, staged,
both composed forms, small chunks, a forced three-CTA grid).  Output elements
no part names stay zero on both sides; canaries around each output catch
stray writes."""
import numpy as np
import pytest
import torch

import oracle
from copy_reduce_datapath_gb300 import purlin as P

import fuzz_layouts as F
from gpu_util import CANARY, SIZE, TORCH, _TBITS, bits, host, to_dev, to_np

pytestmark = pytest.mark.gpu

GUARD = 29


@pytest.fixture(scope="module")
def ctx():
    torch.cuda.set_device(0)
    c = P.pl_ctx_create(0, 8 << 20)
    yield c
    P.pl_ctx_destroy(c)


def device_view(host_arr, dtype, lead):
    """A device copy of host_arr starting `lead` elements into its allocation."""
    full = torch.empty(lead + host_arr.size, dtype=TORCH[dtype], device="cuda")
    full[lead:].copy_(to_dev(host_arr, dtype))
    return full, full[lead:]


@pytest.mark.parametrize("seed", range(96))
def test_random_layout_pair_on_gpu(ctx, seed):
    c = F.case(seed)
    R, dtype, op = c["R"], c["dtype"], c["op"]
    ins = [host("normal", dtype, 900 + seed, r, c["in_sizes"][r]) for r in range(R)]
    want = oracle.collective(op, dtype, c["lin"], c["lout"], ins, c["out_sizes"])
    lead_in, lead_out = seed % 5, (seed * 3) % 7
    dev_in = [device_view(a, dtype, lead_in)[1] for a in ins]
    fulls, outs = [], []
    for n in c["out_sizes"]:
        full = torch.empty(lead_out + n + 2 * GUARD, dtype=TORCH[dtype], device="cuda")
        full.view(_TBITS[dtype]).fill_(CANARY[dtype])
        view = full[lead_out + GUARD:lead_out + GUARD + n]
        view.zero_()
        fulls.append(full)
        outs.append(view)
    lin, lout = P.pl_layout_create(R, c["lin"]), P.pl_layout_create(R, c["lout"])
    s = P.stream_handle()
    P.pl_collective(ctx, lin, lout, op, dtype, R, P.ptrs(dev_in), P.counts(dev_in), P.ptrs(outs), P.counts(outs),
                    F.policy(P, c["policy"]), s)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    canary = CANARY[dtype] & ((1 << (8 * SIZE[dtype])) - 1)
    for r in range(R):
        got = to_np(outs[r], dtype)
        bad = np.nonzero(bits(got) != bits(want[r]))[0]
        assert bad.size == 0, (f"seed {seed} ({c['policy']}, {op}, {dtype}, R={R}) rank {r}: {bad.size} of "
                               f"{got.size} differ, first at {bad[0]}")
        b = bits(to_np(fulls[r], dtype))
        n = c["out_sizes"][r]
        assert np.all(b[:lead_out + GUARD] == canary) and np.all(b[lead_out + GUARD + n:] == canary), \
            f"seed {seed} rank {r}: a write outside the output"
