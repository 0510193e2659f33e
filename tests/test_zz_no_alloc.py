"""The allocation-free AllReduce (pl_allreduce_noalloc) against the oracle.

pl_allreduce_noalloc serves callers that cannot allocate device memory (a
fixed memory budget, an allocator they do not own, or a path where an
allocation's implicit synchronisation is not acceptable): its flag words, work
list and staging ring live in the library's static device array.  Its results
must equal the oracle's AllReduce bit for bit -- the tolerance every parity
test here uses -- on two calls in a row that reuse that array.  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes when run alone in a fresh process.
"""
import pytest
import torch

import oracle
from copy_reduce_datapath_gb300 import purlin as P

from gpu_util import assert_equal, host, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,R,n", [("bf16", 8, (1 << 20) + 77), ("fp32", 3, 3 * 4096), ("bf16", 5, 999),
                                       ("fp16", 8, (1 << 18) + 3)])
def test_matches_oracle_on_two_calls_in_a_row(dtype, R, n):
    torch.cuda.set_device(0)
    s = P.stream_handle()
    calls = []
    for seed in (30, 31):  # two calls in a row with different inputs (the second reuses the uploaded list)
        h = [host("normal", dtype, seed, r, n) for r in range(R)]
        ins = [to_dev(x, dtype) for x in h]
        out = [torch.zeros_like(x) for x in ins]
        calls.append((h, ins, out))
    # Back to back on one stream: the second call reuses the static array at once.
    assert P.pl_allreduce_noalloc(dtype, R, n, P.ptrs(calls[0][1]), P.ptrs(calls[0][2]), False, s) == P.PL_OK
    assert P.pl_allreduce_noalloc(dtype, R, n, P.ptrs(calls[1][1]), P.ptrs(calls[1][2]), True, s) == P.PL_OK
    for k, (h, ins, out) in enumerate(calls):
        want = oracle.allreduce(h, dtype)
        for r in range(R):
            assert_equal(to_np(out[r], dtype), want[r], f"call {k} rank {r}")


def test_allocates_nothing_and_runs_in_place():
    torch.cuda.set_device(0)
    dtype, R, n = "bf16", 8, 1 << 16
    s = P.stream_handle()
    h = [host("normal", dtype, 32, r, n) for r in range(R)]
    want = oracle.allreduce(h, dtype)
    ins = [to_dev(x, dtype) for x in h]
    bufs = [x.clone() for x in ins]
    out = [torch.empty_like(x) for x in ins]
    # First call on this device: sets up the array's address (and loads the kernel).
    assert P.pl_allreduce_noalloc(dtype, R, n, P.ptrs(ins), P.ptrs(out), True, s) == P.PL_OK
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    assert P.pl_allreduce_noalloc(dtype, R, n, P.ptrs(ins), P.ptrs(out), True, s) == P.PL_OK
    assert P.pl_allreduce_noalloc(dtype, R, n, P.ptrs(bufs), P.ptrs(bufs), True, s) == P.PL_OK  # in place
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    for r in range(R):
        assert_equal(to_np(out[r], dtype), want[r], f"rank {r}")
        assert_equal(to_np(bufs[r], dtype), want[r], f"in place rank {r}")


def test_alternating_sizes_upload_their_own_lists():
    """A call whose work list differs from the one the array holds uploads its
    own; going back to the first size uploads that list again."""
    torch.cuda.set_device(0)
    dtype, R = "bf16", 4
    s = P.stream_handle()
    for k, n in enumerate((5000, 70001, 5000)):
        h = [host("normal", dtype, 40 + k, r, n) for r in range(R)]
        ins = [to_dev(x, dtype) for x in h]
        out = [torch.zeros_like(x) for x in ins]
        assert P.pl_allreduce_noalloc(dtype, R, n, P.ptrs(ins), P.ptrs(out), True, s) == P.PL_OK
        want = oracle.allreduce(h, dtype)
        for r in range(R):
            assert_equal(to_np(out[r], dtype), want[r], f"call {k} rank {r}")


def test_rejects_sizes_beyond_its_limit():
    torch.cuda.set_device(0)
    x = [torch.zeros(8, dtype=torch.bfloat16, device="cuda") for _ in range(9)]
    big = (256 << 20) // 2 + 1  # one element beyond 256 MiB per rank
    assert P.pl_allreduce_noalloc("bf16", 8, big, P.ptrs(x[:8]), P.ptrs(x[:8]), True, 0) == P.PL_ERR_NOMEM
    assert P.pl_allreduce_noalloc("bf16", 9, 8, P.ptrs(x), P.ptrs(x), True, 0) == P.PL_ERR_NOMEM
    assert P.pl_allreduce_noalloc("bf16", 2, 8, P.ptrs(x[:2]), P.ptrs(x[:2]), True, 0) == P.PL_OK
    assert P.pl_allreduce_noalloc("fp8", 2, 8, P.ptrs(x[:2]), P.ptrs(x[:2]), True, 0) == P.PL_ERR_INVALID
