"""Host check of the allocation-free AllReduce's sizing (no GPU).

pl_allreduce_noalloc keeps its work list and flag words in a static device
array: a 4 MiB region of which the first 64 KiB hold flag words and counters
(at most 2,048 flags), and a 28 MiB staging ring, with 256 KiB chunks.  Its
documented limit is R <= 8 and 256 MiB per rank.  The same staged, fused
AllReduce plan, derived here on the host for every R and element type at that
limit, must fit those regions, so that no request the entry point accepts is
refused for want of room (and a planner change that outgrows them fails here).
"""
import pytest

import synth
from copy_reduce_datapath_gb300 import purlin as P

LIST_BYTES = (4 << 20) - (64 << 10)
MAX_FLAGS = 2048
RING_BYTES = 28 << 20
CHUNK_BYTES = 256 << 10
LIMIT_BYTES = 256 << 20
ESIZE = {"bf16": 2, "fp16": 2, "fp32": 4}


def _al(n):
    return (n + 255) // 256 * 256


@pytest.mark.parametrize("num_sms", [148, 152])
@pytest.mark.parametrize("dtype", ["bf16", "fp32", "fp16"])
@pytest.mark.parametrize("R", list(range(1, 9)))
def test_work_list_fits_the_static_array_at_the_limit(R, dtype, num_sms):
    count = LIMIT_BYTES // ESIZE[dtype]
    L = P.pl_layout_partitioned(R, synth.equal_lengths(count, R))
    pol = P.pl_policy_default(path=P.PL_PATH_STAGED, allreduce_form=P.PL_AR_FUSED, chunk_bytes=CHUNK_BYTES)
    plan = P.pl_plan_create(L, L, "sum", dtype, R, pol, num_sms, RING_BYTES)
    try:
        st = P.pl_plan_get_stats(plan)
    finally:
        P.pl_plan_destroy(plan)
        P.pl_layout_destroy(L)
    size = _al(st.items * 32) + _al(st.refs * 24) + st.syncs * 16
    assert size <= LIST_BYTES, f"work list {size} bytes"
    assert st.flags <= MAX_FLAGS
    assert st.slots * st.slot_elems * ESIZE[dtype] * R <= RING_BYTES
