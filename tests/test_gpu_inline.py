"""GPU parity of the inline-parameter launches (PL_ATOM_INLINE): small plans
whose whole work list travels in the kernel's parameters, one work item per
CTA.  Every collective, element type and reduction that the form takes,
against the CPU oracle bit for bit, with the plan checked to be in the inline
form; items with a ragged tail; items of many vectors per thread (the form
forced by policy); reductions in place (one thread per vector for all
destinations); buffers that are not 16-byte aligned at launch (the same work
list on the persistent kernel)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from copy_reduce_datapath_gb300 import purlin as P

from gpu_util import Outs, assert_equal, host, run, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    torch.cuda.set_device(0)
    c = P.pl_ctx_create(0, 0)
    yield c
    P.pl_ctx_destroy(c)


def num_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def datapath(lin, lout, op, dtype, R, pol=None):
    plan = P.pl_plan_create(lin, lout, op, dtype, R, pol, num_sms())
    try:
        st = P.pl_plan_get_stats(plan)
        return st.datapath, st.items, st.ctas
    finally:
        P.pl_plan_destroy(plan)


def forced():
    return P.pl_policy_default(datapath=P.PL_ATOM_INLINE)


def lengths(n, R):
    """Partitions of a multiple of 16 elements (16-byte aligned offsets for
    every element size), the remainder, a ragged tail, to the last."""
    q = n // R // 16 * 16
    return [q] * (R - 1) + [n - q * (R - 1)]


REDUCIBLE = ["bf16", "fp16", "fp32"]
ALL = REDUCIBLE + ["fp8"]


@pytest.mark.parametrize("dtype", ALL)
@pytest.mark.parametrize("n", [128, 512, 8 * 64 + 5, 8 * 1024 + 13, 1 << 15])
def test_allgather_inline(ctx, dtype, n):
    R = 8
    lens = lengths(n, R)
    ins = [host("normal", dtype, 40, r, lens[r]) for r in range(R)]
    lin, lout = P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens)
    assert datapath(lin, lout, "copy", dtype, R)[0] == P.PL_ATOM_INLINE
    got = run(ctx, lin, lout, "copy", dtype, ins, [n] * R, None)
    want = oracle.allgather(ins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


@pytest.mark.parametrize("dtype", REDUCIBLE)
@pytest.mark.parametrize("op", ["sum", "max"])
@pytest.mark.parametrize("n", [128, 8 * 64 + 5, 8 * 4096 + 7, 1 << 16])
def test_allreduce_inline(ctx, dtype, op, n):
    R = 8
    ins = [host("normal", dtype, 41, r, n) for r in range(R)]
    L = P.pl_layout_partitioned(R, lengths(n, R))
    assert datapath(L, L, op, dtype, R)[0] == P.PL_ATOM_INLINE
    got = run(ctx, L, L, op, dtype, ins, [n] * R, None)
    want = oracle.allreduce(ins, dtype, op)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


@pytest.mark.parametrize("dtype", REDUCIBLE)
@pytest.mark.parametrize("n", [256, 8 * 1024 + 3, 1 << 19])
def test_reducescatter_inline(ctx, dtype, n):
    R = 8
    lens = lengths(n, R)
    ins = [host("uniform", dtype, 42, r, n) for r in range(R)]
    lin, lout = P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned(R, lens)
    assert datapath(lin, lout, "sum", dtype, R)[0] == P.PL_ATOM_INLINE
    got = run(ctx, lin, lout, "sum", dtype, ins, lens, None)
    want = oracle.reducescatter(ins, lens, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_alltoall_inline(ctx, dtype):
    """MoE-dispatch shape, small: 8 ranks x 8 partitions of 4 tokens x 64 hidden."""
    R, tok, hid = 8, 4, 64
    M = [[tok * hid] * R for _ in range(R)]
    n = R * tok * hid
    ins = [host("normal", dtype, 43, r, n) for r in range(R)]
    lin, lout = P.pl_layout_alltoall_in(R, M), P.pl_layout_alltoall_out(R, M)
    assert datapath(lin, lout, "copy", dtype, R)[0] == P.PL_ATOM_INLINE
    got = run(ctx, lin, lout, "copy", dtype, ins, [n] * R, None)
    want = oracle.alltoall(ins, M, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


def test_small_parameter_block_and_single_rank(ctx):
    """A 1 KiB AllReduce (8 items: the small parameter block) and R = 1 copies and sums."""
    R, n = 8, 512
    L = P.pl_layout_partitioned(R, [n // R] * R)
    form, items, ctas = datapath(L, L, "sum", "bf16", R)
    assert form == P.PL_ATOM_INLINE and items == ctas == 8
    ins = [host("normal", "bf16", 44, r, n) for r in range(R)]
    got = run(ctx, L, L, "sum", "bf16", ins, [n] * R, None)
    want = oracle.allreduce(ins, "bf16")
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")
    for dtype in ("bf16", "fp32"):
        x = host("normal", dtype, 45, 0, 1001)
        L1 = P.pl_layout_rank_owned(1, [1001])
        for op in ("copy", "sum"):
            assert datapath(L1, L1, op, dtype, 1)[0] == P.PL_ATOM_INLINE
            assert_equal(run(ctx, L1, L1, op, dtype, [x], [1001], None)[0], x)


def test_sixteen_ranks_inline_sixty_four_not(ctx):
    """R = 16 fits the parameter block (16 items of 32 references); R = 64 (64
    items of 128 references) does not and runs on the persistent kernel."""
    for R, form in ((16, P.PL_ATOM_INLINE), (64, P.PL_ATOM_VECTOR)):
        n = R * 24
        ins = [host("normal", "bf16", 46, r, n) for r in range(R)]
        L = P.pl_layout_partitioned(R, [24] * R)
        assert datapath(L, L, "sum", "bf16", R)[0] == form
        got = run(ctx, L, L, "sum", "bf16", ins, [n] * R, None)
        want = oracle.allreduce(ins, "bf16")
        for r in range(R):
            assert_equal(got[r], want[r], f"R {R} rank {r}")


@pytest.mark.parametrize("coll", ["allgather", "allreduce", "reducescatter"])
def test_forced_inline_many_vectors_per_thread(ctx, coll):
    """Forced by policy: items of up to tens of vectors per thread (a thread
    per vector and several destinations each) and ragged tails."""
    R, dtype = 8, "bf16"
    pol = forced()
    if coll == "allgather":
        n = (1 << 20) + 8 * 3
        lens = lengths(n, R)
        ins = [host("normal", dtype, 47, r, lens[r]) for r in range(R)]
        lin, lout = P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens)
        form, items, _ = datapath(lin, lout, "copy", dtype, R, pol)
        assert form == P.PL_ATOM_INLINE and items <= 152
        got = run(ctx, lin, lout, "copy", dtype, ins, [n] * R, pol)
        want = oracle.allgather(ins, dtype)
    elif coll == "allreduce":
        n = (1 << 19) + 5
        ins = [host("normal", dtype, 48, r, n) for r in range(R)]
        lin = lout = P.pl_layout_partitioned(R, lengths(n, R))
        assert datapath(lin, lout, "sum", dtype, R, pol)[0] == P.PL_ATOM_INLINE
        got = run(ctx, lin, lout, "sum", dtype, ins, [n] * R, pol)
        want = oracle.allreduce(ins, dtype)
    else:
        n = (1 << 22) + 9
        lens = lengths(n, R)
        ins = [host("uniform", dtype, 49, r, n) for r in range(R)]
        lin, lout = P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned(R, lens)
        assert datapath(lin, lout, "sum", dtype, R, pol)[0] == P.PL_ATOM_INLINE
        got = run(ctx, lin, lout, "sum", dtype, ins, lens, pol)
        want = oracle.reducescatter(ins, lens, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


@pytest.mark.parametrize("dtype", REDUCIBLE)
@pytest.mark.parametrize("op", ["sum", "max"])
@pytest.mark.parametrize("datapath_policy", ["auto", "vector"])
@pytest.mark.parametrize("n", [8 * 8, 8 * 64 + 5, 8 * 512 + 3])
def test_allreduce_in_place_small(ctx, dtype, op, datapath_policy, n):
    """Outputs that are the inputs: every destination of an item is also one of
    its sources.  On the inline form and, with the vector datapath forced, on
    the persistent kernel's small-item path: each vector is reduced whole
    before any of its destinations is written."""
    R = 8
    ins = [host("normal", dtype, 50, r, n) for r in range(R)]
    want = oracle.allreduce(ins, dtype, op)
    pol = P.pl_policy_default(datapath=P.PL_ATOM_VECTOR) if datapath_policy == "vector" else None
    L = P.pl_layout_partitioned(R, lengths(n, R))
    want_form = P.PL_ATOM_VECTOR if pol is not None else P.PL_ATOM_INLINE
    assert datapath(L, L, op, dtype, R, pol)[0] == want_form
    for rep in range(3):
        bufs = [to_dev(a, dtype) for a in ins]
        s = P.stream_handle()
        P.pl_collective(ctx, L, L, op, dtype, R, P.ptrs(bufs), [n] * R, P.ptrs(bufs), [n] * R, pol, s)
        assert P.pl_ctx_status(ctx, s) == P.PL_OK
        for r in range(R):
            assert_equal(to_np(bufs[r], dtype), want[r], f"rep {rep} rank {r}")


@pytest.mark.parametrize("shift", [1, 3, 4])
def test_misaligned_buffers_inline(ctx, shift):
    """An inline-form plan of small items over buffers off 16-byte alignment
    (every output at the same shift): destination heads peeled, sources
    spliced, in the inline kernel."""
    R, n, dtype = 8, 8 * 64, "bf16"
    L = P.pl_layout_partitioned(R, [64] * R)
    assert datapath(L, L, "sum", dtype, R)[0] == P.PL_ATOM_INLINE
    ins = [host("normal", dtype, 51, r, n) for r in range(R)]
    big = [to_dev(np.concatenate([np.zeros(shift + r, np.uint16), a]), dtype) for r, a in enumerate(ins)]
    views = [b[shift + r:] for r, b in enumerate(big)]
    outs = Outs([n + shift] * R, dtype)
    ovs = [v[shift:] for v in outs.views]
    s = P.stream_handle()
    P.pl_collective(ctx, L, L, "sum", dtype, R, P.ptrs(views), P.counts(views), P.ptrs(ovs), P.counts(ovs), None, s)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    outs.check_guards()
    want = oracle.allreduce(ins, dtype)
    for r in range(R):
        assert_equal(to_np(ovs[r], dtype), want[r], f"rank {r}")


def test_inline_plans_that_fall_back(ctx):
    """The same work list on the persistent kernel: (a) small items whose
    destinations are at different addresses mod 16 (outputs at different
    shifts), (b) an inline plan of large items over buffers off alignment."""
    R, dtype = 8, "bf16"
    # (a)
    n = 8 * 64
    L = P.pl_layout_partitioned(R, [64] * R)
    ins = [host("normal", dtype, 52, r, n) for r in range(R)]
    dev = [to_dev(a, dtype) for a in ins]
    outs = Outs([n + 8] * R, dtype)
    ovs = [v[r % 8:] [:n] for r, v in enumerate(outs.views)]
    s = P.stream_handle()
    P.pl_collective(ctx, L, L, "sum", dtype, R, P.ptrs(dev), [n] * R, P.ptrs(ovs), [n] * R, None, s)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    outs.check_guards()
    want = oracle.allreduce(ins, dtype)
    for r in range(R):
        assert_equal(to_np(ovs[r], dtype), want[r], f"(a) rank {r}")
    # (b) AllGather at 8 MiB per rank: inline form, items of thousands of vectors
    n = 1 << 22
    lens = [n // R] * R
    lin, lout = P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens)
    assert datapath(lin, lout, "copy", dtype, R)[0] == P.PL_ATOM_INLINE
    gins = [host("normal", dtype, 53, r, n // R) for r in range(R)]
    got = run(ctx, lin, lout, "copy", dtype, gins, [n] * R, None)  # aligned outputs, then misaligned
    want = oracle.allgather(gins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"(b) rank {r}")


@pytest.mark.parametrize("dtype", ALL)
@pytest.mark.parametrize("N", [(1 << 12) + 7, (1 << 16) + 3, (1 << 19) + 5])
def test_v_forms_inline(ctx, dtype, N):
    """AllGatherV, ReduceScatterV (sum and maximum) and AllToAllV with Zipf
    lengths: partitions at every misalignment, in the inline form."""
    R = 8
    if dtype == "fp32":
        N = N // 2 + 1  # the same bytes
    lens = synth.zipf_lengths(N, R, 0.125, seed=54)
    ins = [host("normal", dtype, 54, r, lens[r]) for r in range(R)]
    lin, lout = P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens)
    assert datapath(lin, lout, "copy", dtype, R)[0] == P.PL_ATOM_INLINE
    got = run(ctx, lin, lout, "copy", dtype, ins, [N] * R, None)
    want = oracle.allgather(ins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"AGV rank {r}")
    if dtype != "fp8":
        rins = [host("normal", dtype, 55, r, N) for r in range(R)]
        for op in ("sum", "max"):
            lin, lout = P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned(R, lens)
            assert datapath(lin, lout, op, dtype, R)[0] == P.PL_ATOM_INLINE
            got = run(ctx, lin, lout, op, dtype, rins, lens, None)
            want = oracle.reducescatter(rins, lens, dtype, op)
            for r in range(R):
                assert_equal(got[r], want[r], f"RSV {op} rank {r}")
    if N < 1 << 17:
        m = synth.zipf_matrix(N, R, 0.125, seed=56)
        ains = [host("normal", dtype, 56, r, sum(m[r])) for r in range(R)]
        lin, lout = P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m)
        assert datapath(lin, lout, "copy", dtype, R)[0] == P.PL_ATOM_INLINE
        got = run(ctx, lin, lout, "copy", dtype, ains, [sum(m[j][r] for j in range(R)) for r in range(R)], None)
        want = oracle.alltoall(ains, m, dtype)
        for r in range(R):
            assert_equal(got[r], want[r], f"A2AV rank {r}")
