"""GPU parity: every collective through the C ABI against the CPU oracle,
element by element and bit for bit (copies, V offsets and rank-ordered fp32
sums are all exact by construction)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from copy_reduce_datapath_gb300 import purlin as P

from gpu_util import NP, TORCH, Outs, ar_policies, assert_equal, empty, host, policies, run, to_dev, to_np

pytestmark = pytest.mark.gpu

SCRATCH = 64 << 20


@pytest.fixture(scope="module")
def ctx():
    torch.cuda.set_device(0)
    c = P.pl_ctx_create(0, SCRATCH)
    yield c
    P.pl_ctx_destroy(c)


# ------------------------------------------------------- the five workloads


@pytest.mark.parametrize("name", list(ar_policies()))
def test_allreduce_three_ranks_fp32_integers(ctx, name):
    """R = 3, 3 x 4096 fp32 integers in [-8, 8], seed 0: exact, and equal to the oracle."""
    R, n = 3, 3 * 4096
    ins = [synth.int_uniform_f32(0, r, n) for r in range(R)]
    L = P.pl_layout_partitioned(R, [4096] * 3)
    got = run(ctx, L, L, "sum", "fp32", ins, [n] * R, ar_policies()[name])
    want = oracle.allreduce(ins, "fp32")
    exact = np.sum(np.stack([a.astype(np.int64) for a in ins]), axis=0)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")
        assert np.array_equal(got[r].astype(np.int64), exact)


@pytest.mark.parametrize("T", [1 << 10, 1 << 14, (1 << 20) + 0, 1 << 22])
@pytest.mark.parametrize("name", list(policies()))
def test_allgather_bf16(ctx, T, name):
    R = 8
    n = T // 2 // R
    ins = [host("normal", "bf16", 1, r, n) for r in range(R)]
    lin, lout = P.pl_layout_rank_owned(R, [n] * R), P.pl_layout_partitioned(R, [n] * R)
    got = run(ctx, lin, lout, "copy", "bf16", ins, [n * R] * R, policies()[name])
    want = oracle.allgather(ins, "bf16")
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


@pytest.mark.parametrize("T", [1 << 10, 1 << 16, 1 << 22])
@pytest.mark.parametrize("name", list(ar_policies()))
def test_allreduce_bf16(ctx, T, name):
    R = 8
    n = T // 2
    ins = [host("normal", "bf16", 1, r, n) for r in range(R)]
    got_dev = [to_dev(a, "bf16") for a in ins]
    outs = Outs([n] * R, "bf16")
    s = P.stream_handle()
    P.pl_allreduce(ctx, "bf16", R, n, P.ptrs(got_dev), outs.ptrs(), ar_policies()[name], s)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    outs.check_guards()
    want = oracle.allreduce(ins, "bf16")
    for r in range(R):
        assert_equal(outs.host(r), want[r], f"rank {r}")


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("T", [1 << 20, 1 << 22])
@pytest.mark.parametrize("variant", ["zs", "zs_in_place", "staged"])
def test_reducescatter(ctx, dtype, T, variant):
    R = 8
    S = 4 if dtype == "fp32" else 2
    N = T // S
    lens = [N // R] * R
    ins = [host("uniform", dtype, 2, r, N) for r in range(R)]
    want = oracle.reducescatter(ins, lens, dtype)
    lin = P.pl_layout_partitioned(R, lens)
    s = P.stream_handle()
    if variant == "zs_in_place":
        bufs = [to_dev(a, dtype) for a in ins]
        lout = P.pl_layout_rank_owned_inplace(R, lens)
        P.pl_collective(ctx, lin, lout, "sum", dtype, R, P.ptrs(bufs), P.counts(bufs), P.ptrs(bufs),
                        P.counts(bufs), None, s)
        assert P.pl_ctx_status(ctx, s) == P.PL_OK
        for k in range(R):
            o = k * lens[0]
            assert_equal(to_np(bufs[k][o:o + lens[k]], dtype), want[k], f"rank {k}")
    else:
        pol = P.pl_policy_default(path=P.PL_PATH_STAGED) if variant == "staged" else None
        got = run(ctx, lin, P.pl_layout_rank_owned(R, lens), "sum", dtype, ins, lens, pol)
        for k in range(R):
            assert_equal(got[k], want[k], f"rank {k}")


@pytest.mark.parametrize("name", ["zs", "staged"])
def test_alltoall_moe_dispatch_shape(ctx, name):
    """MoE token dispatch shape: per rank [tokens, 7168] bf16 split into 8 equal token groups
    (512 tokens per rank here; the full 4096-token shape runs in the sampled test)."""
    R, tokens, hidden = 8, 512, 7168
    n = tokens * hidden
    ins = [host("normal", "bf16", 3, r, n) for r in range(R)]
    m = [[n // R] * R for _ in range(R)]
    lin, lout = P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m)
    got = run(ctx, lin, lout, "copy", "bf16", ins, [n] * R, policies()[name])
    want = oracle.alltoall(ins, m, "bf16")
    for j in range(R):
        assert_equal(got[j], want[j], f"rank {j}")


@pytest.mark.parametrize("name", ["zs", "zs_small_chunks", "staged"])
def test_ulysses_sequence_to_head(ctx, name):
    """Ulysses re-partition [S, 32 heads, 128] per rank -> heads 4j..4j+3 of all ranks (S = 256 here)."""
    R, S, H, D = 8, 256, 32, 128
    ins = [host("normal", "bf16", 3, r, S * H * D) for r in range(R)]
    lin, lout = P.pl_layout_ulysses_in(R, S, H, D), P.pl_layout_ulysses_out(R, S, H, D)
    got = run(ctx, lin, lout, "copy", "bf16", ins, [S * H * D] * R, policies()[name])
    want = oracle.ulysses_a2a(ins, S, H, D, "bf16")
    for j in range(R):
        assert_equal(got[j], want[j], f"rank {j}")


@pytest.mark.parametrize("T", [1 << 20, (1 << 22) + 6])
@pytest.mark.parametrize("name", list(policies()))
def test_v_collectives_zipf(ctx, T, name):
    """AllGatherV, ReduceScatterV, AllToAllV with Zipf(s = 0.125) lengths: unaligned offsets."""
    R, dtype = 8, "bf16"
    N = T // 2
    pol = policies()[name]
    # AllGatherV: rank lengths sum to N.
    lens = synth.zipf_lengths(N, R, 0.125, seed=4)
    ins = [host("normal", dtype, 4, r, lens[r]) for r in range(R)]
    got = run(ctx, P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy", dtype, ins,
              [N] * R, pol)
    want = oracle.allgather(ins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"AGV rank {r}")
    # ReduceScatterV
    ins = [host("normal", dtype, 4, 100 + r, N) for r in range(R)]
    got = run(ctx, P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned(R, lens), "sum", dtype, ins,
              lens, pol)
    want = oracle.reducescatter(ins, lens, dtype)
    for k in range(R):
        assert_equal(got[k], want[k], f"RSV rank {k}")
    # AllToAllV: every source row is its own Zipf split.
    m = synth.zipf_matrix(N // R, R, 0.125, seed=4)
    ins = [host("normal", dtype, 4, 200 + r, sum(m[r])) for r in range(R)]
    outn = [sum(m[r][j] for r in range(R)) for j in range(R)]
    got = run(ctx, P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m), "copy", dtype, ins, outn, pol)
    want = oracle.alltoall(ins, m, dtype)
    for j in range(R):
        assert_equal(got[j], want[j], f"A2AV rank {j}")


# -------------------------------------------------------------- edge cases


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("n", [0, 1, 2, 7, 8, 9, 15, 17, 31, 33, 1000, 4099])
def test_small_and_ragged(ctx, dtype, n):
    R = 5
    ins = [host("normal", dtype, 9, r, n) for r in range(R)]
    L = P.pl_layout_partitioned(R, synth.equal_lengths(n, R))
    got = run(ctx, L, L, "sum", dtype, ins, [n] * R, None)
    want = oracle.allreduce(ins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")
    lens = [(n * (r + 1)) % 13 for r in range(R)]
    gins = [host("normal", dtype, 10, r, lens[r]) for r in range(R)]
    got = run(ctx, P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy", dtype, gins,
              [sum(lens)] * R, None)
    want = oracle.allgather(gins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


@pytest.mark.parametrize("shift", [1, 2, 3, 5, 7])
def test_misaligned_buffers(ctx, shift):
    """Sources and destinations at every misalignment mod 16 bytes (bf16 element offsets)."""
    R, n, dtype = 4, 3001, "bf16"
    ins = [host("normal", dtype, 11, r, n) for r in range(R)]
    big = [to_dev(np.concatenate([np.zeros(shift * (r + 1), np.uint16), a]), dtype) for r, a in enumerate(ins)]
    views = [b[shift * (r + 1):] for r, b in enumerate(big)]
    outs = Outs([n + shift] * R, dtype)
    ovs = [v[shift:] for v in outs.views]
    L = P.pl_layout_partitioned(R, synth.equal_lengths(n, R))
    s = P.stream_handle()
    P.pl_collective(ctx, L, L, "sum", dtype, R, P.ptrs(views), P.counts(views), P.ptrs(ovs), P.counts(ovs), None, s)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    outs.check_guards()
    want = oracle.allreduce(ins, dtype)
    for r in range(R):
        assert_equal(to_np(ovs[r], dtype), want[r], f"rank {r}")


def test_single_rank_is_a_copy(ctx):
    for dtype in ("bf16", "fp32"):
        x = host("normal", dtype, 12, 0, 777)
        L = P.pl_layout_rank_owned(1, [777])
        for op in ("copy", "sum"):
            got = run(ctx, L, L, op, dtype, [x], [777], None)
            assert_equal(got[0], x)


def test_sixty_four_ranks(ctx):
    R, n, dtype = 64, 640, "bf16"
    ins = [host("normal", dtype, 13, r, n) for r in range(R)]
    L = P.pl_layout_partitioned(R, [10] * R)
    got = run(ctx, L, L, "sum", dtype, ins, [n] * R, None)
    want = oracle.allreduce(ins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


def test_rounding_ties_and_order(ctx):
    """Constructed sums: exact ties in bf16 rounding, and fp32 sums whose value depends on the order."""
    # bf16: a + b where the fp32 sum lies exactly between two bf16 numbers.
    a = np.array([1.0078125, 1.0, -1.0078125, 2.0 ** -130, 3.0e38], np.float32)
    b = np.array([2.0 ** -8, 2.0 ** -8, -(2.0 ** -8), 2.0 ** -131, 3.0e38], np.float32)
    ins = [oracle.f32_to_bf16(a), oracle.f32_to_bf16(b)]
    L = P.pl_layout_partitioned(2, [3, 2])
    got = run(ctx, L, L, "sum", "bf16", ins, [5, 5], None)
    want = oracle.allreduce(ins, "bf16")
    assert_equal(got[0], want[0])
    # fp32: (2^24, 1, -2^24) sums to 0 only in rank order.
    x = [np.array([2.0 ** 24, -0.0], np.float32), np.array([1.0, -0.0], np.float32),
         np.array([-(2.0 ** 24), -0.0], np.float32)]
    L = P.pl_layout_partitioned(3, [1, 1, 0])
    got = run(ctx, L, L, "sum", "fp32", x, [2] * 3, None)
    assert got[0][0] == 0.0 and got[0][1].view(np.uint32) == 0x80000000


# ---------------------------------------------------------- boundary errors


def test_host_validation_errors(ctx):
    R, n = 2, 64
    a = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    L = P.pl_layout_partitioned(R, [32, 32])
    s = P.stream_handle()
    # output overlapping another output
    with pytest.raises(P.PurlinError) as e:
        P.pl_collective(ctx, L, L, "sum", "bf16", R, P.ptrs(a), [n] * R, [a[0].data_ptr()] * 2, [n] * R, None, s)
    assert e.value.status == P.PL_ERR_ALIAS
    # a part beyond its buffer
    with pytest.raises(P.PurlinError) as e:
        P.pl_collective(ctx, L, L, "sum", "bf16", R, P.ptrs(a), [n] * R, P.ptrs(a), [n - 1] * R, None, s)
    assert e.value.status == P.PL_ERR_LAYOUT
    # misaligned pointer (odd byte address for bf16)
    with pytest.raises(P.PurlinError) as e:
        P.pl_collective(ctx, L, L, "sum", "bf16", R, [p + 1 for p in P.ptrs(a)], [n] * R,
                        P.ptrs(a), [n] * R, None, s)
    assert e.value.status == P.PL_ERR_INVALID
    # an output partially overlapping an input
    b = torch.zeros(2 * n, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(P.PurlinError) as e:
        P.pl_collective(ctx, L, L, "sum", "bf16", R, [b.data_ptr(), a[1].data_ptr()], [n] * R,
                        [b.data_ptr() + 2, a[0].data_ptr()], [n] * R, None, s)
    assert e.value.status == P.PL_ERR_ALIAS


def test_allreduce_in_place(ctx):
    R, n, dtype = 8, 100003, "bf16"
    ins = [host("normal", dtype, 14, r, n) for r in range(R)]
    want = oracle.allreduce(ins, dtype)
    for name, pol in ar_policies().items():
        bufs = [to_dev(a, dtype) for a in ins]
        s = P.stream_handle()
        P.pl_allreduce(ctx, dtype, R, n, P.ptrs(bufs), P.ptrs(bufs), pol, s)
        assert P.pl_ctx_status(ctx, s) == P.PL_OK
        for r in range(R):
            assert_equal(to_np(bufs[r], dtype), want[r], f"{name} rank {r}")


def test_repeated_calls_reuse_plans_and_flags(ctx):
    """Back-to-back launches of flagged plans (new epoch each) stay correct."""
    R, n, dtype = 8, 1 << 16, "bf16"
    ins = [host("normal", dtype, 15, r, n) for r in range(R)]
    dev = [to_dev(a, dtype) for a in ins]
    want = oracle.allreduce(ins, dtype)
    outs = [torch.empty_like(d) for d in dev]
    s = P.stream_handle()
    before = P.pl_ctx_launches(ctx)
    for i in range(6):
        pols = list(ar_policies().values())
        pol = pols[i % len(pols)]
        P.pl_allreduce(ctx, dtype, R, n, P.ptrs(dev), P.ptrs(outs), pol, s)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    assert P.pl_ctx_launches(ctx) - before == 6
    for r in range(R):
        assert_equal(to_np(outs[r], dtype), want[r], f"rank {r}")


def test_dropped_notify_times_out_and_recovers(ctx):
    """A Notify that never happens: consumers' bounded waits expire, the status
    word reports PL_ERR_TIMEOUT, the kernel returns, and the next call works."""
    R, n, dtype = 4, 4096, "bf16"
    ins = [host("normal", dtype, 16, r, n) for r in range(R)]
    dev = [to_dev(a, dtype) for a in ins]
    outs = [torch.empty_like(d) for d in dev]
    s = P.stream_handle()
    pol = P.pl_policy_default(path=P.PL_PATH_STAGED, chunk_bytes=2048, poll_timeout_ns=50_000_000,
                              debug_drop_notify=0)
    P.pl_allreduce(ctx, dtype, R, n, P.ptrs(dev), P.ptrs(outs), pol, s)
    assert P.pl_ctx_status(ctx, s) == P.PL_ERR_TIMEOUT
    P.pl_allreduce(ctx, dtype, R, n, P.ptrs(dev), P.ptrs(outs), P.pl_policy_default(path=P.PL_PATH_STAGED), s)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    want = oracle.allreduce(ins, dtype)
    for r in range(R):
        assert_equal(to_np(outs[r], dtype), want[r], f"rank {r}")


# ------------------------------------------------- bulk-copy ring datapath


@pytest.mark.parametrize("stages", [1, 2, 3, 4, 8])
def test_bulk_ring_datapath(ctx, stages):
    """The cp.async.bulk shared-memory ring (1..8 stages) on aligned copies; the
    unaligned V forms and strided rows fall back to the vector path."""
    R, dtype = 8, "bf16"
    pol = P.pl_policy_default(datapath=P.PL_ATOM_BULK, stages=stages)
    n = (1 << 20) // 2 // R + 8  # a piece count that does not divide evenly
    ins = [host("normal", dtype, 17, r, n) for r in range(R)]
    got = run(ctx, P.pl_layout_rank_owned(R, [n] * R), P.pl_layout_partitioned(R, [n] * R), "copy", dtype, ins,
              [n * R] * R, pol)
    want = oracle.allgather(ins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"AG rank {r}")
    m = [[(n // R) + 3 * ((r + j) % 2) for j in range(R)] for r in range(R)]
    ains = [host("normal", dtype, 18, r, sum(m[r])) for r in range(R)]
    outn = [sum(m[r][j] for r in range(R)) for j in range(R)]
    got = run(ctx, P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m), "copy", dtype, ains, outn, pol)
    want = oracle.alltoall(ains, m, dtype)
    for j in range(R):
        assert_equal(got[j], want[j], f"A2A rank {j}")
    S, H, D = 64, 32, 128
    uins = [host("normal", dtype, 19, r, S * H * D) for r in range(R)]
    got = run(ctx, P.pl_layout_ulysses_in(R, S, H, D), P.pl_layout_ulysses_out(R, S, H, D), "copy", dtype, uins,
              [S * H * D] * R, pol)
    want = oracle.ulysses_a2a(uins, S, H, D, dtype)
    for j in range(R):
        assert_equal(got[j], want[j], f"Ulysses rank {j}")


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("stages", [0, 4, 6, 8])
def test_bulk_shift_copy(ctx, dtype, stages):
    """Copies whose source sits at a byte shift from the (aligned) destinations
    through the bulk ring: bulk load, realignment in shared memory, bulk stores.
    AllGatherV with Zipf lengths (every shift, odd ones for one-byte elements),
    ragged last pieces; stages = 0 is the automatic policy (chosen for
    write-heavy copies of 64 MiB or more)."""
    R = 8
    pol = P.pl_policy_default(datapath=P.PL_ATOM_AUTO if stages == 0 else P.PL_ATOM_BULK, stages=stages)
    N = (8 << 20) // (1 if dtype == "fp8" else 2) + 13  # 8 MiB per output: 72 MiB moved
    lens = synth.zipf_lengths(N, R, 0.125, seed=50 + stages)
    ins = [host(None if dtype == "fp8" else "normal", dtype, 50, r, lens[r]) for r in range(R)]
    got = run(ctx, P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy", dtype, ins,
              [N] * R, pol)
    want = oracle.allgather(ins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"AGV rank {r}")


@pytest.mark.parametrize("form", [P.PL_AR_FUSED, P.PL_AR_COMPOSED, P.PL_AR_NOTIFIED])
def test_bulk_ring_in_flagged_paths(ctx, form):
    """Bulk copies inside staged and composed plans (stage, gather) with flags."""
    R, n, dtype = 8, 1 << 18, "bf16"
    ins = [host("normal", dtype, 20, r, n) for r in range(R)]
    want = oracle.allreduce(ins, dtype)
    for path in (P.PL_PATH_ZS, P.PL_PATH_STAGED):
        pol = P.pl_policy_default(datapath=P.PL_ATOM_BULK, stages=4, path=path, allreduce_form=form,
                                  chunk_bytes=64 << 10)
        dev = [to_dev(a, dtype) for a in ins]
        outs = Outs([n] * R, dtype)
        s = P.stream_handle()
        P.pl_allreduce(ctx, dtype, R, n, P.ptrs(dev), outs.ptrs(), pol, s)
        assert P.pl_ctx_status(ctx, s) == P.PL_OK
        outs.check_guards()
        for r in range(R):
            assert_equal(outs.host(r), want[r], f"path {path} rank {r}")


# ---------------------------------------------------- forced small grids


@pytest.mark.parametrize("ctas", [8, 16, 32])
@pytest.mark.parametrize("datapath,stages", [("vector", 0), ("bulk", 1), ("bulk", 8)])
def test_forced_small_grids(ctx, ctas, datapath, stages):
    """The grids and ring depths the depth x CTA sweep times: a few CTAs each
    run many items in a row, so the bulk ring carries on from item to item
    (aligned copies, copies realigned in shared memory and vector items in one
    CTA), and reductions and copies share the claim order.  AllGatherV with
    Zipf lengths (bf16 and one-byte elements), AllToAllV, ReduceScatterV and
    AllReduce, each against the oracle."""
    R = 8
    pol = P.pl_policy_default(datapath=P.PL_ATOM_VECTOR if datapath == "vector" else P.PL_ATOM_BULK,
                              stages=stages, ctas=ctas)
    small = P.pl_policy_default(datapath=pol.datapath, stages=stages, ctas=ctas, chunk_bytes=16384)
    for dtype, S in (("bf16", 2), ("fp8", 1)):
        N = (4 << 20) // S + 13
        lens = synth.zipf_lengths(N, R, 0.125, seed=60 + ctas)
        ins = [host(None if dtype == "fp8" else "normal", dtype, 60, r, lens[r]) for r in range(R)]
        want = oracle.allgather(ins, dtype)
        for p in (pol, small):
            got = run(ctx, P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy", dtype, ins,
                      [N] * R, p)
            for r in range(R):
                assert_equal(got[r], want[r], f"AGV {dtype} rank {r}")
    dtype = "bf16"
    N = (1 << 20) + 7
    m = synth.zipf_matrix(N, R, 0.125, seed=61)
    ains = [host("normal", dtype, 61, r, sum(m[r])) for r in range(R)]
    outn = [sum(m[r][j] for r in range(R)) for j in range(R)]
    want = oracle.alltoall(ains, m, dtype)
    got = run(ctx, P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m), "copy", dtype, ains, outn, pol)
    for j in range(R):
        assert_equal(got[j], want[j], f"A2AV rank {j}")
    lens = synth.zipf_lengths(N, R, 0.125, seed=62)
    rins = [host("normal", dtype, 62, r, N) for r in range(R)]
    want = oracle.reducescatter(rins, lens, dtype)
    got = run(ctx, P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned(R, lens), "sum", dtype, rins, lens, pol)
    for k in range(R):
        assert_equal(got[k], want[k], f"RSV rank {k}")
    L = P.pl_layout_partitioned(R, synth.equal_lengths(N, R))
    want = oracle.allreduce(rins, dtype)
    got = run(ctx, L, L, "sum", dtype, rins, [N] * R, pol)
    for r in range(R):
        assert_equal(got[r], want[r], f"AR rank {r}")
