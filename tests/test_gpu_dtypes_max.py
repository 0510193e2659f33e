"""GPU parity of the further element types and the maximum reduction, through
the C ABI against the CPU oracle, bit for bit:

* fp16 (IEEE binary16): sums accumulate in fp32 in rank order and round once;
* fp8 (any one-byte element): copies only, at every byte misalignment;
* PL_MAX: the rank-ordered maximum (rank r's element replaces the running
  value only when it compares greater), for bf16, fp16 and fp32, on every
  path and AllReduce form.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from copy_reduce_datapath_gb300 import purlin as P

from gpu_util import NP, Outs, ar_policies, assert_equal, bits, host, policies, run, to_dev, to_np

pytestmark = pytest.mark.gpu

SCRATCH = 64 << 20


@pytest.fixture(scope="module")
def ctx():
    torch.cuda.set_device(0)
    c = P.pl_ctx_create(0, SCRATCH)
    yield c
    P.pl_ctx_destroy(c)


# ------------------------------------------------------------------ fp16


@pytest.mark.parametrize("T", [1 << 10, 1 << 16, (1 << 21) + 6])
@pytest.mark.parametrize("name", list(ar_policies()))
def test_allreduce_fp16(ctx, T, name):
    R = 8
    n = T // 2
    ins = [host("normal", "fp16", 20, r, n) for r in range(R)]
    L = P.pl_layout_partitioned(R, synth.equal_lengths(n, R))
    got = run(ctx, L, L, "sum", "fp16", ins, [n] * R, ar_policies()[name])
    want = oracle.allreduce(ins, "fp16")
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


@pytest.mark.parametrize("name", list(policies()))
def test_v_collectives_fp16(ctx, name):
    """AllGatherV and ReduceScatterV with Zipf lengths: 2-byte offsets at every misalignment."""
    R, dtype, N = 8, "fp16", (1 << 19) + 3
    pol = policies()[name]
    lens = synth.zipf_lengths(N, R, 0.125, seed=21)
    ins = [host("normal", dtype, 21, r, lens[r]) for r in range(R)]
    got = run(ctx, P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy", dtype, ins,
              [N] * R, pol)
    want = oracle.allgather(ins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"AGV rank {r}")
    ins = [host("uniform", dtype, 22, r, N) for r in range(R)]
    got = run(ctx, P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned(R, lens), "sum", dtype, ins,
              lens, pol)
    want = oracle.reducescatter(ins, lens, dtype)
    for k in range(R):
        assert_equal(got[k], want[k], f"RSV rank {k}")


def test_fp16_rounding_overflow_and_subnormals(ctx):
    """Sums that round at a tie, overflow past 65504 to infinity, and land in
    the subnormal range, against the oracle's definition-based rounding."""
    a = np.array([1.0, 65504.0, 2.0 ** -24, -(2.0 ** -14), 2048.0, 1.0], np.float32)
    b = np.array([2.0 ** -11, 16.0, 2.0 ** -24, 2.0 ** -24, 1.0, -(2.0 ** -11)], np.float32)
    ins = [oracle.f32_to_f16(a), oracle.f32_to_f16(b)]
    L = P.pl_layout_partitioned(2, [3, 3])
    got = run(ctx, L, L, "sum", "fp16", ins, [6, 6], None)
    want = oracle.allreduce(ins, "fp16")
    for r in range(2):
        assert_equal(got[r], want[r], f"rank {r}")
    assert bits(got[0])[1] == 0x7C00  # 65504 + 16 rounds to infinity


# ------------------------------------------------------------------- fp8


@pytest.mark.parametrize("name", list(policies()))
def test_allgather_alltoall_fp8(ctx, name):
    """One-byte elements: AllGatherV and AllToAllV with Zipf lengths (byte
    offsets at every misalignment mod 16) and the equal MoE-shaped AllToAll."""
    R, dtype, N = 8, "fp8", (1 << 20) + 5
    pol = policies()[name]
    lens = synth.zipf_lengths(N, R, 0.125, seed=23)
    ins = [host(None, dtype, 23, r, lens[r]) for r in range(R)]
    got = run(ctx, P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy", dtype, ins,
              [N] * R, pol)
    want = oracle.allgather(ins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"AGV rank {r}")
    m = synth.zipf_matrix(N // R, R, 0.125, seed=24)
    ins = [host(None, dtype, 24, r, sum(m[r])) for r in range(R)]
    outn = [sum(m[r][j] for r in range(R)) for j in range(R)]
    got = run(ctx, P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m), "copy", dtype, ins, outn, pol)
    want = oracle.alltoall(ins, m, dtype)
    for j in range(R):
        assert_equal(got[j], want[j], f"A2AV rank {j}")
    m = [[4096] * R for _ in range(R)]
    ins = [host(None, dtype, 25, r, sum(m[r])) for r in range(R)]
    got = run(ctx, P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m), "copy", dtype, ins,
              [R * 4096] * R, pol)
    want = oracle.alltoall(ins, m, dtype)
    for j in range(R):
        assert_equal(got[j], want[j], f"A2A rank {j}")


@pytest.mark.parametrize("name", ["zs", "staged"])
def test_ulysses_fp8(ctx, name):
    """Strided rows of one-byte elements (D = 24 bytes per head row: rows not
    16-byte multiples, so the row path rather than the flat path)."""
    R, S, H, D, dtype = 4, 96, 8, 24, "fp8"
    ins = [host(None, dtype, 26, r, S * H * D) for r in range(R)]
    got = run(ctx, P.pl_layout_ulysses_in(R, S, H, D), P.pl_layout_ulysses_out(R, S, H, D), "copy", dtype, ins,
              [S * H * D] * R, policies()[name])
    want = oracle.ulysses_a2a(ins, S, H, D, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


@pytest.mark.parametrize("shift", [1, 3, 7, 8, 15])
def test_fp8_misaligned_buffers(ctx, shift):
    """Source and destination buffers at odd byte addresses (the splicing
    copy path with a byte shift that is not a multiple of 2)."""
    R, n, dtype = 4, 70001, "fp8"
    ins = [host(None, dtype, 27, r, n) for r in range(R)]
    big = [to_dev(np.concatenate([np.zeros(shift * (r + 1), np.uint8), a]), dtype) for r, a in enumerate(ins)]
    views = [b[shift * (r + 1):] for r, b in enumerate(big)]
    outs = Outs([R * n + shift] * R, dtype)
    ovs = [v[shift:] for v in outs.views]
    s = P.stream_handle()
    P.pl_collective(ctx, P.pl_layout_rank_owned(R, [n] * R), P.pl_layout_partitioned(R, [n] * R), "copy", dtype,
                    R, P.ptrs(views), P.counts(views), P.ptrs(ovs), P.counts(ovs), None, s)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    outs.check_guards()
    want = oracle.allgather(ins, dtype)
    for r in range(R):
        assert_equal(to_np(ovs[r], dtype), want[r], f"rank {r}")


@pytest.mark.parametrize("n", [0, 1, 2, 15, 16, 17, 31, 33, 1000, 4099])
def test_fp8_small_and_ragged(ctx, n):
    R, dtype = 5, "fp8"
    lens = [(n * (r + 1)) % 29 for r in range(R)]
    ins = [host(None, dtype, 28, r, lens[r]) for r in range(R)]
    got = run(ctx, P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy", dtype, ins,
              [sum(lens)] * R, None)
    want = oracle.allgather(ins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


def test_fp8_bulk_ring(ctx):
    """The cp.async.bulk ring datapath moves one-byte elements too."""
    R, n, dtype = 8, 1 << 20, "fp8"
    ins = [host(None, dtype, 29, r, n) for r in range(R)]
    pol = P.pl_policy_default(datapath=P.PL_ATOM_BULK, stages=4)
    got = run(ctx, P.pl_layout_rank_owned(R, [n] * R), P.pl_layout_partitioned(R, [n] * R), "copy", dtype, ins,
              [R * n] * R, pol)
    want = oracle.allgather(ins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


def test_fp8_reductions_are_refused(ctx):
    R, n = 2, 64
    ins = [torch.zeros(n, dtype=torch.uint8, device="cuda") for _ in range(R)]
    outs = [torch.zeros(n, dtype=torch.uint8, device="cuda") for _ in range(R)]
    L = P.pl_layout_partitioned(R, [32, 32])
    for op in ("sum", "max"):
        with pytest.raises(P.PurlinError) as e:
            P.pl_collective(ctx, L, L, op, "fp8", R, P.ptrs(ins), P.counts(ins), P.ptrs(outs), P.counts(outs))
        assert e.value.status == P.PL_ERR_UNSUPPORTED
    with pytest.raises(P.PurlinError) as e:
        P.pl_allreduce_op(ctx, "max", "fp8", R, n, P.ptrs(ins), P.ptrs(outs))
    assert e.value.status == P.PL_ERR_UNSUPPORTED


# ------------------------------------------------------------------- max


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("name", list(ar_policies()))
def test_allreduce_max(ctx, dtype, name):
    R, n = 8, (1 << 17) + 3
    ins = [host("normal", dtype, 30, r, n) for r in range(R)]
    outs = Outs([n] * R, dtype)
    dins = [to_dev(a, dtype) for a in ins]
    s = P.stream_handle()
    P.pl_allreduce_op(ctx, "max", dtype, R, n, P.ptrs(dins), outs.ptrs(), ar_policies()[name], s)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    outs.check_guards()
    want = oracle.allreduce(ins, dtype, op="max")
    for r in range(R):
        assert_equal(outs.host(r), want[r], f"rank {r}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("name", list(policies()))
def test_reducescatter_v_max(ctx, dtype, name):
    """Zipf partitions: sources at mixed misalignments (the spliced and the
    one-source-at-a-time reduction paths)."""
    R, N = 8, (1 << 19) + 1
    lens = synth.zipf_lengths(N, R, 0.125, seed=31)
    ins = [host("uniform", dtype, 31, r, N) for r in range(R)]
    got = run(ctx, P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned(R, lens), "max", dtype, ins, lens,
              policies()[name])
    want = oracle.reducescatter(ins, lens, dtype, op="max")
    for k in range(R):
        assert_equal(got[k], want[k], f"rank {k}")


@pytest.mark.parametrize("R", [2, 3, 64])
def test_max_rank_counts(ctx, R):
    n = 64 * 40 + 7
    ins = [host("int8range", "bf16", 32, r, n) for r in range(R)]  # many equal values: ties everywhere
    L = P.pl_layout_partitioned(R, synth.equal_lengths(n, R))
    got = run(ctx, L, L, "max", "bf16", ins, [n] * R, None)
    want = oracle.allreduce(ins, "bf16", op="max")
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_max_special_values(ctx, dtype):
    """Signed zeros keep the earlier rank's sign; infinities win or lose as
    numbers; a NaN counts only from rank 0.  Bit patterns are compared except
    for NaN results, whose payload a conversion may canonicalise: there only
    NaN-ness is required."""
    nan, inf = np.float32("nan"), np.float32("inf")
    cols = [  # rank 0, rank 1, rank 2
        (0.0, -0.0, 0.0), (-0.0, 0.0, -0.0), (-inf, -1.0, -inf), (1.0, inf, 2.0),
        (nan, 5.0, 7.0), (1.0, nan, 0.5), (-3.0, nan, -1.0), (-inf, -inf, -inf), (0.0, 0.0, 1e-30),
    ]
    f32 = [np.array([c[r] for c in cols], np.float32) for r in range(3)]
    conv = {"bf16": oracle.f32_to_bf16, "fp16": oracle.f32_to_f16, "fp32": lambda a: a}[dtype]
    ins = [conv(a) for a in f32]
    n = len(cols)
    L = P.pl_layout_partitioned(3, [n, 0, 0])
    got = run(ctx, L, L, "max", dtype, ins, [n] * 3, None)
    want = oracle.allreduce(ins, dtype, op="max")
    wf = [np.asarray(w) for w in want]
    for r in range(3):
        g, w = got[r], wf[r]
        if dtype == "fp32":
            gnan, wnan = np.isnan(g), np.isnan(w)
        else:
            gf = oracle.f16_to_f32(g) if dtype == "fp16" else oracle.bf16_to_f32(g)
            wf32 = oracle.f16_to_f32(w) if dtype == "fp16" else oracle.bf16_to_f32(w)
            gnan, wnan = np.isnan(gf), np.isnan(wf32)
        assert np.array_equal(gnan, wnan), f"rank {r}: NaN positions"
        assert gnan[4] and not gnan[5] and not gnan[6]
        keep = ~wnan
        assert_equal(g[keep], w[keep], f"rank {r}")


# -------------------------------------------------- sums of special values


def _nan_mask(a, dtype):
    if dtype == "fp32":
        return np.isnan(a)
    f = oracle.f16_to_f32(a) if dtype == "fp16" else oracle.bf16_to_f32(a)
    return np.isnan(f)


@pytest.mark.parametrize("R", [3, 8])
@pytest.mark.parametrize("pol", ["zs", "zs_small_chunks", "staged"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_sum_special_values(ctx, dtype, pol, R):
    """The rank-ordered fp32 sum on NaN inputs, inf + (-inf), infinities and
    sums that overflow: in the fp32 accumulation, or only at the final
    rounding to bf16 / fp16 (a finite fp32 sum at or beyond the type's
    rounding boundary to infinity).  NaN results are compared by position
    only (the payload of a NaN produced by an addition or by a conversion is
    not unique); every other element bit for bit.  Columns are tiled to
    thousands of elements so that every launch form runs them."""
    nan, inf = np.float32("nan"), np.float32("inf")
    big = {"bf16": (np.float32(2.0 ** 127 * (2 - 2 ** -7)), np.float32(2.0 ** 119)),  # bf16 max + half an ulp
           "fp16": (np.float32(65504.0), np.float32(16.0)),                           # fp16 max + half an ulp
           "fp32": (np.float32(3e38), np.float32(3e38))}[dtype]
    cols = [  # values of ranks 0, 1, 2; ranks 3.. add zeros
        (nan, 1.0, 2.0), (1.0, nan, 2.0), (1.0, 2.0, nan), (inf, -inf, 0.0), (-inf, 1.0, inf),
        (inf, 1.0, 2.0), (-inf, -inf, 1.0), (big[0], big[1], 0.0), (-big[0], -big[1], 0.0),
        (1.0, 2.0, 3.0), (-0.0, -0.0, -0.0),
    ]
    reps = 1500
    f32 = [np.tile(np.array([c[r] if r < 3 else 0.0 for c in cols], np.float32), reps) for r in range(R)]
    if R > 3:  # a -0 column stays -0 only if every rank adds -0
        for r in range(3, R):
            f32[r][10::len(cols)] = -0.0
    conv = {"bf16": oracle.f32_to_bf16, "fp16": oracle.f32_to_f16, "fp32": lambda a: a}[dtype]
    ins = [conv(a) for a in f32]
    n = ins[0].size
    L = P.pl_layout_partitioned(R, synth.equal_lengths(n, R))
    got = run(ctx, L, L, "sum", dtype, ins, [n] * R, policies()[pol])
    want = oracle.allreduce(ins, dtype)
    nan_cols = np.zeros(len(cols), bool)
    nan_cols[[0, 1, 2, 3, 4]] = True
    expect_nan = np.tile(nan_cols, reps)
    for r in range(R):
        g, w = got[r], np.asarray(want[r])
        gnan, wnan = _nan_mask(g, dtype), _nan_mask(w, dtype)
        assert np.array_equal(wnan, expect_nan), "oracle: NaN positions"
        assert np.array_equal(gnan, wnan), f"rank {r}: NaN positions"
        keep = ~wnan
        assert_equal(g[keep], w[keep], f"rank {r}")
    # the overflow columns are infinite with the sign of their inputs
    wf = np.asarray(want[0]).astype(np.float32) if dtype == "fp32" else \
        (oracle.f16_to_f32 if dtype == "fp16" else oracle.bf16_to_f32)(np.asarray(want[0]))
    assert np.isposinf(wf[7]) and np.isneginf(wf[8])
