"""GPU parity of the composed AllReduce of Figure 6 against the oracle, bit for
bit: PL_AR_COMPOSED, which composes at the grain of one vector in the
kernels for aligned plans (the reduced vector is stored to the owner's
output, read back from there and written to the other ranks) and per item in
the realigning kernels (outputs off 16-byte alignment), and PL_AR_NOTIFIED,
the per-chunk form with a Notify between the owner's reduce and the gather.
Cases: sum and maximum, bf16 / fp16 / fp32, equal partitions and a ragged
last partition, in place, multi-row (strided) partitions, and the 1 GiB
AllReduce of the benchmark in the composed form (windows against the oracle).
"""
import numpy as np
import pytest
import torch

import bench
import oracle
from copy_reduce_datapath_gb300 import purlin as P

from gpu_util import Outs, aligned_guard, assert_equal, host, run, to_dev, to_np

pytestmark = pytest.mark.gpu

FORMS = {"composed": P.PL_AR_COMPOSED, "notified": P.PL_AR_NOTIFIED}
ELEMS16 = {"bf16": 8, "fp16": 8, "fp32": 4}  # elements per 16-byte vector


@pytest.fixture(scope="module")
def ctx():
    torch.cuda.set_device(0)
    c = P.pl_ctx_create(0, 0)
    yield c
    P.pl_ctx_destroy(c)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("op", ["sum", "max"])
@pytest.mark.parametrize("form", list(FORMS))
@pytest.mark.parametrize("shape", ["equal", "ragged_tail"])
def test_composed_allreduce(ctx, dtype, op, form, shape):
    """R = 8 partitions at 16-byte aligned offsets (equal, or the last one a
    few elements longer, so its last vector is moved element by element);
    outputs aligned and misaligned (the helper runs both)."""
    R, E = 8, ELEMS16[dtype]
    lens = [E * 4099] * R if shape == "equal" else [E * 1024] * (R - 1) + [E * 1024 + 5]
    n = sum(lens)
    ins = [host("normal", dtype, 80, r, n) for r in range(R)]
    L = P.pl_layout_partitioned(R, lens)
    got = run(ctx, L, L, op, dtype, ins, [n] * R, P.pl_policy_default(allreduce_form=FORMS[form]))
    want = oracle.allreduce(ins, dtype, op=op)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("n", [8 * 8192, 8 * 8192 + 13])
@pytest.mark.parametrize("form", list(FORMS))
def test_composed_allreduce_in_place(ctx, dtype, n, form):
    """Outputs equal to the inputs: with n = 8 x 8192 every partition is
    16-byte aligned (the vector-grain composition, each vector read whole by
    its thread before it is written anywhere); with 13 more elements the
    partitions are not (the per-item composition)."""
    R = 8
    ins = [host("normal", dtype, 81, r, n) for r in range(R)]
    want = oracle.allreduce(ins, dtype)
    bufs = [to_dev(a, dtype) for a in ins]
    s = P.stream_handle()
    P.pl_allreduce(ctx, dtype, R, n, P.ptrs(bufs), P.ptrs(bufs), P.pl_policy_default(allreduce_form=FORMS[form]), s)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    for r in range(R):
        assert_equal(to_np(bufs[r], dtype), want[r], f"rank {r}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("form", list(FORMS))
def test_composed_allreduce_multi_row(ctx, dtype, form):
    """Each rank's input is rows x (R x cols) row-major and partition k is
    column block k (rows of cols elements, stride R x cols); every rank's
    output holds the reduced blocks one after another: multi-row items with
    strided sources (the flat two-dimensional body composes per vector when
    aligned)."""
    R, rows, cols = 4, 96, 64
    lin_parts = [[(k, k * cols, cols, rows, R * cols) for k in range(R)]] * R
    lout_parts = [[(k, k * rows * cols, rows * cols) for k in range(R)]] * R
    lin, lout = P.pl_layout_create(R, lin_parts), P.pl_layout_create(R, lout_parts)
    n = rows * R * cols
    ins = [host("normal", dtype, 82, r, n) for r in range(R)]
    got = run(ctx, lin, lout, "sum", dtype, ins, [n] * R, P.pl_policy_default(allreduce_form=FORMS[form]))
    want = oracle.collective("sum", dtype, lin_parts, lout_parts, ins, [n] * R)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")


def test_composed_allreduce_ctas_and_small_chunks(ctx):
    """The vector-grain form with forced grids and chunk sizes: items in a
    row on few CTAs, and chunks of a few vectors per thread."""
    R, dtype, n = 8, "bf16", 8 * 8 * 3001
    ins = [host("normal", dtype, 83, r, n) for r in range(R)]
    want = oracle.allreduce(ins, dtype)
    dev = [to_dev(a, dtype) for a in ins]
    s = P.stream_handle()
    for ctas, chunk in ((1, 0), (8, 4096), (32, 256), (0, 1 << 20)):
        outs = Outs([n] * R, dtype, aligned_guard(dtype))
        pol = P.pl_policy_default(allreduce_form=P.PL_AR_COMPOSED, ctas=ctas, chunk_bytes=chunk)
        P.pl_allreduce(ctx, dtype, R, n, P.ptrs(dev), outs.ptrs(), pol, s)
        assert P.pl_ctx_status(ctx, s) == P.PL_OK
        outs.check_guards()
        for r in range(R):
            assert_equal(outs.host(r), want[r], f"ctas {ctas} chunk {chunk} rank {r}")


def test_composed_allreduce_1GiB(ctx):
    """The benchmark's AllReduce (R = 8, bf16, 1 GiB per rank) in the composed
    form: windows of the outputs against the oracle, every rank's output
    identical over the whole buffer."""
    W = 4096
    wl = bench.Workload(1 << 30, torch.device("cuda:0"))
    s = torch.cuda.current_stream().cuda_stream
    try:
        P.pl_allreduce(ctx, "bf16", 8, wl.n_ar, P.ptrs(wl.ar_in), P.ptrs(wl.ar_out),
                       P.pl_policy_default(allreduce_form=P.PL_AR_COMPOSED), s)
        assert P.pl_ctx_status(ctx, s) == P.PL_OK
        part = wl.n_ar // 8
        rng = np.random.default_rng(5)
        starts = {int(x) for x in rng.integers(0, wl.n_ar - W, 6)}
        starts |= {k * part - W // 2 for k in range(1, 8)} | {wl.n_ar - W}
        for i in sorted(starts):
            want = oracle.allreduce([to_np(x[i:i + W], "bf16") for x in wl.ar_in], "bf16")[0]
            for r in (0, 3, 7):
                assert_equal(to_np(wl.ar_out[r][i:i + W], "bf16"), want, f"rank {r} window {i}")
        for r in range(1, 8):
            assert torch.equal(wl.ar_out[r].view(torch.int16), wl.ar_out[0].view(torch.int16)), f"rank {r}"
    finally:
        del wl
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


@pytest.mark.parametrize("form", list(FORMS))
def test_composed_allreduce_64_ranks(ctx, form):
    """R = 64, the most sources and destinations an item holds: the owner first
    among 64 destinations, outputs aligned and misaligned."""
    R, dtype = 64, "bf16"
    lens = [8 * 37] * R
    n = sum(lens)
    ins = [host("normal", dtype, 84, r, n) for r in range(R)]
    L = P.pl_layout_partitioned(R, lens)
    got = run(ctx, L, L, "sum", dtype, ins, [n] * R, P.pl_policy_default(allreduce_form=FORMS[form]))
    want = oracle.allreduce(ins, dtype)
    for r in range(R):
        assert_equal(got[r], want[r], f"rank {r}")
