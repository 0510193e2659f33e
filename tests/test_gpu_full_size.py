"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (automatic policy, one launch per collective).  The oracle
cannot run a 1 GiB collective in a test's time, so each check takes windows
of the outputs the oracle computes from the matching input windows (random
offsets plus every partition boundary and the last elements), and, for the
copies, the exact property that every output block equals its source block,
compared on the device over the whole buffers.

Workloads (seeded, synthetic):
  * AllGather and AllReduce, R = 8, bf16 ~ N(0,1), T = 1 GiB each (seed 1);
  * ReduceScatter, R = 8, fp32 and bf16 ~ U(-1,1), T = 1 GiB, also in place (seed 2);
  * MoE-dispatch AllToAll (4096 x 7168 bf16 per rank) and the Ulysses
    sequence-to-head swap (16384 x 32 x 128 bf16 per rank), R = 8 (seed 3);
  * AllGatherV, ReduceScatterV, AllToAllV with Zipf(s = 0.125) lengths,
    R = 8, bf16, T = 1 GiB (seed 4).
"""
import numpy as np
import pytest
import torch

import bench
import oracle
import synth
from copy_reduce_datapath_gb300 import purlin as P

from gpu_util import assert_equal, to_np

pytestmark = pytest.mark.gpu

R = 8
GiB = 1 << 30
W = 4096  # elements per window


@pytest.fixture(scope="module")
def ctx():
    torch.cuda.set_device(0)
    c = P.pl_ctx_create(0, 0)
    yield c
    P.pl_ctx_destroy(c)


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def windows(n, boundaries=(), count=6, seed=0, w=W):
    """Start offsets of windows of w elements in [0, n): random ones, one
    straddling each boundary, and the last w elements."""
    rng = np.random.default_rng(seed)
    starts = [int(x) for x in rng.integers(0, max(1, n - w), count)]
    starts += [min(max(0, b - w // 2), n - w) for b in boundaries]
    starts.append(max(0, n - w))
    return sorted(set(starts))


def h(t, dtype):
    return to_np(t, dtype)


def status_ok(ctx):
    s = torch.cuda.current_stream().cuda_stream
    assert P.pl_ctx_status(ctx, s) == P.PL_OK


def test_allgather_allreduce_1GiB(ctx):
    dev = torch.device("cuda:0")
    wl = bench.Workload(GiB, dev)
    s = torch.cuda.current_stream().cuda_stream
    wl.allgather(ctx, s)
    wl.allreduce(ctx, s)
    status_ok(ctx)
    # AllGather: every output is the concatenation of the inputs.
    cat = torch.cat(wl.ag_in)
    for r in range(R):
        assert torch.equal(wl.ag_out[r].view(torch.int16), cat.view(torch.int16)), f"AllGather rank {r}"
    del cat
    mid = R // 2
    for i in windows(wl.n_ag, seed=1):
        want = oracle.allgather([h(x[i:i + W], "bf16") for x in wl.ag_in], "bf16")[0]
        got = np.concatenate([h(wl.ag_out[R - 1][q * wl.n_ag + i:q * wl.n_ag + i + W], "bf16") for q in range(R)])
        assert_equal(got, want, f"AllGather window {i}")
    # AllReduce: windows against the oracle; every rank's output identical.
    part = wl.n_ar // R
    for i in windows(wl.n_ar, boundaries=[k * part for k in range(1, R)], seed=2):
        want = oracle.allreduce([h(x[i:i + W], "bf16") for x in wl.ar_in], "bf16")[0]
        for r in (0, mid, R - 1):
            assert_equal(h(wl.ar_out[r][i:i + W], "bf16"), want, f"AllReduce rank {r} window {i}")
    for r in range(1, R):
        assert torch.equal(wl.ar_out[r].view(torch.int16), wl.ar_out[0].view(torch.int16)), f"AllReduce rank {r}"


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("in_place", [False, True])
def test_reducescatter_1GiB(ctx, dtype, in_place):
    dev = torch.device("cuda:0")
    tdt = torch.float32 if dtype == "fp32" else torch.bfloat16
    S = 4 if dtype == "fp32" else 2
    N = GiB // S
    lens = [N // R] * R
    ins = [synth.device_uniform_pm1(2, r, N, dev, tdt) for r in range(R)]
    offs = [k * (N // R) for k in range(R)]
    # input windows first: the in-place variant overwrites them
    wins = {k: windows(lens[k], seed=10 + k, count=2) for k in range(R)}
    want = {}
    for k in range(R):
        for i in wins[k]:
            want[k, i] = oracle.allreduce([h(x[offs[k] + i:offs[k] + i + W], dtype) for x in ins], dtype)[0]
    lin = P.pl_layout_partitioned(R, lens)
    if in_place:
        outs, lout = ins, P.pl_layout_rank_owned_inplace(R, lens)
    else:
        outs, lout = [torch.empty(lens[k], dtype=tdt, device=dev) for k in range(R)], P.pl_layout_rank_owned(R, lens)
    s = torch.cuda.current_stream().cuda_stream
    P.pl_collective(ctx, lin, lout, "sum", dtype, R, P.ptrs(ins), P.counts(ins), P.ptrs(outs), P.counts(outs),
                    None, s)
    status_ok(ctx)
    for (k, i), w in want.items():
        base = offs[k] if in_place else 0
        assert_equal(h(outs[k][base + i:base + i + W], dtype), w, f"rank {k} window {i}")


def test_alltoall_moe_and_ulysses(ctx):
    dev = torch.device("cuda:0")
    # MoE dispatch: 4096 tokens x 7168 hidden per rank, 8 equal token partitions.
    n = 4096 * 7168
    part = n // R
    m = [[part] * R for _ in range(R)]
    ins = [synth.device_normal_bf16(3, r, n, dev) for r in range(R)]
    outs = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    s = torch.cuda.current_stream().cuda_stream
    P.pl_collective(ctx, P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m), "copy", "bf16", R,
                    P.ptrs(ins), P.counts(ins), P.ptrs(outs), P.counts(outs), None, s)
    status_ok(ctx)
    for j in range(R):
        for r in range(R):
            assert torch.equal(outs[j][r * part:(r + 1) * part].view(torch.int16),
                               ins[r][j * part:(j + 1) * part].view(torch.int16)), f"A2A block {r}->{j}"
    for i in windows(part, seed=3, count=2):
        small = [np.concatenate([h(x[q * part + i:q * part + i + W], "bf16") for q in range(R)]) for x in ins]
        want = oracle.alltoall(small, [[W] * R for _ in range(R)], "bf16")
        for j in (0, R - 1):
            got = np.concatenate([h(outs[j][r * part + i:r * part + i + W], "bf16") for r in range(R)])
            assert_equal(got, want[j], f"A2A rank {j} window {i}")
    del ins, outs
    torch.cuda.empty_cache()
    # Ulysses: [16384 seq, 32 heads, 128 dim] per rank -> rank j holds heads j*4 .. j*4+3 of every sequence.
    Sq, H, D = 16384, 32, 128
    ins = [synth.device_normal_bf16(3, 10 + r, Sq * H * D, dev) for r in range(R)]
    outs = [torch.empty(Sq * H * D, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    P.pl_collective(ctx, P.pl_layout_ulysses_in(R, Sq, H, D), P.pl_layout_ulysses_out(R, Sq, H, D), "copy",
                    "bf16", R, P.ptrs(ins), P.counts(ins), P.ptrs(outs), P.counts(outs), None, s)
    status_ok(ctx)
    hs = H // R
    for j in range(R):
        got = outs[j].view(R, Sq, hs, D)
        for r in range(R):
            assert torch.equal(got[r].view(torch.int16),
                               ins[r].view(Sq, H, D)[:, j * hs:(j + 1) * hs].view(torch.int16)), f"Ulysses {r}->{j}"
    ws = 16
    for s0 in windows(Sq, seed=4, count=2, w=ws):
        small = [h(x[s0 * H * D:(s0 + ws) * H * D], "bf16") for x in ins]
        want = oracle.ulysses_a2a(small, ws, H, D, "bf16")
        for j in (0, R - 1):
            row = hs * D
            got = np.concatenate([h(outs[j][(r * Sq + s0) * row:(r * Sq + s0 + ws) * row], "bf16") for r in range(R)])
            assert_equal(got, want[j], f"Ulysses rank {j} seq {s0}")


def test_v_collectives_1GiB(ctx):
    dev = torch.device("cuda:0")
    N = GiB // 2
    lens = synth.zipf_lengths(N, R, 0.125, seed=4)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    s = torch.cuda.current_stream().cuda_stream
    # AllGatherV
    ins = [synth.device_normal_bf16(4, r, lens[r], dev) for r in range(R)]
    outs = [torch.empty(N, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    P.pl_collective(ctx, P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy", "bf16", R,
                    P.ptrs(ins), P.counts(ins), P.ptrs(outs), P.counts(outs), None, s)
    status_ok(ctx)
    cat = torch.cat(ins).view(torch.int16)
    for r in range(R):
        assert torch.equal(outs[r].view(torch.int16), cat), f"AllGatherV rank {r}"
    del cat
    for i in windows(min(lens), seed=5, count=2):
        want = oracle.allgather([h(x[i:i + W], "bf16") for x in ins], "bf16")[R - 1]
        got = np.concatenate([h(outs[R - 1][offs[q] + i:offs[q] + i + W], "bf16") for q in range(R)])
        assert_equal(got, want, f"AllGatherV window {i}")
    del ins, outs
    torch.cuda.empty_cache()
    # ReduceScatterV
    ins = [synth.device_normal_bf16(4, 100 + r, N, dev) for r in range(R)]
    outs = [torch.empty(lens[k], dtype=torch.bfloat16, device=dev) for k in range(R)]
    P.pl_collective(ctx, P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned(R, lens), "sum", "bf16", R,
                    P.ptrs(ins), P.counts(ins), P.ptrs(outs), P.counts(outs), None, s)
    status_ok(ctx)
    for k in range(R):
        for i in windows(lens[k], seed=20 + k, count=1):
            want = oracle.allreduce([h(x[offs[k] + i:offs[k] + i + W], "bf16") for x in ins], "bf16")[0]
            assert_equal(h(outs[k][i:i + W], "bf16"), want, f"ReduceScatterV rank {k} window {i}")
    del ins, outs
    torch.cuda.empty_cache()
    # AllToAllV: every source row is its own Zipf split of N / R elements.
    m = synth.zipf_matrix(N // R, R, 0.125, seed=4)
    ins = [synth.device_normal_bf16(4, 200 + r, sum(m[r]), dev) for r in range(R)]
    outn = [sum(m[r][j] for r in range(R)) for j in range(R)]
    outs = [torch.empty(outn[j], dtype=torch.bfloat16, device=dev) for j in range(R)]
    P.pl_collective(ctx, P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m), "copy", "bf16", R,
                    P.ptrs(ins), P.counts(ins), P.ptrs(outs), P.counts(outs), None, s)
    status_ok(ctx)
    for j in range(R):
        o = 0
        for r in range(R):
            src0 = sum(m[r][:j])
            blk = m[r][j]
            assert torch.equal(outs[j][o:o + blk].view(torch.int16),
                               ins[r][src0:src0 + blk].view(torch.int16)), f"AllToAllV block {r}->{j}"
            o += blk
    # the oracle on the first W elements of every block
    mw = [[min(W, m[r][j]) for j in range(R)] for r in range(R)]
    small = [np.concatenate([h(ins[r][sum(m[r][:j]):sum(m[r][:j]) + mw[r][j]], "bf16") for j in range(R)])
             for r in range(R)]
    want = oracle.alltoall(small, mw, "bf16")
    for j in range(R):
        starts = np.concatenate([[0], np.cumsum([m[r][j] for r in range(R)])])
        got = np.concatenate([h(outs[j][starts[r]:starts[r] + mw[r][j]], "bf16") for r in range(R)])
        assert_equal(got, want[j], f"AllToAllV rank {j}")
