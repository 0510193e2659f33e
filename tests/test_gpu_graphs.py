"""Collectives captured in a CUDA graph and replayed: every replay repeats the
launch's parameters, so the SNAC flag tags of a launch come from a device
epoch that the last CTA out of each launch advances (not from the host).
Each replay, on fresh inputs, must equal the oracle bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synth
from copy_reduce_datapath_gb300 import purlin as P

from gpu_util import assert_equal, host, to_np

pytestmark = pytest.mark.gpu

SCRATCH = 64 << 20


@pytest.fixture(scope="module")
def ctx():
    torch.cuda.set_device(0)
    c = P.pl_ctx_create(0, SCRATCH)
    yield c
    P.pl_ctx_destroy(c)


def policies():
    return {
        "zs": None,
        "zs_composed": P.pl_policy_default(allreduce_form=P.PL_AR_COMPOSED, chunk_bytes=8192),
        "zs_notified": P.pl_policy_default(allreduce_form=P.PL_AR_NOTIFIED, chunk_bytes=8192),
        "staged_fused": P.pl_policy_default(path=P.PL_PATH_STAGED, chunk_bytes=8192),
        "staged_composed": P.pl_policy_default(path=P.PL_PATH_STAGED, allreduce_form=P.PL_AR_COMPOSED,
                                               chunk_bytes=8192),
        "zs_vector": P.pl_policy_default(datapath=P.PL_ATOM_VECTOR, chunk_bytes=8192),
    }


@pytest.mark.parametrize("name", list(policies()))
def test_allreduce_replayed_from_a_cuda_graph(ctx, name):
    R, n, dtype = 8, 8 * 6000 + 5, "bf16"
    pol = policies()[name]
    L = P.pl_layout_partitioned(R, synth.equal_lengths(n, R))
    ins = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]

    def fill(seed):
        hs = [host("normal", dtype, seed, r, n) for r in range(R)]
        for r in range(R):
            ins[r].view(torch.int16).copy_(torch.from_numpy(hs[r].view(np.int16)))
        return hs

    def check(hs, what):
        want = oracle.allreduce(hs, dtype)
        for r in range(R):
            assert_equal(to_np(outs[r], dtype), want[r], f"{what} rank {r}")

    # The first call derives and uploads the work list (not capturable).
    hs = fill(60)
    s = P.stream_handle()
    P.pl_collective(ctx, L, L, "sum", dtype, R, P.ptrs(ins), [n] * R, P.ptrs(outs), [n] * R, pol, s)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    check(hs, "eager")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        P.pl_collective(ctx, L, L, "sum", dtype, R, P.ptrs(ins), [n] * R, P.ptrs(outs), [n] * R, pol,
                        P.stream_handle())
    for rep in range(3):
        hs = fill(61 + rep)
        for o in outs:
            o.fill_(0)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert P.pl_ctx_status(ctx, P.stream_handle()) == P.PL_OK
        check(hs, f"replay {rep}")
    # an eager call after the replays still sees fresh tags
    hs = fill(70)
    P.pl_collective(ctx, L, L, "sum", dtype, R, P.ptrs(ins), [n] * R, P.ptrs(outs), [n] * R, pol, s)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    check(hs, "eager after replays")


def test_staged_allgather_replayed_twice_in_one_graph(ctx):
    """Two launches of one staged plan inside one graph, replayed: four epochs."""
    R, dtype = 8, "bf16"
    lens = synth.zipf_lengths(30001, R, 0.125, seed=62)
    N = sum(lens)
    pol = P.pl_policy_default(path=P.PL_PATH_STAGED, chunk_bytes=4096)
    lin, lout = P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens)
    src = [torch.empty(m, dtype=torch.bfloat16, device="cuda") for m in lens]
    mid = [torch.empty(N, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    s = P.stream_handle()

    def fill(seed):
        hs = [host("normal", dtype, seed, r, lens[r]) for r in range(R)]
        for r in range(R):
            src[r].view(torch.int16).copy_(torch.from_numpy(hs[r].view(np.int16)))
        return hs

    fill(63)
    P.pl_collective(ctx, lin, lout, "copy", dtype, R, P.ptrs(src), lens, P.ptrs(mid), [N] * R, pol, s)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = P.stream_handle()
        P.pl_collective(ctx, lin, lout, "copy", dtype, R, P.ptrs(src), lens, P.ptrs(mid), [N] * R, pol, cs)
        P.pl_collective(ctx, lin, lout, "copy", dtype, R, P.ptrs(src), lens, P.ptrs(mid), [N] * R, pol, cs)
    for rep in range(2):
        hs = fill(64 + rep)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert P.pl_ctx_status(ctx, P.stream_handle()) == P.PL_OK
        want = oracle.allgather(hs, dtype)
        for r in range(R):
            assert_equal(to_np(mid[r], dtype), want[r], f"replay {rep} rank {r}")
