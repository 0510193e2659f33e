"""SNAC derivation on the host (no GPU): work lists derived from layout pairs,
executed by a host emulation under random interleavings, equal the oracle."""
import numpy as np
import pytest

import oracle
import synth
from copy_reduce_datapath_gb300 import purlin as P

import plan_interp

NP = plan_interp.NPDT


def rand(dtype, seed, rank, n):
    t = synth.host_tensor("normal", dtype, seed, rank, n)
    if dtype in ("bf16", "fp16"):
        import torch
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def policy(path, ar_form=P.PL_AR_AUTO, chunk=256):
    return P.pl_policy_default(path=path, allreduce_form=ar_form, chunk_bytes=chunk)


def plan_for(lin, lout, op, dtype, R, pol, scratch=0):
    return P.pl_plan_create(lin, lout, op, dtype, R, pol, num_sms=4, scratch_bytes=scratch)


PATHS = [(P.PL_PATH_ZS, 0), (P.PL_PATH_STAGED, 8 * 2 * 1024)]
WINDOWS = [1, 3, 16]


def run_and_check(plan, R, dtype, ins, outs, want, window, seed=0):
    outs = [o.copy() for o in outs]
    plan_interp.run(plan, R, dtype, ins, outs, window=window, seed=seed)
    for r in range(R):
        assert np.array_equal(outs[r], want[r]), f"rank {r}"


@pytest.mark.parametrize("dtype", ["bf16", "fp32", "fp16", "fp8"])
@pytest.mark.parametrize("path,scratch", PATHS)
@pytest.mark.parametrize("window", WINDOWS)
def test_allgather_v(dtype, path, scratch, window):
    R = 5
    lens = [37, 0, 300, 1, 129]
    ins = [rand(dtype, 1, r, lens[r]) for r in range(R)]
    want = oracle.allgather(ins, dtype)
    lin, lout = P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens)
    pl = plan_for(lin, lout, "copy", dtype, R, policy(path), scratch)
    outs = [np.zeros(sum(lens), NP[dtype]) for _ in range(R)]
    run_and_check(pl, R, dtype, ins, outs, want, window, seed=window)


@pytest.mark.parametrize("dtype,op", [("bf16", "sum"), ("fp32", "sum"), ("fp16", "sum"), ("bf16", "max"),
                                      ("fp16", "max")])
@pytest.mark.parametrize("path,scratch", PATHS)
@pytest.mark.parametrize("window", WINDOWS)
def test_reducescatter_v(dtype, op, path, scratch, window):
    R = 4
    lens = [100, 3, 0, 250]
    N = sum(lens)
    ins = [rand(dtype, 2, r, N) for r in range(R)]
    want = oracle.reducescatter(ins, lens, dtype, op=op)
    lin, lout = P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned(R, lens)
    pl = plan_for(lin, lout, op, dtype, R, policy(path), scratch)
    outs = [np.zeros(lens[k], NP[dtype]) for k in range(R)]
    run_and_check(pl, R, dtype, ins, outs, want, window, seed=window)


@pytest.mark.parametrize("path,scratch", PATHS)
def test_reducescatter_in_place(path, scratch):
    R, dtype = 4, "bf16"
    lens = [64, 65, 7, 200]
    N = sum(lens)
    ins = [rand(dtype, 3, r, N) for r in range(R)]
    want = oracle.reducescatter(ins, lens, dtype)
    lin, lout = P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned_inplace(R, lens)
    pl = plan_for(lin, lout, "sum", dtype, R, policy(path), scratch)
    bufs = [a.copy() for a in ins]
    plan_interp.run(pl, R, dtype, bufs, bufs, window=8, seed=1)
    o = 0
    for k in range(R):
        assert np.array_equal(bufs[k][o:o + lens[k]], want[k])
        o += lens[k]


@pytest.mark.parametrize("dtype,op", [("bf16", "sum"), ("fp32", "sum"), ("fp16", "sum"), ("fp32", "max"),
                                      ("bf16", "max")])
@pytest.mark.parametrize("path,scratch", PATHS)
@pytest.mark.parametrize("form", [P.PL_AR_FUSED, P.PL_AR_COMPOSED, P.PL_AR_NOTIFIED])
@pytest.mark.parametrize("window", WINDOWS)
def test_allreduce(dtype, op, path, scratch, form, window):
    R = 3
    N = 3 * 301
    ins = [rand(dtype, 4, r, N) for r in range(R)]
    want = oracle.allreduce(ins, dtype, op=op)
    lens = synth.equal_lengths(N, R)
    L = P.pl_layout_partitioned(R, lens)
    pl = plan_for(L, L, op, dtype, R, policy(path, form), scratch)
    outs = [np.zeros(N, NP[dtype]) for _ in range(R)]
    run_and_check(pl, R, dtype, ins, outs, want, window, seed=window)


@pytest.mark.parametrize("dtype", ["bf16", "fp32", "fp8"])
@pytest.mark.parametrize("path,scratch", PATHS)
@pytest.mark.parametrize("window", WINDOWS)
def test_alltoall_v(dtype, path, scratch, window):
    R = 4
    m = [[(7 * r + 13 * j) % 90 for j in range(R)] for r in range(R)]
    ins = [rand(dtype, 5, r, sum(m[r])) for r in range(R)]
    want = oracle.alltoall(ins, m, dtype)
    lin, lout = P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m)
    pl = plan_for(lin, lout, "copy", dtype, R, policy(path), scratch)
    outs = [np.zeros(len(w), NP[dtype]) for w in want]
    run_and_check(pl, R, dtype, ins, outs, want, window, seed=window)


@pytest.mark.parametrize("path,scratch", PATHS)
@pytest.mark.parametrize("window", WINDOWS)
def test_ulysses(path, scratch, window):
    R, S, H, D, dtype = 4, 9, 8, 16, "bf16"
    ins = [rand(dtype, 6, r, S * H * D) for r in range(R)]
    want = oracle.ulysses_a2a(ins, S, H, D, dtype)
    lin, lout = P.pl_layout_ulysses_in(R, S, H, D), P.pl_layout_ulysses_out(R, S, H, D)
    pl = plan_for(lin, lout, "copy", dtype, R, policy(path, chunk=64 * 2), scratch)
    st = P.pl_plan_get_stats(pl)
    it, refs, _ = P.pl_plan_get_item(pl, 0)
    assert it.rows > 1 or st.items >= R * R  # strided rows are kept as rows
    outs = [np.zeros(len(w), np.uint16) for w in want]
    run_and_check(pl, R, dtype, ins, outs, want, window, seed=window)


def test_zero_staging_traffic_is_algorithmic():
    """ZS plans read and write exactly the algorithmic bytes of each collective."""
    R, n = 8, 1 << 16
    S = 2
    lens = [n] * R
    ag = plan_for(P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy", "bf16", R,
                  P.pl_policy_default())
    st = P.pl_plan_get_stats(ag)
    T = R * n * S
    assert (st.bytes_read, st.bytes_written) == (T, R * T)
    L = P.pl_layout_partitioned(R, lens)
    rs = plan_for(L, P.pl_layout_rank_owned(R, lens), "sum", "bf16", R, P.pl_policy_default())
    st = P.pl_plan_get_stats(rs)
    assert (st.bytes_read, st.bytes_written) == (R * T, T)
    ar = plan_for(L, L, "sum", "bf16", R, P.pl_policy_default())
    st = P.pl_plan_get_stats(ar)
    assert (st.bytes_read, st.bytes_written) == (R * T, R * T)
    assert st.flags == 0


def test_staged_plans_wait_only_on_earlier_items():
    """Every wait of item j is satisfied by items claimed before j (deadlock freedom)."""
    R, n = 4, 1000
    L = P.pl_layout_partitioned(R, [n] * R)
    pl = plan_for(L, L, "sum", "bf16", R, policy(P.PL_PATH_STAGED, P.PL_AR_COMPOSED), 4 * 2 * 300)
    st, items = plan_interp.load_plan(pl)
    notified, credited = {}, {}
    for j, (it, refs, syncs) in enumerate(items):
        for s in syncs[:it.nwait]:
            key = (s.flag, s.use)
            if s.type == P.PL_SYNC_WAIT_FULL:
                assert key in notified and notified[key] < j
            else:
                assert key in credited and credited[key][0] == credited[key][1]
        for s in syncs[it.nwait:]:
            key = (s.flag, s.use)
            if s.type == P.PL_SYNC_NOTIFY:
                notified[key] = j
            else:
                c = credited.get(key, [0, s.count])
                credited[key] = [c[0] + 1, s.count]
    assert st.slots >= 2 and st.uses_tickets == 1


def test_invalid_layout_pairs_are_refused():
    R = 2
    a = P.pl_layout_create(R, [[(0, 0, 4)], [(1, 0, 4)]])
    missing = P.pl_layout_create(R, [[(2, 0, 4)], []])
    short = P.pl_layout_create(R, [[(0, 0, 3)], []])
    two_on_one = P.pl_layout_create(R, [[(0, 0, 2), (0, 2, 2)], []])
    for lin, lout, op in ((a, missing, "copy"), (a, short, "copy"), (two_on_one, P.pl_layout_create(R, [[(0, 0, 2)], []]), "sum"),
                          (P.pl_layout_create(R, [[(0, 0, 4)], [(0, 0, 4)]]), P.pl_layout_create(R, [[(0, 0, 4)], []]), "copy")):
        with pytest.raises(P.PurlinError) as e:
            plan_for(lin, lout, op, "fp32", R, None)
        assert e.value.status == P.PL_ERR_LAYOUT
    # two strided regions of one name with different row lengths
    s1 = P.pl_layout_create(1, [[(0, 0, 4, 6, 10)]])
    s2 = P.pl_layout_create(1, [[(0, 0, 6, 4, 10)]])
    with pytest.raises(P.PurlinError) as e:
        plan_for(s1, s2, "copy", "bf16", 1, None)
    assert e.value.status == P.PL_ERR_UNSUPPORTED


def test_layout_arguments_are_checked():
    with pytest.raises(P.PurlinError):
        P.pl_layout_create(0, [])
    with pytest.raises(P.PurlinError):
        P.pl_layout_create(65, [[]] * 65)
    with pytest.raises(P.PurlinError):
        P.pl_layout_create(1, [[(0, 0, 8, 0, 8)]])       # rows = 0
    with pytest.raises(P.PurlinError):
        P.pl_layout_create(1, [[(0, 0, 8, 2, 4)]])       # stride < len
    with pytest.raises(P.PurlinError):
        P.pl_layout_ulysses_in(3, 4, 8, 2)              # H not a multiple of R


def test_staged_needs_a_ring():
    R = 4
    L = P.pl_layout_partitioned(R, [1000] * R)
    with pytest.raises(P.PurlinError) as e:
        plan_for(L, L, "sum", "bf16", R, policy(P.PL_PATH_STAGED, chunk=1024), scratch=R * 1024)
    assert e.value.status == P.PL_ERR_NOMEM


def test_op_and_dtype_codes_are_checked():
    """One-byte elements are moved, never reduced; unknown codes are invalid."""
    R = 2
    L = P.pl_layout_partitioned(R, [8, 8])
    for op in ("sum", "max"):
        with pytest.raises(P.PurlinError) as e:
            plan_for(L, L, op, "fp8", R, None)
        assert e.value.status == P.PL_ERR_UNSUPPORTED
    plan_for(P.pl_layout_rank_owned(R, [8, 8]), L, "copy", "fp8", R, None)
    for op, dt in ((3, "bf16"), (-1, "bf16"), ("sum", 4), ("copy", -1)):
        with pytest.raises(P.PurlinError) as e:
            plan_for(L, L, op, dt, R, None)
        assert e.value.status == P.PL_ERR_INVALID


def test_reduction_items_name_their_op():
    """Work items that reduce carry the op (1 sum, 2 maximum); copies carry 0:
    the notified composed form's gathers copy, the vector-grain form's items
    all reduce."""
    R = 4
    L = P.pl_layout_partitioned(R, [64] * R)
    for op, code in (("sum", 1), ("max", 2)):
        for form, want in ((P.PL_AR_NOTIFIED, {0, code}), (P.PL_AR_COMPOSED, {code})):
            pl = plan_for(L, L, op, "bf16", R, policy(P.PL_PATH_ZS, form))
            ops = {P.pl_plan_get_item(pl, i)[0].op for i in range(P.pl_plan_get_stats(pl).items)}
            assert ops == want


def test_one_byte_chunks_and_alignment():
    """Chunks of one-byte elements are whole 16-byte vectors; a plan whose
    byte offsets are all multiples of 16 covers every element exactly once."""
    R = 8
    lens = [4096 + 16 * r for r in range(R)]
    pl = plan_for(P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy", "fp8", R,
                  policy(P.PL_PATH_ZS, chunk=1024))
    st = P.pl_plan_get_stats(pl)
    assert st.chunk_elems % 16 == 0
    assert st.bytes_read == sum(lens) and st.bytes_written == R * sum(lens)


@pytest.mark.parametrize("scale", [1, 20])
@pytest.mark.parametrize("kind", ["allgatherv", "reducescatterv", "alltoallv", "ulysses", "allreduce_max"])
def test_automatic_chunking_covers_every_element(kind, scale):
    """Automatic chunks of plans whose items never wait (zero-staging), on a
    4-SM grid: about one item per CTA for small messages (scale 1: under
    256 KiB per CTA, and the misaligned ReduceScatterV up to 1 MiB per CTA,
    so at both scales); for larger ones (scale 20) guided sizes that shrink
    along the list, claimed in order once there are more items than CTAs.
    Executed by the emulator, the result equals the oracle.  (The vector
    datapath: the persistent kernel's chunk rule, not the inline form's.)"""
    R, dtype = 8, "bf16"
    pol = P.pl_policy_default(datapath=P.PL_ATOM_VECTOR)
    if kind == "allgatherv":
        lens = synth.zipf_lengths(60001 * scale, R, 0.125, seed=40)
        ins = [rand(dtype, 40, r, lens[r]) for r in range(R)]
        lin, lout, op = P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy"
        want = oracle.allgather(ins, dtype)
    elif kind == "reducescatterv":
        lens = synth.zipf_lengths(60001 * scale, R, 0.125, seed=41)
        ins = [rand(dtype, 41, r, sum(lens)) for r in range(R)]
        lin, lout, op = P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned(R, lens), "sum"
        want = oracle.reducescatter(ins, lens, dtype)
    elif kind == "alltoallv":
        m = synth.zipf_matrix(7001 * scale, R, 0.125, seed=42)
        ins = [rand(dtype, 42, r, sum(m[r])) for r in range(R)]
        lin, lout, op = P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m), "copy"
        want = oracle.alltoall(ins, m, dtype)
    elif kind == "ulysses":
        S_, H, D = 40 * scale, 16, 24
        ins = [rand(dtype, 43, r, S_ * H * D) for r in range(R)]
        lin, lout, op = P.pl_layout_ulysses_in(R, S_, H, D), P.pl_layout_ulysses_out(R, S_, H, D), "copy"
        want = oracle.ulysses_a2a(ins, S_, H, D, dtype)
    else:
        n = 100003 * scale
        ins = [rand(dtype, 44, r, n) for r in range(R)]
        L = P.pl_layout_partitioned(R, synth.equal_lengths(n, R))
        lin, lout, op = L, L, "max"
        want = oracle.allreduce(ins, dtype, op="max")
    pl = plan_for(lin, lout, op, dtype, R, pol)
    st, items = plan_interp.load_plan(pl)
    sizes = [it.rows * it.cols for it, _, _ in items]
    assert st.uses_tickets == (1 if st.items > st.ctas else 0)
    if kind == "reducescatterv":
        assert st.items <= st.ctas and st.uses_tickets == 0
    elif scale > 1 and kind != "alltoallv":  # (64 short transfers on 4 SMs: one item each, in turn)
        assert st.items > st.ctas
        assert max(sizes) <= 2 * sizes[0]  # the list starts with its largest items
        assert sum(sizes[: len(sizes) // 4]) >= sum(sizes[-(len(sizes) // 4):])  # and ends with small ones
    outs = [np.zeros(len(w), NP[dtype]) for w in want]
    run_and_check(pl, R, dtype, ins, outs, want, window=8, seed=3)


def test_staged_stages_of_a_row_merge():
    """In a staged plan, the stages one rank makes in one chunk row (its chunk of
    every partition into consecutive ring slots) form one strided item, and the
    plan still equals the oracle under the emulator."""
    R, dtype = 4, "bf16"
    n = 4 * 2048
    ins = [rand(dtype, 60, r, n) for r in range(R)]
    L = P.pl_layout_partitioned(R, synth.equal_lengths(n, R))
    pl = plan_for(L, L, "sum", dtype, R, policy(P.PL_PATH_STAGED, P.PL_AR_FUSED, chunk=1024), 64 * 1024)
    st, items = plan_interp.load_plan(pl)
    stages = [(it, refs) for it, refs, _ in items if it.kind == P.PL_ITEM_STAGE]
    assert stages and all(it.rows == R for it, _ in stages)
    for it, refs in stages:
        src, dst = refs[0], refs[1]
        assert src.stride == n // R and dst.space == P.PL_SPACE_SCRATCH and dst.stride >= it.cols
        assert it.npost == R  # one notify per slot
    want = oracle.allreduce(ins, dtype)
    outs = [np.zeros(n, NP[dtype]) for _ in range(R)]
    run_and_check(pl, R, dtype, ins, outs, want, window=8, seed=5)


# ------------------------------------------------ the inline-parameter form


def small_layouts(coll, R, n):
    """Layout pair and op of an equal-partition collective over n elements per rank."""
    lens = [n // R] * R
    if coll == "allgather":
        return P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy"
    if coll == "reducescatter":
        return P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned(R, lens), "sum"
    L = P.pl_layout_partitioned(R, lens)
    return L, L, "sum"


def oracle_of(coll, ins, R, n, dtype):
    if coll == "allgather":
        return oracle.allgather(ins, dtype)
    if coll == "reducescatter":
        return oracle.reducescatter(ins, [n // R] * R, dtype)
    return oracle.allreduce(ins, dtype)


@pytest.mark.parametrize("T", [1 << 10, 1 << 13, 1 << 16, 1 << 18])
@pytest.mark.parametrize("coll", ["allgather", "allreduce", "reducescatter"])
def test_inline_form_for_small_aligned_plans(coll, T):
    """Zero-staging one-row plans between 16-byte aligned regions, small enough:
    the whole list in the launch parameters, one item per CTA (at most 152
    items, 2432 references); a 1 KiB message fits the small parameter block.
    Executed by the emulator, the result equals the oracle."""
    R, dtype = 8, "bf16"
    n = T // 2
    lin, lout, op = small_layouts(coll, R, n)
    pl = P.pl_plan_create(lin, lout, op, dtype, R, None, num_sms=152)
    st, items = plan_interp.load_plan(pl)
    assert st.datapath == P.PL_ATOM_INLINE
    assert st.ctas == st.items <= 152 and st.refs <= 2432 and st.threads == 512 and st.uses_tickets == 0
    if T == 1 << 10:
        assert st.items <= 16 and st.refs <= 256
    for it, refs, syncs in items:
        assert it.rows == 1 and not syncs and it.kind == P.PL_ITEM_MOVE
        assert all(f.offset * 2 % 16 == 0 for f in refs)
    in_n = n // R if coll == "allgather" else n
    ins = [rand(dtype, 70, r, in_n) for r in range(R)]
    want = oracle_of(coll, ins, R, n, dtype)
    outs = [np.zeros(len(w), NP[dtype]) for w in want]
    run_and_check(pl, R, dtype, ins, outs, want, window=8, seed=7)


def test_inline_form_not_taken():
    """Plans the inline form does not take: moving more than 320 MiB (unless
    every transfer reduces into one destination between aligned regions),
    misaligned regions whose items would exceed one vector per thread,
    destinations of one name at different offsets mod 16 bytes, staged,
    composed, strided, a fixed grid, a forced datapath, too many references;
    the form forced on a plan it cannot take leaves the vector datapath."""
    R, dtype, n = 8, "bf16", 1 << 12

    def form(lin, lout, op, pol=None, R_=R):
        pl = P.pl_plan_create(lin, lout, op, dtype, R_, pol, num_sms=152, scratch_bytes=1 << 20)
        try:
            return P.pl_plan_get_stats(pl).datapath
        finally:
            P.pl_plan_destroy(pl)

    ag = small_layouts("allgather", R, n)
    ar = small_layouts("allreduce", R, n)
    assert form(*ag) == P.PL_ATOM_INLINE and form(*ar) == P.PL_ATOM_INLINE
    assert form(*small_layouts("allgather", R, 1 << 23)) == P.PL_ATOM_INLINE        # 16 MiB per rank: 144 MiB moved
    assert form(*small_layouts("allgather", R, 1 << 25)) == P.PL_ATOM_BULK          # 64 MiB: the bulk ring
    assert form(*small_layouts("allreduce", R, 1 << 23)) == P.PL_ATOM_INLINE        # 256 MiB moved
    assert form(*small_layouts("allreduce", R, 1 << 24)) == P.PL_ATOM_VECTOR        # 512 MiB moved
    assert form(*small_layouts("reducescatter", R, 1 << 29)) == P.PL_ATOM_INLINE    # 1 GiB: the ReduceScatter shape
    assert form(*ag, P.pl_policy_default(path=P.PL_PATH_STAGED)) == P.PL_ATOM_VECTOR
    assert form(*ar, P.pl_policy_default(allreduce_form=P.PL_AR_COMPOSED)) == P.PL_ATOM_VECTOR
    assert form(*ar, P.pl_policy_default(allreduce_form=P.PL_AR_COMPOSED, datapath=P.PL_ATOM_INLINE)) == \
        P.PL_ATOM_VECTOR
    assert form(*ar, P.pl_policy_default(allreduce_form=P.PL_AR_NOTIFIED)) == P.PL_ATOM_VECTOR
    assert form(*ag, P.pl_policy_default(ctas=64)) == P.PL_ATOM_VECTOR
    assert form(*ag, P.pl_policy_default(datapath=P.PL_ATOM_VECTOR)) == P.PL_ATOM_VECTOR
    assert form(*ag, P.pl_policy_default(datapath=P.PL_ATOM_BULK)) == P.PL_ATOM_BULK
    assert form(*ag, P.pl_policy_default(chunk_bytes=1024)) == P.PL_ATOM_VECTOR
    uly = (P.pl_layout_ulysses_in(R, 16, 16, 8), P.pl_layout_ulysses_out(R, 16, 16, 8), "copy")
    assert form(*uly) == P.PL_ATOM_VECTOR
    assert form(*uly, P.pl_policy_default(datapath=P.PL_ATOM_INLINE)) == P.PL_ATOM_VECTOR
    lens = synth.zipf_lengths(3001, R, 0.125, seed=71)
    assert form(P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy") == P.PL_ATOM_INLINE
    lens = synth.zipf_lengths((1 << 22) + 1, R, 0.125, seed=71)                       # 8 MiB AllGatherV
    assert form(P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy") == P.PL_ATOM_INLINE
    lens = synth.zipf_lengths((1 << 23) + 1, R, 0.125, seed=71)                       # 16 MiB AllGatherV
    assert form(P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens), "copy") == P.PL_ATOM_BULK
    lens = synth.zipf_lengths((1 << 25) + 1, R, 0.125, seed=71)                       # 64 MiB ReduceScatterV
    assert form(P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned(R, lens), "sum") == P.PL_ATOM_VECTOR
    # one name's two destinations at offsets 0 and 3 (elements): not congruent mod 16 bytes
    lin2 = P.pl_layout_create(2, [[(0, 0, 64)], [(1, 0, 64)]])
    lout2 = P.pl_layout_create(2, [[(0, 0, 64), (1, 64, 64)], [(0, 3, 64), (1, 67, 64)]])
    assert form(lin2, lout2, "copy", None, 2) == P.PL_ATOM_VECTOR
    lout3 = P.pl_layout_create(2, [[(0, 0, 64), (1, 64, 64)], [(0, 8, 64), (1, 72, 64)]])
    assert form(lin2, lout3, "copy", None, 2) == P.PL_ATOM_INLINE
    L64 = P.pl_layout_partitioned(64, [64] * 64)
    assert form(L64, L64, "sum", None, 64) == P.PL_ATOM_VECTOR                     # 64 x 128 references


def test_forced_inline_cuts_at_most_152_items():
    """PL_ATOM_INLINE forced on a 2 MiB AllGather: at most 152 items, as large
    as the message needs; the emulator gives the oracle's result."""
    R, dtype, n = 8, "bf16", (1 << 20) + 8 * 16
    lin, lout, op = small_layouts("allgather", R, n)
    pl = P.pl_plan_create(lin, lout, op, dtype, R, P.pl_policy_default(datapath=P.PL_ATOM_INLINE), num_sms=152)
    st, items = plan_interp.load_plan(pl)
    assert st.datapath == P.PL_ATOM_INLINE and st.items <= 152
    assert sum(it.cols for it, _, _ in items) == n
    ins = [rand(dtype, 72, r, n // R) for r in range(R)]
    want = oracle.allgather(ins, dtype)
    outs = [np.zeros(n, NP[dtype]) for _ in range(R)]
    run_and_check(pl, R, dtype, ins, outs, want, window=16, seed=9)


def test_flagged_reductions_take_two_ctas_per_sm():
    """Lists with flags that reduce (staged, notified composed) are sized for
    the two-CTA spliced kernels (512 threads) even when aligned; aligned lists
    without flags that only reduce (the fused and vector-grain composed
    AllReduce) for two CTAs of 256 threads per SM; staged copies and aligned
    copies keep one CTA of 512 per SM."""
    R, dtype, n = 8, "bf16", 1 << 22
    L = P.pl_layout_partitioned(R, [n // R] * R)
    lo = P.pl_layout_rank_owned(R, [n // R] * R)

    def shape(lin, lout, op, pol):
        pl = P.pl_plan_create(lin, lout, op, dtype, R, pol, num_sms=152, scratch_bytes=64 << 20)
        try:
            st = P.pl_plan_get_stats(pl)
            return st.ctas, st.threads
        finally:
            P.pl_plan_destroy(pl)

    staged = P.pl_policy_default(path=P.PL_PATH_STAGED)
    composed = P.pl_policy_default(allreduce_form=P.PL_AR_COMPOSED)
    notified = P.pl_policy_default(allreduce_form=P.PL_AR_NOTIFIED)
    vector = P.pl_policy_default(datapath=P.PL_ATOM_VECTOR)
    assert shape(L, L, "sum", staged) == (304, 512)
    assert shape(L, lo, "sum", staged) == (304, 512)
    assert shape(L, L, "sum", notified) == (304, 512)
    assert shape(L, L, "sum", composed) == (304, 256)
    assert shape(L, L, "sum", vector) == (304, 256)
    assert shape(lo, L, "copy", staged) == (152, 512)
    assert shape(lo, L, "copy", vector) == (152, 512)


def test_notified_gather_reads_the_owners_chunk_once():
    """Zero-staging notified composed AllReduce (Figure 6): per chunk, the owner's reduce
    (R sources, one destination, then a Notify) and one gather item that waits
    for it and copies the reduced chunk to the R - 1 other ranks.  Bytes over
    all chunks: the reduces read R x n and write n elements, the gathers read n
    and write (R - 1) x n.  The emulator gives the oracle's result."""
    R, dtype, n = 8, "bf16", 8 * 3000 + 5
    ins = [rand(dtype, 73, r, n) for r in range(R)]
    L = P.pl_layout_partitioned(R, synth.equal_lengths(n, R))
    pl = plan_for(L, L, "sum", dtype, R, P.pl_policy_default(allreduce_form=P.PL_AR_NOTIFIED, chunk_bytes=1024))
    st, items = plan_interp.load_plan(pl)
    reduces = [(it, syncs) for it, _, syncs in items if it.nsrc == R]
    gathers = [(it, syncs) for it, _, syncs in items if it.nsrc == 1]
    assert len(reduces) == len(gathers) > 0
    assert all(it.ndst == 1 and it.npost == 1 for it, _ in reduces)
    assert all(it.ndst == R - 1 and it.nwait == 1 for it, _ in gathers)
    S = 2
    assert st.bytes_read == R * n * S + n * S
    assert st.bytes_written == n * S + (R - 1) * n * S
    want = oracle.allreduce(ins, dtype)
    outs = [np.zeros(n, NP[dtype]) for _ in range(R)]
    run_and_check(pl, R, dtype, ins, outs, want, window=8, seed=11)


def test_one_to_one_plans_take_one_item_per_cta():
    """One-to-one transfers take one item per CTA up to 512 KiB per CTA when
    aligned and up to 2 MiB when not: an AllToAllV (Zipf rows, misaligned) of
    64 MiB per rank (about 1.8 MB per CTA of a 304-CTA grid) runs one item per
    CTA with no ticket, of 128 MiB guided items claimed in order; the aligned
    AllToAll of 32 MiB per rank (1.8 MB per CTA of 152) near-equal items."""
    R = 8

    def stats(lin, lout):
        pl = P.pl_plan_create(lin, lout, "copy", "bf16", R, P.pl_policy_default(datapath=P.PL_ATOM_VECTOR),
                              num_sms=152)
        try:
            return P.pl_plan_get_stats(pl)
        finally:
            P.pl_plan_destroy(pl)

    def a2av(T):
        m = synth.zipf_matrix(T // 2, R, 0.125, seed=4)
        return stats(P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m))

    st = a2av(16 << 20)
    assert st.items == st.ctas and st.uses_tickets == 0
    st = a2av(64 << 20)
    assert st.items <= st.ctas and st.uses_tickets == 0
    st = a2av(128 << 20)
    assert st.items > st.ctas and st.uses_tickets == 1
    m = [[(32 << 20) // 2 // R] * R for _ in range(R)]
    st = stats(P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m))
    assert st.items > st.ctas


@pytest.mark.parametrize("op", ["sum", "max"])
@pytest.mark.parametrize("chunk", [0, 1024])
def test_vector_grain_composition_writes_the_owner_first(op, chunk):
    """Zero-staging PL_AR_COMPOSED (Figure 6 at the grain of one vector): one
    kCompose item per chunk, no flags and no tickets; its first destination is
    the output of the partition's owner (rank k for partition k), followed by
    every other rank's output.  Bytes: the reduce reads R x n and writes n,
    the reread reads n, the gather writes (R - 1) x n.  The emulator, which
    writes the other ranks from what it reads back from the owner, gives the
    oracle's result."""
    R, dtype, n = 8, "bf16", 8 * 3000 + 5
    ins = [rand(dtype, 74, r, n) for r in range(R)]
    lens = synth.equal_lengths(n, R)
    L = P.pl_layout_partitioned(R, lens)
    pl = plan_for(L, L, op, dtype, R, P.pl_policy_default(allreduce_form=P.PL_AR_COMPOSED, chunk_bytes=chunk))
    st, items = plan_interp.load_plan(pl)
    assert st.syncs == 0 and st.flags == 0 and st.items == len(items) > 0
    starts = np.cumsum([0] + lens)
    for it, refs, syncs in items:
        assert it.kind == P.PL_ITEM_COMPOSE and it.nsrc == R and it.ndst == R and not syncs
        srcs, dsts = refs[:R], refs[R:]
        assert [(f.space, f.index) for f in srcs] == [(P.PL_SPACE_IN, r) for r in range(R)]
        owner = int(np.searchsorted(starts, srcs[0].offset, side="right")) - 1
        assert (dsts[0].space, dsts[0].index) == (P.PL_SPACE_OUT, owner)
        assert sorted(f.index for f in dsts[1:]) == [r for r in range(R) if r != owner]
        assert all(f.offset == srcs[0].offset for f in refs)
    S = 2
    assert st.bytes_read == R * n * S + n * S
    assert st.bytes_written == R * n * S
    want = oracle.allreduce(ins, dtype, op=op)
    outs = [np.zeros(n, NP[dtype]) for _ in range(R)]
    run_and_check(pl, R, dtype, ins, outs, want, window=8, seed=12)



def test_equal_bulk_lists_end_with_half_size_items():
    """An AllGather on the bulk ring (equal transfers): near-equal items, then
    about two grids of half-size items at the end of the list; every element
    covered once, and the emulator gives the oracle's result."""
    R, dtype = 8, "bf16"
    n = 1 << 19  # 1 MiB per rank: 2 MiB per CTA of a 4-SM grid
    lin, lout, op = P.pl_layout_rank_owned(R, [n] * R), P.pl_layout_partitioned(R, [n] * R), "copy"
    pl = plan_for(lin, lout, op, dtype, R, P.pl_policy_default(datapath=P.PL_ATOM_BULK))
    st, items = plan_interp.load_plan(pl)
    sizes = [it.cols for it, _, _ in items]
    assert st.datapath == P.PL_ATOM_BULK and sum(sizes) == R * n
    tail = 2 * st.ctas
    assert max(sizes[-tail:]) * 2 <= max(sizes[:-tail]) + 128  # halves (grain-rounded) of the equal items
    ins = [rand(dtype, 75, r, n) for r in range(R)]
    want = oracle.allgather(ins, dtype)
    outs = [np.zeros(n * R, NP[dtype]) for _ in range(R)]
    run_and_check(pl, R, dtype, ins, outs, want, window=6, seed=13)
