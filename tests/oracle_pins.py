"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with what the Purlin pages or the mathematics fix:

* hand-worked Figure 4 placements on three ranks (tests/golden/);
* exact sums of small integers, compared with numpy's int64 sum;
* a summation order that only the rank-ordered fp32 fold gets right, and the
  sign of a zero sum;
* Higham's forward-error bound for recursive summation, against an fp64 sum;
* PyTorch's own fp32 -> bf16 cast on a large sweep of bit patterns;
* numpy concatenate / split / reshape-transpose as library statements of the
  placements;
* the invariants AllReduce = AllGather o ReduceScatter and AllToAll o AllToAll = id;
* R = 1 reducing every collective to a copy;
* brute force on tiny inputs against per-element definitions written here.

``tests/test_oracle_pins.py`` runs them on the committed oracle;
``tests/test_oracle_mutations.py`` runs them on mutated copies and expects a failure.
"""
from __future__ import annotations

import numpy as np

import synth
from _golden import load as load_golden


def _as(dtype, vals):
    a = np.asarray(vals, dtype=np.float32)
    if dtype == "fp32":
        return a
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)  # exact for these small ints


def _vals(dtype, a):
    a = np.asarray(a)
    if dtype == "fp32":
        return a.astype(np.float64)
    return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _rand(dtype, seed, rank, n, kind="normal"):
    t = synth.host_tensor(kind, dtype, seed, rank, n)
    if dtype == "bf16":
        import torch
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


# ------------------------------------------------------------ golden fixtures


def check_fig4_golden(orc):
    g = load_golden("fig4_three_ranks.txt")
    for dt in ("fp32", "bf16"):
        ins = [_as(dt, g["input"][r]) for r in range(3)]
        rs = orc.reducescatter(ins, [2, 2, 2], dt)
        for k in range(3):
            assert list(_vals(dt, rs[k])) == g["reducescatter"][k], ("RS", dt, k)
        ag = orc.allgather(rs, dt)
        for r in range(3):
            assert list(_vals(dt, ag[r])) == g["allgather"][r], ("AG", dt, r)
        ar = orc.allreduce(ins, dt)
        for r in range(3):
            assert list(_vals(dt, ar[r])) == g["allreduce"][r], ("AR", dt, r)
        a2a = orc.alltoall(ins, [[2, 2, 2]] * 3, dt)
        for j in range(3):
            assert list(_vals(dt, a2a[j])) == g["alltoall"][j], ("A2A", dt, j)


def check_v_golden(orc):
    g = load_golden("v_forms_three_ranks.txt")
    for dt in ("fp32", "bf16"):
        agv = orc.allgather([_as(dt, g["agv_input"][r]) for r in range(3)], dt)
        for r in range(3):
            assert list(_vals(dt, agv[r])) == g["allgatherv"][r], ("AGV", dt, r)
        rsv = orc.reducescatter([_as(dt, g["rsv_input"][r]) for r in range(3)], g["rsv_lens"][0], dt)
        for k in range(3):
            assert list(_vals(dt, rsv[k])) == g["reducescatterv"][k], ("RSV", dt, k)
        m = [g["a2av_lens"][r] for r in range(3)]
        a2av = orc.alltoall([_as(dt, g["a2av_input"][r]) for r in range(3)], m, dt)
        for j in range(3):
            assert list(_vals(dt, a2av[j])) == g["alltoallv"][j], ("A2AV", dt, j)


# ---------------------------------------------------------------- arithmetic


def check_integer_sums_exact(orc):
    """Small integers sum exactly in any order: compare with numpy's int64 sum."""
    # The three-rank AllReduce workload: 3 x 4096 fp32 integers in [-8, 8], seed 0.
    R, n = 3, 3 * 4096
    ins = [synth.int_uniform_f32(0, r, n) for r in range(R)]
    exact = np.sum(np.stack([a.astype(np.int64) for a in ins]), axis=0)
    for out in orc.allreduce(ins, "fp32"):
        assert np.array_equal(out.astype(np.int64), exact)
    rs = orc.reducescatter(ins, [4096] * 3, "fp32")
    for k in range(R):
        assert np.array_equal(rs[k].astype(np.int64), exact[4096 * k:4096 * (k + 1)])
    # Eight ranks in bf16: |sum| <= 64 is exact in bf16's 8-bit significand.
    R, n = 8, 1000
    ins32 = [synth.int_uniform_f32(7, r, n) for r in range(R)]
    exact = np.sum(np.stack([a.astype(np.int64) for a in ins32]), axis=0)
    ins16 = [_as("bf16", a) for a in ins32]
    for out in orc.allreduce(ins16, "bf16"):
        assert np.array_equal(_vals("bf16", out).astype(np.int64), exact)
    lens = [100, 0, 250, 1, 149, 300, 100, 100]
    rs = orc.reducescatter(ins16, lens, "bf16")
    o = 0
    for k in range(R):
        assert np.array_equal(_vals("bf16", rs[k]).astype(np.int64), exact[o:o + lens[k]])
        o += lens[k]


def check_rank_order(orc):
    """Only a fold in rank order 0, 1, 2 maps (2^24, 1, -2^24) to 0 in fp32.

    2^24 + 1 is a tie between 2^24 and 2^24 + 2 and rounds to the even 2^24,
    so the rank-ordered sum is 0; summing ranks 2, 1, 0 or pairing ranks 1 and 2
    first gives 1.  A fold that starts from +0 instead of the rank-0 value turns
    (-0) + (-0) + (-0) into +0.
    """
    a = [np.array([2.0 ** 24, 1.0], np.float32), np.array([1.0, 2.0 ** 24], np.float32),
         np.array([-(2.0 ** 24), -(2.0 ** 24)], np.float32)]
    for out in orc.allreduce(a, "fp32"):
        assert out[0] == 0.0 and out[1] == 0.0, out
    # x = (1, -2^24, 2^24): the rank-ordered fold gives (1 - 2^24) + 2^24 = 1 exactly.
    b = [np.array([1.0], np.float32), np.array([-(2.0 ** 24)], np.float32),
         np.array([2.0 ** 24], np.float32)]
    assert orc.allreduce(b, "fp32")[0][0] == 1.0
    z = [np.array([-0.0], np.float32)] * 3
    out = orc.allreduce(z, "fp32")[0]
    assert out.view(np.uint32)[0] == 0x80000000, hex(out.view(np.uint32)[0])
    zb = [np.array([0x8000], np.uint16)] * 3
    assert orc.allreduce(zb, "bf16")[0][0] == 0x8000


def check_fp64_error_bound(orc):
    """|fold - exact| <= gamma_{R-1} * sum|x| (Higham, recursive summation), plus
    one bf16 rounding (relative 2^-8) for bf16 outputs."""
    for dt, R in (("fp32", 8), ("bf16", 8), ("fp32", 5), ("bf16", 3)):
        n = 20000
        ins = [_rand(dt, 11, r, n) for r in range(R)]
        x = np.stack([_vals(dt, a) for a in ins])
        exact = x.sum(axis=0)
        absum = np.abs(x).sum(axis=0)
        u = 2.0 ** -24
        gam = (R - 1) * u / (1 - (R - 1) * u)
        fp32_err = gam * absum
        out = _vals(dt, orc.allreduce(ins, dt)[R - 1])
        bound = fp32_err if dt == "fp32" else fp32_err + 2.0 ** -8 * (np.abs(exact) + fp32_err)
        assert np.all(np.abs(out - exact) <= bound * (1 + 1e-12) + 1e-300), dt
        # and it is not a trivially loose match: most elements are within 1 ulp-ish
        assert np.mean(np.abs(out - exact) <= 2.0 ** -7 * np.abs(exact) + 1e-6) > 0.99


def check_bf16_rounding_vs_torch(orc):
    """The oracle's fp32->bf16 rounding equals PyTorch's CPU cast (a library
    round-to-nearest-even) on every upper half with a spread of lower halves:
    exact ties, just below/above a tie, zero, all-ones and random."""
    import torch
    hi = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = [0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000]
    rng = np.random.default_rng(5)
    lows += list(rng.integers(0, 1 << 16, size=8))
    pats = np.concatenate([hi | np.uint32(l) for l in lows])
    f = pats.view(np.float32)
    mine = orc.f32_to_bf16(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(mine[~nan], ref[~nan])
    mine_nan = mine[nan]
    assert np.all(((mine_nan & 0x7F80) == 0x7F80) & ((mine_nan & 0x7F) != 0))


# ---------------------------------------------------------------- placement


def check_library_placements(orc):
    """AllGather is concatenation; AllToAll is split-then-concatenate (numpy)."""
    for dt in ("fp32", "bf16"):
        R = 5
        lens = [3, 0, 7, 1, 12]
        ins = [_rand(dt, 2, r, lens[r]) for r in range(R)]
        want = np.concatenate(ins)
        for out in orc.allgather(ins, dt):
            assert np.array_equal(out, want)
        m = [[(r * 3 + j * 5) % 4 for j in range(R)] for r in range(R)]
        ins = [_rand(dt, 3, r, sum(m[r])) for r in range(R)]
        pieces = [np.split(ins[r], np.cumsum(m[r])[:-1]) for r in range(R)]
        outs = orc.alltoall(ins, m, dt)
        for j in range(R):
            assert np.array_equal(outs[j], np.concatenate([pieces[r][j] for r in range(R)]))


def check_ulysses_vs_numpy(orc):
    """Sequence->head re-partition equals numpy's reshape/slice/concatenate."""
    R, S, H, D = 4, 5, 8, 3
    for dt in ("bf16", "fp32"):
        ins = [_rand(dt, 3, r, S * H * D) for r in range(R)]
        outs = orc.ulysses_a2a(ins, S, H, D, dt)
        hs = H // R
        for j in range(R):
            want = np.concatenate([ins[r].reshape(S, H, D)[:, j * hs:(j + 1) * hs, :] for r in range(R)])
            assert np.array_equal(outs[j], want.ravel())


def check_invariants(orc):
    """AllReduce == AllGather(ReduceScatter(x)) bit for bit (Figure 6), and
    AllToAll applied twice (transposed lengths for V) is the identity."""
    for dt in ("fp32", "bf16"):
        for R, lens in ((2, [5, 4]), (3, [7, 0, 9]), (8, [13, 1, 0, 40, 2, 9, 16, 3])):
            ins = [_rand(dt, 9, r, sum(lens)) for r in range(R)]
            ar = orc.allreduce(ins, dt)
            ag = orc.allgather(orc.reducescatter(ins, lens, dt), dt)
            for r in range(R):
                assert np.array_equal(ar[r], ag[r]), (dt, R, r)
        R = 6
        ins = [_rand(dt, 4, r, 6 * 5) for r in range(R)]
        once = orc.alltoall(ins, [[5] * R] * R, dt)
        twice = orc.alltoall(once, [[5] * R] * R, dt)
        for r in range(R):
            assert np.array_equal(twice[r], ins[r])
        m = synth.zipf_matrix(57, R, 0.125, seed=4)
        mt = [[m[j][r] for j in range(R)] for r in range(R)]
        ins = [_rand(dt, 4, r, sum(m[r])) for r in range(R)]
        back = orc.alltoall(orc.alltoall(ins, m, dt), mt, dt)
        for r in range(R):
            assert np.array_equal(back[r], ins[r])


def check_single_rank_is_copy(orc):
    for dt in ("fp32", "bf16"):
        x = _rand(dt, 1, 0, 37)
        assert np.array_equal(orc.allgather([x], dt)[0], x)
        assert np.array_equal(orc.reducescatter([x], [37], dt)[0], x)
        assert np.array_equal(orc.allreduce([x], dt)[0], x)
        assert np.array_equal(orc.alltoall([x], [[37]], dt)[0], x)


# -------------------------------------------------------------- brute force


def _bf_fold(dt, vals):
    acc = np.float32(_vals(dt, [vals[0]])[0])
    for v in vals[1:]:
        acc = np.float32(acc + np.float32(_vals(dt, [v])[0]))
    if dt == "fp32":
        return acc
    import torch
    return torch.tensor([float(acc)], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[0]


def check_bruteforce(orc):
    """Tiny cases against per-element definitions written independently here."""
    rng = np.random.default_rng(123)
    for dt in ("fp32", "bf16"):
        for R in (1, 2, 3, 5):
            lens = [int(x) for x in rng.integers(0, 5, size=R)]
            N = sum(lens)
            ins = [_rand(dt, 21 + R, r, N) for r in range(R)]
            rs = orc.reducescatter(ins, lens, dt)
            starts = [sum(lens[:k]) for k in range(R)]
            for k in range(R):
                for i in range(lens[k]):
                    want = _bf_fold(dt, [ins[r][starts[k] + i] for r in range(R)])
                    assert rs[k][i] == want or (np.isnan(rs[k][i]) and np.isnan(want))
            gins = [_rand(dt, 31 + R, r, lens[r]) for r in range(R)]
            ag = orc.allgather(gins, dt)
            for r in range(R):
                pos = 0
                for j in range(R):
                    for i in range(lens[j]):
                        assert ag[r][pos] == gins[j][i]
                        pos += 1
            m = [[int(x) for x in rng.integers(0, 4, size=R)] for _ in range(R)]
            ains = [_rand(dt, 41 + R, r, sum(m[r])) for r in range(R)]
            a2a = orc.alltoall(ains, m, dt)
            for j in range(R):
                pos = 0
                for r in range(R):
                    src = sum(m[r][:j])
                    for i in range(m[r][j]):
                        assert a2a[j][pos] == ains[r][src + i]
                        pos += 1


# ------------------------------------------------------ layout-pair semantics


def check_layout_pair_definition(orc):
    """The generic layout-pair definition reproduces each collective written out
    separately (two independent writings of the same placement rules), including
    strided regions (the Ulysses head partitions)."""
    for dt in ("fp32", "bf16"):
        R = 4
        lens = [3, 6, 0, 5]
        N = sum(lens)
        offs = [sum(lens[:k]) for k in range(R)]
        # AllGather(V): input r is one region named r; every output lists all names.
        gins = [_rand(dt, 51, r, lens[r]) for r in range(R)]
        lin = [[(r, 0, lens[r])] for r in range(R)]
        lout = [[(k, offs[k], lens[k]) for k in range(R)] for _ in range(R)]
        got = orc.collective("copy", dt, lin, lout, gins, [N] * R)
        want = orc.allgather(gins, dt)
        assert all(np.array_equal(a, b) for a, b in zip(got, want))
        # ReduceScatter(V)
        ins = [_rand(dt, 52, r, N) for r in range(R)]
        lin = [[(k, offs[k], lens[k]) for k in range(R)] for _ in range(R)]
        lout = [[(k, 0, lens[k])] for k in range(R)]
        got = orc.collective("sum", dt, lin, lout, ins, lens)
        want = orc.reducescatter(ins, lens, dt)
        assert all(np.array_equal(a, b) for a, b in zip(got, want))
        # AllReduce as one layout pair: every output names every partition.
        lout = [[(k, offs[k], lens[k]) for k in range(R)] for _ in range(R)]
        got = orc.collective("sum", dt, lin, lout, ins, [N] * R)
        want = orc.allreduce(ins, dt)
        assert all(np.array_equal(a, b) for a, b in zip(got, want))
        # AllToAll(V): names are (source, destination) pairs.
        m = [[(r + 2 * j) % 3 for j in range(R)] for r in range(R)]
        ains = [_rand(dt, 53, r, sum(m[r])) for r in range(R)]
        lin = [[(r * R + j, sum(m[r][:j]), m[r][j]) for j in range(R)] for r in range(R)]
        lout = [[(r * R + j, sum(m[rr][j] for rr in range(r)), m[r][j]) for r in range(R)]
                for j in range(R)]
        got = orc.collective("copy", dt, lin, lout, ains, [sum(m[r][j] for r in range(R)) for j in range(R)])
        want = orc.alltoall(ains, m, dt)
        assert all(np.array_equal(a, b) for a, b in zip(got, want))
        # Ulysses: source r's partition j is strided (S rows of hs*D, stride H*D).
        S, H, D = 3, 8, 2
        hs = H // R
        uins = [_rand(dt, 54, r, S * H * D) for r in range(R)]
        lin = [[(r * R + j, j * hs * D, hs * D, S, H * D) for j in range(R)] for r in range(R)]
        lout = [[(r * R + j, r * S * hs * D, S * hs * D) for r in range(R)] for j in range(R)]
        got = orc.collective("copy", dt, lin, lout, uins, [R * S * hs * D] * R)
        want = orc.ulysses_a2a(uins, S, H, D, dt)
        assert all(np.array_equal(a, b) for a, b in zip(got, want))


def check_layout_pair_rejects(orc):
    """Layout pairs that name no collective are refused."""
    x = [np.zeros(4, np.float32)] * 2
    bad = [
        ("copy", [[(0, 0, 4)], [(1, 0, 4)]], [[(2, 0, 4)], []]),            # name without a source
        ("copy", [[(0, 0, 4)], [(0, 0, 4)]], [[(0, 0, 4)], []]),            # COPY with two sources
        ("sum", [[(0, 0, 4)], [(1, 0, 4)]], [[(0, 0, 4)], []]),             # SUM without one per rank
        ("copy", [[(0, 0, 4)], [(1, 0, 4)]], [[(0, 0, 3)], []]),            # length mismatch
        ("sum", [[(0, 0, 2), (0, 2, 2)], []], [[(0, 0, 2)], []]),           # two sources on rank 0, none on 1
    ]
    for op, lin, lout in bad:
        try:
            orc.collective(op, "fp32", lin, lout, x, [4, 4])
        except ValueError:
            continue
        raise AssertionError(f"accepted an invalid layout pair: {op} {lin} {lout}")


# ------------------------------------------- fp16, 1-byte elements, maximum


def _as16(vals):
    return np.asarray(vals, dtype=np.float32).astype(np.float16).view(np.uint16)


def check_fp16_rounding_vs_torch(orc):
    """fp32 -> binary16 rounding equals PyTorch's CPU cast: every binary16 value,
    every midpoint between neighbours (exact ties), points just beside them,
    specials and a million random fp32 patterns."""
    import torch
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = h.view(np.float16).astype(np.float64)
    fin = np.isfinite(vals)
    v = np.sort(np.unique(vals[fin]))
    mids = (v[:-1] + v[1:]) / 2
    pts = np.concatenate([v, mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)).astype(np.float64),
                          np.nextafter(mids.astype(np.float32), np.float32(-np.inf)).astype(np.float64),
                          [65504.0, 65519.99, 65520.0, 65536.0, 1e30, 2.0 ** -25, 2.0 ** -26, 3 * 2.0 ** -26]])
    f = np.concatenate([pts.astype(np.float32), -pts.astype(np.float32)])
    rng = np.random.default_rng(6)
    f = np.concatenate([f, rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32).view(np.float32)])
    mine = orc.f32_to_f16(f)
    ref = torch.from_numpy(f.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.all(((mine[nan] & 0x7C00) == 0x7C00) & ((mine[nan] & 0x3FF) != 0))


def check_fp16_sums(orc):
    """fp16 sums: small integers are exact (numpy int64), and random sums stay
    within recursive-summation error plus one binary16 rounding of fp64."""
    R, n = 8, 4000
    ints = [synth.int_uniform_f32(8, r, n) for r in range(R)]
    exact = np.sum(np.stack([a.astype(np.int64) for a in ints]), axis=0)
    out = orc.allreduce([_as16(a) for a in ints], "fp16")[0]
    assert np.array_equal(out.view(np.float16).astype(np.int64), exact)
    rs = orc.reducescatter([_as16(a) for a in ints], [500] * R, "fp16")
    assert np.array_equal(rs[3].view(np.float16).astype(np.int64), exact[1500:2000])
    x = [_as16(synth.normal_f32(12, r, n)) for r in range(R)]
    xv = np.stack([a.view(np.float16).astype(np.float64) for a in x])
    ex = xv.sum(axis=0)
    gam = (R - 1) * 2.0 ** -24 / (1 - (R - 1) * 2.0 ** -24)
    err = gam * np.abs(xv).sum(axis=0)
    got = orc.allreduce(x, "fp16")[R - 1].view(np.float16).astype(np.float64)
    assert np.all(np.abs(got - ex) <= err + 2.0 ** -11 * (np.abs(ex) + err) + 2.0 ** -25)


def check_max(orc):
    """The maximum against numpy's maximum.reduce on data without zeros or NaN,
    the Figure 4 sentinels (rank 2 holds every maximum), and the rank-order
    rules for signed zeros and NaN."""
    for dt, conv in (("fp32", lambda a: a), ("bf16", lambda a: _as("bf16", a)), ("fp16", _as16)):
        R, n = 5, 3000
        raw = [synth.normal_f32(13, r, n) for r in range(R)]
        ins = [conv(a) for a in raw]
        vals = np.stack([(_vals(dt, a) if dt != "fp16" else a.view(np.float16).astype(np.float64)) for a in ins])
        want = np.maximum.reduce(vals, axis=0)
        got = orc.allreduce(ins, dt, op="max")[2]
        gotv = _vals(dt, got) if dt != "fp16" else got.view(np.float16).astype(np.float64)
        assert np.array_equal(gotv, want), dt
        lens = [600, 0, 1200, 1, 1199]
        rs = orc.reducescatter(ins, lens, dt, op="max")
        o = 0
        for k in range(R):
            gk = _vals(dt, rs[k]) if dt != "fp16" else rs[k].view(np.float16).astype(np.float64)
            assert np.array_equal(gk, want[o:o + lens[k]]), (dt, k)
            o += lens[k]
    g = load_golden("fig4_three_ranks.txt")
    ins = [_as("fp32", g["input"][r]) for r in range(3)]
    rs = orc.reducescatter(ins, [2, 2, 2], "fp32", op="max")
    assert [list(r) for r in rs] == [[20, 21], [22, 23], [24, 25]]
    z = [np.array([-0.0, 0.0, np.nan, 1.0], np.float32), np.array([0.0, -0.0, 7.0, np.nan], np.float32)]
    out = orc.allreduce(z, "fp32", op="max")[1]
    assert out.view(np.uint32)[0] == 0x80000000 and out.view(np.uint32)[1] == 0
    assert np.isnan(out[2]) and out[3] == 1.0


def check_one_byte_elements(orc):
    """1-byte (fp8) elements move bit for bit (numpy concatenate / split) and are never reduced."""
    R = 4
    rng = np.random.default_rng(14)
    lens = [5, 0, 17, 3]
    ins = [rng.integers(0, 256, size=n, dtype=np.uint8) for n in lens]
    for out in orc.allgather(ins, "fp8"):
        assert np.array_equal(out, np.concatenate(ins))
    m = [[(r + j) % 3 + r for j in range(R)] for r in range(R)]
    ins = [rng.integers(0, 256, size=sum(m[r]), dtype=np.uint8) for r in range(R)]
    pieces = [np.split(ins[r], np.cumsum(m[r])[:-1]) for r in range(R)]
    outs = orc.alltoall(ins, m, "fp8")
    for j in range(R):
        assert np.array_equal(outs[j], np.concatenate([pieces[r][j] for r in range(R)]))
    for call in (lambda: orc.allreduce(ins[:1], "fp8"), lambda: orc.reducescatter(ins[:1], [sum(m[0])], "fp8")):
        try:
            call()
        except ValueError:
            continue
        raise AssertionError("1-byte elements were reduced")
    try:
        orc.collective("sum", "fp8", [[(0, 0, 4)]], [[(0, 0, 4)]], [np.zeros(4, np.uint8)], [4])
    except ValueError:
        pass
    else:
        raise AssertionError("the layout-pair definition reduced 1-byte elements")


ALL_CHECKS = [
    check_fig4_golden,
    check_v_golden,
    check_integer_sums_exact,
    check_rank_order,
    check_fp64_error_bound,
    check_bf16_rounding_vs_torch,
    check_library_placements,
    check_ulysses_vs_numpy,
    check_invariants,
    check_single_rank_is_copy,
    check_bruteforce,
    check_layout_pair_definition,
    check_layout_pair_rejects,
    check_fp16_rounding_vs_torch,
    check_fp16_sums,
    check_max,
    check_one_byte_elements,
]
