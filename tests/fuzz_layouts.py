"""Seeded random layout pairs for the fuzz tests (test infrastructure).

Each case is a valid collective specification (abstract: an input layout, an
output layout and a copy or a reduction) that the pages' rules accept:
  * a copy names every partition in exactly one input region and in one or
    more output regions;
  * a reduction names every partition in one region of every rank's input
    (R sources of one length) and in one or more output regions.
Regions sit at random element offsets with random gaps, so every alignment
occurs; some inputs are strided (rows x cols with a row stride), some
regions empty.  The same cases drive the host emulation of the derived work list and the GPU,
each against the oracle.  Nothing here computes a collective.
"""
from __future__ import annotations

import random

DTYPES = ("bf16", "fp16", "fp32", "fp8")


def _place(rng, sizes, max_gap):
    """Offsets of regions of the given sizes laid out one after another with
    random gaps; returns (offsets, total length)."""
    offs, pos = [], 0
    for n in sizes:
        pos += rng.randint(0, max_gap)
        offs.append(pos)
        pos += n
    return offs, pos + rng.randint(0, max_gap)


def case(seed: int):
    """One random case: a dict with R, dtype, op, the two layouts (per rank, a
    list of (name, offset, len[, rows, row_stride]) parts), the input and
    output buffer lengths, and a policy name."""
    rng = random.Random(seed)
    R = rng.choice([1, 2, 3, 4, 5, 8])
    dtype = rng.choice(DTYPES)
    op = "copy" if dtype == "fp8" else rng.choice(["copy", "sum", "sum", "max"])
    m = rng.randint(1, 2 * R)                       # partitions
    strided = rng.random() < 0.25
    lens, shapes = [], []
    for _ in range(m):
        if strided:
            rows, cols = rng.randint(1, 24), rng.randint(0, 300)
            shapes.append((rows, cols))
            lens.append(rows * cols)
        else:
            n = rng.choice([0, rng.randint(1, 40), rng.randint(1, 3000), rng.randint(3000, 40000)])
            shapes.append((1, n))
            lens.append(n)
    max_gap = rng.choice([0, 3, 17])

    def regions_in(rank_names, may_stride):
        """Parts of one buffer holding the partitions in rank_names, and its length."""
        if strided and may_stride and rank_names:
            # a row-major matrix whose column blocks are the partitions (rows padded
            # to the tallest partition), each partition a rows x cols block
            starts, col = [], rng.randint(0, max_gap)
            for k in rank_names:
                starts.append(col)
                col += shapes[k][1] + rng.randint(0, max_gap)
            stride = max(1, col + rng.randint(0, max_gap))
            parts = []
            for k, c0 in zip(rank_names, starts):
                rows, cols = shapes[k]
                parts.append((k, c0, cols, rows, stride) if rows > 1 else (k, c0, cols))
            height = max(shapes[k][0] for k in rank_names)
            return parts, stride * height
        offs, total = _place(rng, [lens[k] for k in rank_names], max_gap)
        return [(k, o, lens[k]) for k, o in zip(rank_names, offs)], total

    in_names = [[] for _ in range(R)]
    if op == "copy":
        for k in range(m):
            in_names[rng.randrange(R)].append(k)
    else:
        for r in range(R):
            in_names[r] = list(range(m))
            rng.shuffle(in_names[r])
    out_names = [[] for _ in range(R)]
    for k in range(m):
        for r in rng.sample(range(R), rng.randint(1, R)):
            out_names[r].append(k)
    for r in range(R):
        rng.shuffle(out_names[r])
    lin, in_sizes, lout, out_sizes = [], [], [], []
    for r in range(R):
        parts, n = regions_in(in_names[r], True)
        lin.append(parts)
        in_sizes.append(max(n, 1))
        # outputs stay one row per part: interleaved strided outputs would share
        # address ranges, which the library refuses as possible aliases
        parts, n = regions_in(out_names[r], False)
        lout.append(parts)
        out_sizes.append(max(n, 1))
    policy = rng.choice(["auto", "auto", "vector", "bulk", "inline", "staged", "composed", "notified",
                         "small_chunks", "few_ctas"])
    return {"seed": seed, "R": R, "dtype": dtype, "op": op, "lin": lin, "lout": lout,
            "in_sizes": in_sizes, "out_sizes": out_sizes, "policy": policy}


def policy(P, name):
    """The pl_policy of a case's policy name."""
    return {
        "auto": P.pl_policy_default(),
        "vector": P.pl_policy_default(datapath=P.PL_ATOM_VECTOR),
        "bulk": P.pl_policy_default(datapath=P.PL_ATOM_BULK, stages=3),
        "inline": P.pl_policy_default(datapath=P.PL_ATOM_INLINE),
        "staged": P.pl_policy_default(path=P.PL_PATH_STAGED, chunk_bytes=4096),
        "composed": P.pl_policy_default(allreduce_form=P.PL_AR_COMPOSED, chunk_bytes=2048),
        "notified": P.pl_policy_default(allreduce_form=P.PL_AR_NOTIFIED, chunk_bytes=2048),
        "small_chunks": P.pl_policy_default(chunk_bytes=512),
        "few_ctas": P.pl_policy_default(ctas=3),
    }[name]

