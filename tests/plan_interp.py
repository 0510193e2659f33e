"""Host emulation of a derived SNAC work list (test infrastructure, no GPU).

Executes the items of a plan on numpy buffers the way concurrent CTAs would:
items are claimed in index order into a window of in-flight items, and the
phases of in-flight items (wait, read sources, write destinations, notify /
credit) interleave at random.  A wait may only pass when the flags allow it.
If the derived orchestration were wrong -- a slot reused before every
consumer read it, a consumer reading before the producer notified, a wait
that nothing satisfies -- the outputs would differ from the oracle's or the
emulation would stall, and the test fails.
"""
from __future__ import annotations

import random
from collections import defaultdict

import numpy as np
import torch

from copy_reduce_datapath_gb300 import purlin as P


def _to_f32(dtype, a):
    if dtype == "fp32":
        return a.astype(np.float32)
    if dtype == "fp16":
        return np.ascontiguousarray(a, np.uint16).view(np.float16).astype(np.float32)
    return (a.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _from_f32(dtype, a):
    if dtype == "fp32":
        return a.astype(np.float32)
    if dtype == "fp16":
        return np.ascontiguousarray(a, np.float32).astype(np.float16).view(np.uint16)
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


NPDT = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.float32, "fp8": np.uint8}


class Stall(AssertionError):
    pass


def load_plan(plan):
    st = P.pl_plan_get_stats(plan)
    items = [P.pl_plan_get_item(plan, i) for i in range(st.items)]
    return st, items


def _index(ref, rows, cols):
    r = np.arange(rows, dtype=np.int64)[:, None]
    c = np.arange(cols, dtype=np.int64)[None, :]
    return (ref.offset + r * ref.stride + c).ravel()


def run(plan, R, dtype, ins, outs, *, window=1, seed=0):
    """Execute `plan` over numpy buffers `ins`/`outs` (modified in place)."""
    st, items = load_plan(plan)
    npdt = NPDT[dtype]
    scratch = np.zeros(max(1, R * st.slots * st.slot_elems), dtype=npdt)
    space = {P.PL_SPACE_IN: ins, P.PL_SPACE_OUT: outs, P.PL_SPACE_SCRATCH: [scratch]}
    full = defaultdict(int)
    done = defaultdict(int)
    count = defaultdict(int)
    rng = random.Random(seed)

    def can_wait(syncs, nwait):
        for s in syncs[:nwait]:
            tagged = s.use + 1
            if s.type == P.PL_SYNC_WAIT_FULL and full[s.flag] < tagged:
                return False
            if s.type == P.PL_SYNC_WAIT_FREE and done[s.flag] < tagged:
                return False
        return True

    def read(it, refs):
        vals = []
        for ref in refs[:it.nsrc]:
            buf = space[ref.space][ref.index]
            vals.append(buf[_index(ref, it.rows, it.cols)].copy())
        if it.nsrc == 1:
            return vals[0]
        assert dtype != "fp8", "a reduction of one-byte elements"
        acc = _to_f32(dtype, vals[0])
        for v in vals[1:]:
            x = _to_f32(dtype, v)
            if it.op == 2:  # maximum: the later rank's value only when greater
                acc = np.where(x > acc, x, acc).astype(np.float32)
            else:
                acc = (acc + x).astype(np.float32)
        return _from_f32(dtype, acc)

    def write(it, refs, data):
        dsts = refs[it.nsrc:]
        if it.kind == P.PL_ITEM_COMPOSE:
            # Figure 6 at vector grain: destination 0 (the owner) first; the
            # others receive what is read back from it
            own = space[dsts[0].space][dsts[0].index]
            idx = _index(dsts[0], it.rows, it.cols)
            own[idx] = data
            data = own[idx].copy()
            dsts = dsts[1:]
        for ref in dsts:
            buf = space[ref.space][ref.index]
            buf[_index(ref, it.rows, it.cols)] = data

    def post(it, syncs):
        for s in syncs[it.nwait:]:
            if s.type == P.PL_SYNC_NOTIFY:
                full[s.flag] = max(full[s.flag], s.use + 1)
            elif s.type == P.PL_SYNC_CREDIT:
                count[s.flag] += 1
                if count[s.flag] == s.count:
                    count[s.flag] = 0
                    done[s.flag] = max(done[s.flag], s.use + 1)

    nxt = 0
    inflight = []  # [phase, item, refs, syncs, data]
    while nxt < len(items) or inflight:
        choices = []
        if nxt < len(items) and len(inflight) < window:
            choices.append("claim")
        for k, f in enumerate(inflight):
            if f[0] != "wait" or can_wait(f[3], f[1].nwait):
                choices.append(k)
        if not choices:
            raise Stall(f"no in-flight item can progress (next={nxt}, window={window})")
        c = rng.choice(choices)
        if c == "claim":
            it, refs, syncs = items[nxt]
            inflight.append(["wait", it, refs, syncs, None])
            nxt += 1
            continue
        f = inflight[c]
        if f[0] == "wait":
            f[0] = "read"
        elif f[0] == "read":
            f[4] = read(f[1], f[2])
            f[0] = "write"
        elif f[0] == "write":
            write(f[1], f[2], f[4])
            f[0] = "post"
        else:
            post(f[1], f[3])
            inflight.pop(c)
    return outs
