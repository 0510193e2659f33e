"""Random layout pairs (tests/fuzz_layouts.py): the derived work list, run by
the host emulation of concurrent CTAs, gives the oracle's outputs bit for bit
(unnamed output elements stay zero on both sides)."""
import numpy as np
import pytest

import oracle
import plan_interp
from copy_reduce_datapath_gb300 import purlin as P

import fuzz_layouts as F
from gpu_util import NP, host


@pytest.mark.parametrize("seed", range(48))
def test_random_layout_pair_emulated(seed):
    c = F.case(seed)
    R, dtype, op = c["R"], c["dtype"], c["op"]
    ins = [host("normal", dtype, 900 + seed, r, c["in_sizes"][r]) for r in range(R)]
    want = oracle.collective(op, dtype, c["lin"], c["lout"], ins, c["out_sizes"])
    lin, lout = P.pl_layout_create(R, c["lin"]), P.pl_layout_create(R, c["lout"])
    pl = P.pl_plan_create(lin, lout, op, dtype, R, F.policy(P, c["policy"]), num_sms=4, scratch_bytes=1 << 20)
    outs = [np.zeros(n, NP[dtype]) for n in c["out_sizes"]]
    plan_interp.run(pl, R, dtype, ins, outs, window=1 + seed % 7, seed=seed)
    for r in range(R):
        assert np.array_equal(outs[r].view(np.uint8), want[r].view(np.uint8)), f"seed {seed} rank {r} ({c['policy']})"
