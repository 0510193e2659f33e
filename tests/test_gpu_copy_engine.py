"""The copy-engine AllGather (one device-to-device memcpy per source and
destination pair, no kernel: the route the pages' copy-engine AllGather
baseline takes) against the oracle, element by element.  The benchmark times
this route beside the library's AllGather kernel."""
import pytest
import torch

import bench
import oracle
import synth

from gpu_util import assert_equal, host, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "fp32", "fp8"])
@pytest.mark.parametrize("n", [1, 1000, (1 << 18) + 5])
def test_copy_engine_allgather_matches_oracle(dtype, n):
    torch.cuda.set_device(0)
    R = 8
    ins_h = [host(None if dtype == "fp8" else "normal", dtype, 70, r, n) for r in range(R)]
    ins = [to_dev(a, dtype) for a in ins_h]
    outs = [torch.zeros(n * R, dtype=ins[0].dtype, device="cuda") for _ in range(R)]
    bench.copy_engine_allgather(ins, outs, n)
    torch.cuda.synchronize()
    want = oracle.allgather(ins_h, dtype)
    for r in range(R):
        assert_equal(to_np(outs[r], dtype), want[r], f"rank {r}")
