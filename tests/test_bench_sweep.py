"""The benchmark sweep's host logic, on CPU: the launch form each collective
takes under the automatic policy (from the derived plan's stats) at the sizes
the sweep spans."""
import bench
from copy_reduce_datapath_gb300 import purlin as P


def workload_without_buffers():
    wl = bench.Workload.__new__(bench.Workload)
    wl.P = P
    wl._sweep = {}
    wl._lay = {}
    return wl


def test_sweep_launch_forms():
    wl = workload_without_buffers()
    names = ("allgather", "allreduce") + bench.SWEEP_OTHERS
    small = {n: wl.sweep_form(n, 1 << 10, 152) for n in names}
    assert set(small.values()) == {"inline"}, small
    mid = {n: wl.sweep_form(n, 1 << 20, 152) for n in names}
    assert set(mid.values()) == {"inline"}, mid
    full = {n: wl.sweep_form(n, 1 << 30, 152) for n in names}
    assert full == {"allgather": "bulk", "allreduce": "vector", "reducescatter": "inline", "alltoall": "bulk",
                    "allgatherv": "bulk", "reducescatterv": "vector", "alltoallv": "vector"}, full


def test_sweep_layouts_cover_the_partitions():
    """Every sweep layout at T bytes per rank covers T / 2 bf16 elements of each input."""
    wl = workload_without_buffers()
    T = (1 << 20)
    N = T // 2
    for name in bench.SWEEP_OTHERS:
        lin, lout, shape = wl._sweep_layouts(name, T)
        R_, parts = P.pl_layout_info(lin)
        assert R_ == bench.R and parts >= bench.R
        if name in ("reducescatter", "reducescatterv", "allgatherv"):
            assert sum(shape) == N
        else:
            assert all(sum(row) == N for row in shape)
