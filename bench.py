"""Benchmark of the Purlin collectives' data path on one GB300 (and N replicas).

One step = AllGather(T) then AllReduce(T) over R = 8 logical ranks held in one
GPU's memory, bf16 inputs ~ N(0, 1) (seed 1), equal partitions, T = 1 GiB per
collective (the 8-rank AllGather / AllReduce workload at its largest size).
Reported value: algorithm bandwidth of the step, (T_AG + T_AR) / step time, in
GB/s (1 GB = 1e9 bytes), summed over replicas when run on N GPUs.

Also reported on the same line:
  - sweep: latency (us) and algbw (GB/s) of every collective (AllGather, AllReduce, ReduceScatter,
    AllToAll and the three V forms) for T = 1 KiB .. 1 GiB
  - roofline: the dominant kernel (the AllReduce launch) against the measured HBM copy peak
  - e2e: the same step through the C ABI with host buffers (pinned), copies inside the timing
  - cpu_baseline: the CPU oracle on a bounded sample of the same workload
  - clocks: SM clock samples taken during the timed region

`--impl reference` times the CPU oracle instead (the only reference this build has).
Under torchrun (WORLD_SIZE > 1) every rank runs an independent replica on its own
GPU (the method shards no data across GPUs); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

R = 8
SEED = 1
GiB = 1 << 30
METRIC = "algbw GB/s (AllGather + AllReduce, R=8 logical ranks, bf16, T=1 GiB each)"
UNIT = "GB/s"
ORACLE_SAMPLE_T = 128 << 20    # bytes per collective in the CPU-baseline sample (about 10-15 s)
REFERENCE_SAMPLE_T = 64 << 20  # bytes per collective per reference-arm step (0.2 s on 16 Grace cores)
REFERENCE_BUDGET_S = 120.0     # timed reference steps stop once they have taken this long


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--T", type=int, default=GiB, help="bytes per collective")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--case", default=None, choices=sorted(CASES),
                    help="time one collective of the other workloads instead of the step (prints its own line)")
    ap.add_argument("--policy", default="", help="policy overrides for --case, e.g. path=2,chunk_bytes=262144")
    ap.add_argument("--scratch", type=int, default=1 << 30,
                    help="scratch ring bytes of the context for --case with the staged path (path=2)")
    ap.add_argument("--depth-sweep", action="store_true",
                    help="Atom copy of 256 MiB: bandwidth vs CTA count and bulk-ring depth (prints its own line)")
    ap.add_argument("--copy-engine", action="store_true",
                    help="AllGather by one device-to-device memcpy per (source, destination) pair, beside the kernel")
    ap.add_argument("--policy-sweep", action="store_true",
                    help="automatic chunk size against fixed chunk sizes, AllGather and AllReduce, T = 1 MiB .. 1 GiB")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("atom_impl.cuh", "atom.cu", "snac.h"):
        with open(os.path.join(ROOT, "copy_reduce_datapath_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; otherwise None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("kernel_source") != kernel_source_hash():
        return None
    return e.get("bytes_per_launch")


def committed_traffic_note(kernel: str):
    """How the committed DRAM traffic figure was taken (None when it is not
    valid for the current kernel source)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if committed_traffic(kernel) is None:
        return None
    with open(p) as f:
        return json.load(f)[kernel].get("note")


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.rows = []
        self.proc = None
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        rows = [r for r in self.rows if self.uuid is None or r[1] == self.uuid or r[1].endswith(self.uuid)]
        if not rows:
            rows = self.rows
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[6 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(ms: float, ws: int, device) -> float:
    """The slowest rank's time (the job's time) when N replicas run side by side."""
    if ws <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(ms_total_max: float, steps: int, T: int, ws: int):
    """(ms per step, whole-job algbw in GB/s): every replica moves 2*T bytes of
    collective payload (AllGather + AllReduce) per step."""
    ms_step = ms_total_max / steps
    return ms_step, ws * 2 * T / (ms_step * 1e-3) / 1e9


# ----------------------------------------------------------- our arm (GPU)


class Workload:
    """Device buffers of one replica: AllGather and AllReduce at T bytes each."""

    def __init__(self, T: int, device):
        import torch
        import synth
        from copy_reduce_datapath_gb300 import purlin as P
        self.P = P
        self.T = T
        self.n_ag = T // 2 // R           # elements each rank contributes to the AllGather
        self.n_ar = T // 2                # elements per rank of the AllReduce
        self.ag_in = [synth.device_normal_bf16(SEED, r, self.n_ag, device) for r in range(R)]
        self.ag_out = [torch.empty(self.n_ag * R, dtype=torch.bfloat16, device=device) for _ in range(R)]
        self.ar_in = [synth.device_normal_bf16(SEED, 100 + r, self.n_ar, device) for r in range(R)]
        self.ar_out = [torch.empty(self.n_ar, dtype=torch.bfloat16, device=device) for _ in range(R)]
        lens = [self.n_ag] * R
        self.ag_lin = P.pl_layout_rank_owned(R, lens)
        self.ag_lout = P.pl_layout_partitioned(R, lens)
        self._lay = {}    # AllGather layouts per element count
        self._sweep = {}  # the other collectives' layouts per (name, T)

    def allgather(self, ctx, stream, n=None, ins=None, outs=None):
        P = self.P
        ins = ins or self.ag_in
        outs = outs or self.ag_out
        if n is None:
            P.pl_collective(ctx, self.ag_lin, self.ag_lout, "copy", "bf16", R, P.ptrs(ins), P.counts(ins),
                            P.ptrs(outs), P.counts(outs), None, stream)
        else:
            lin = self._layouts(n)
            P.pl_collective(ctx, lin[0], lin[1], "copy", "bf16", R, P.ptrs(ins), [n] * R, P.ptrs(outs),
                            [n * R] * R, None, stream)

    def allreduce(self, ctx, stream, n=None, ins=None, outs=None):
        P = self.P
        P.pl_allreduce(ctx, "bf16", R, self.n_ar if n is None else n, P.ptrs(ins or self.ar_in),
                       P.ptrs(outs or self.ar_out), None, stream)

    def _layouts(self, n):
        if n not in self._lay:
            self._lay[n] = (self.P.pl_layout_rank_owned(R, [n] * R), self.P.pl_layout_partitioned(R, [n] * R))
        return self._lay[n]

    # The other collectives of the sweep, at T bytes per rank (the conventions
    # of their algbw: ReduceScatter(V) and AllToAll(V) input bytes per rank,
    # AllGatherV output bytes per rank), over the AllReduce's buffers (and, for
    # the AllToAllV's column sums, buffers of their own).  V forms: Zipf
    # s = 0.125 lengths, seed 4.
    def _sweep_layouts(self, name, T):
        import synth
        P = self.P
        key = (name, T)
        if key not in self._sweep:
            N = T // 2
            if name == "reducescatter":
                lens = [N // R] * R
                self._sweep[key] = (P.pl_layout_partitioned(R, lens), P.pl_layout_rank_owned(R, lens), lens)
            elif name == "alltoall":
                m = [[N // R] * R for _ in range(R)]
                self._sweep[key] = (P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m), m)
            elif name in ("allgatherv", "reducescatterv"):
                lens = synth.zipf_lengths(N, R, 0.125, seed=4)
                lo, lp = P.pl_layout_rank_owned(R, lens), P.pl_layout_partitioned(R, lens)
                self._sweep[key] = (lo, lp, lens) if name == "allgatherv" else (lp, lo, lens)
            else:
                m = synth.zipf_matrix(N, R, 0.125, seed=4)
                self._sweep[key] = (P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m), m)
        return self._sweep[key]

    def sweep_call(self, name, T, ctx, stream):
        """A closure that launches collective `name` at T bytes per rank on `stream`."""
        import torch
        P = self.P
        N = T // 2
        lin, lout, shape = self._sweep_layouts(name, T)
        if name in ("reducescatter", "reducescatterv"):
            ins, outs = self.ar_in, [o[: shape[r]] for r, o in enumerate(self.ar_out)]
            cin, cout, op = [N] * R, list(shape), "sum"
        elif name == "allgatherv":
            ins, outs = [x[: shape[r]] for r, x in enumerate(self.ar_in)], self.ag_out
            cin, cout, op = list(shape), [N] * R, "copy"
        else:
            cols = [sum(shape[j][r] for j in range(R)) for r in range(R)]
            if name == "alltoall":
                outs = self.ar_out
            else:
                if not hasattr(self, "a2av_out") or self.a2av_out[0].numel() < max(cols):
                    self.a2av_out = [torch.empty(max(cols), dtype=torch.bfloat16, device=self.ar_in[0].device)
                                     for _ in range(R)]
                outs = self.a2av_out
            ins, cin, cout, op = self.ar_in, [N] * R, cols, "copy"
        pi, po = P.ptrs(ins), P.ptrs(outs)
        return lambda: P.pl_collective(ctx, lin, lout, op, "bf16", R, pi, cin, po, cout, None, stream)

    def sweep_form(self, name, T, num_sms):
        """The launch form the automatic policy takes for collective `name` at T
        bytes per rank (host-side plan derivation; 16-byte aligned buffers)."""
        import synth
        P = self.P
        if name == "allgather":
            lin, lout = self._layouts(T // 2 // R)
            op = "copy"
        elif name == "allreduce":
            key = ("allreduce", T)
            if key not in self._sweep:
                L = P.pl_layout_partitioned(R, synth.equal_lengths(T // 2, R))
                self._sweep[key] = (L, L, None)
            lin, lout, _ = self._sweep[key]
            op = "sum"
        else:
            lin, lout, _ = self._sweep_layouts(name, T)
            op = "sum" if name in ("reducescatter", "reducescatterv") else "copy"
        plan = P.pl_plan_create(lin, lout, op, "bf16", R, None, num_sms)
        try:
            st = P.pl_plan_get_stats(plan)
        finally:
            P.pl_plan_destroy(plan)
        return {P.PL_ATOM_INLINE: "inline", P.PL_ATOM_BULK: "bulk", P.PL_ATOM_VECTOR: "vector"}.get(st.datapath, "?")


def sampled_parity(wl, device):
    """Windows of the full-size outputs against the oracle on the same input windows."""
    import numpy as np
    import torch
    import oracle
    rng = np.random.default_rng(0)

    def h(t):
        return t.cpu().view(torch.int16).numpy().view(np.uint16)

    bad = 0
    w = 4096
    for _ in range(4):
        i = int(rng.integers(0, wl.n_ar - w))
        want = oracle.allreduce([h(x[i:i + w]) for x in wl.ar_in], "bf16")
        for r in (0, R - 1):
            bad += int(not np.array_equal(h(wl.ar_out[r][i:i + w]), want[r]))
        j = int(rng.integers(0, R))
        k = int(rng.integers(0, wl.n_ag - w))
        src = h(wl.ag_in[j][k:k + w])
        for r in (0, R - 1):
            off = j * wl.n_ag + k
            bad += int(not np.array_equal(h(wl.ag_out[r][off:off + w]), src))
    return bad == 0


SWEEP_OTHERS = ("reducescatter", "alltoall", "allgatherv", "reducescatterv", "alltoallv")


# Algorithmic HBM bytes of each swept collective at T bytes (per the T
# convention of each: AllGather(V) output per rank, ReduceScatter(V) and
# AllToAll(V) input per rank, AllReduce buffer per rank).
SWEEP_MOVED = {"allgather": R + 1, "allreduce": 2 * R, "reducescatter": R + 1, "alltoall": 2 * R,
               "allgatherv": R + 1, "reducescatterv": R + 1, "alltoallv": 2 * R}


def time_sweep(ctx, wl, stream, torch, peak):
    """Latency, algbw and fraction of the copy peak per size and collective
    (R = 8, bf16; V forms with Zipf lengths).  Up to 64 MiB each point is a
    CUDA graph of `calls` launches replayed on the launch stream (device time
    per call, no host launch overhead); above that, events around back-to-back
    calls."""
    out = []
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    for e in range(10, 31):
        T = 1 << e
        if T > wl.T:
            break
        row = {"T": T}
        for name in ("allgather", "allreduce"):
            n = T // 2 // R if name == "allgather" else T // 2
            fn = getattr(wl, name)
            us, how = time_call(lambda: fn(ctx, stream.cuda_stream, n), T, stream, torch)
            row[name] = point(us, T, SWEEP_MOVED[name] * T, peak, how, wl.sweep_form(name, T, sms))
        for name in SWEEP_OTHERS:
            us, how = time_call(wl.sweep_call(name, T, ctx, stream.cuda_stream), T, stream, torch)
            row[name] = point(us, T, SWEEP_MOVED[name] * T, peak, how, wl.sweep_form(name, T, sms))
        out.append(row)
    return out


def time_call(call, T, stream, torch):
    """Mean device time of one `call` (which launches on `stream`) after 3
    warm-ups: up to 64 MiB from a CUDA graph of 10-50 calls replayed 5 times
    (no host launch overhead), above that from events around 5 calls."""
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    if T <= (64 << 20):
        calls = 50 if T <= (4 << 20) else 10
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(calls):
                call()
        with torch.cuda.stream(stream):
            g.replay()
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * calls), "graph"
    a.record(stream)
    for _ in range(reps):
        call()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / reps, "events"


def plan_form(P, lin, lout, op, dtype, Rr, num_sms):
    """The launch form the automatic policy takes for a layout pair (host-side
    plan derivation; 16-byte aligned buffers)."""
    plan = P.pl_plan_create(lin, lout, op, dtype, Rr, None, num_sms)
    try:
        st = P.pl_plan_get_stats(plan)
    finally:
        P.pl_plan_destroy(plan)
    return {P.PL_ATOM_INLINE: "inline", P.PL_ATOM_BULK: "bulk", P.PL_ATOM_VECTOR: "vector"}.get(st.datapath, "?")


def plan_bytes(P, lin, lout, op, dtype, Rr, pol, num_sms, scratch):
    """Device bytes one launch of the plan reads and writes (its own bytes:
    staging and rereads included)."""
    plan = P.pl_plan_create(lin, lout, op, dtype, Rr, pol, num_sms, scratch)
    try:
        st = P.pl_plan_get_stats(plan)
    finally:
        P.pl_plan_destroy(plan)
    return int(st.bytes_read + st.bytes_written)


def point(us, T, moved, peak, how, form=None):
    """One timed point: latency, algbw (T / time), algorithmic HBM bandwidth
    and its fraction of the copy peak."""
    d = {"us": round(us, 3), "algbw_GBps": round(T / (us * 1e-6) / 1e9, 2),
         "hbm_GBps": round(moved / (us * 1e-6) / 1e9, 1), "frac_of_peak": round(moved / (us * 1e-6) / 1e9 / peak, 4),
         "timed": how}
    if form:
        d["form"] = form
    return d


def copy_engine_allgather(ins, outs, n):
    """AllGather of n elements per rank by one device-to-device copy per
    (source, destination) pair on the current stream: the copy-engine route,
    which launches no kernel (the reference line beside the library's
    AllGather kernel)."""
    R_ = len(ins)
    for r in range(R_):
        for j in range(R_):
            outs[r][j * n:(j + 1) * n].copy_(ins[j][:n], non_blocking=True)


def time_configs(ctx, wl, stream, torch, peak):
    """The other workloads of the benchmark's configuration list, timed by the
    same rules as the sweep (graphs up to 64 MiB, events above), each with its
    algorithmic bytes against the copy peak:
      - three-rank fp32 AllReduce of integers in [-8, 8]: 3 x 4096 elements per
        rank (latency), and scaled up to 1 GiB per rank;
      - ReduceScatter, R = 8, fp32 and bf16 U(-1,1), T = 1 MiB .. 1 GiB per rank,
        zero-staging out of place and in place (rank k's output is partition k
        of its own input);
      - AllToAll shaped like MoE token dispatch ([4096, 7168] bf16 per rank, 8
        token groups) and the Ulysses sequence-to-head swap ([16384, 32, 128]
        bf16 per rank);
      - the copy-engine AllGather (one memcpy per source and destination pair,
        no kernel) beside the library's AllGather at 64 MiB and 1 GiB;
      - the AllReduce of the benchmark (R = 8, bf16) in its three forms at
        64 MiB, 128 MiB and 1 GiB: fused, composed at vector grain and composed
        per chunk with a Notify (Figure 6), each against the fused form's
        algorithmic bytes (16T) and with the plan's own bytes;
      - the staged SNAC path (Stage, Notify, Consume through a scratch ring) at
        128 MiB and 1 GiB: ReduceScatter and the fused and composed AllReduce,
        each against its plan's own bytes (staging included).
    The Zipf V forms are in the sweep."""
    import synth
    P = wl.P
    dev = wl.ar_in[0].device
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    s = stream.cuda_stream
    out = {}

    # three ranks, fp32 integers
    r3 = {}
    for label, n in (("3x4096", 3 * 4096), ("1GiB", GiB // 4)):
        ins = [synth.device_int_f32(0, r, n, dev) for r in range(3)]
        outs = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(3)]
        L = P.pl_layout_partitioned(3, synth.equal_lengths(n, 3))
        pi, po = P.ptrs(ins), P.ptrs(outs)
        us, how = time_call(lambda: P.pl_allreduce(ctx, "fp32", 3, n, pi, po, None, s), n * 4, stream, torch)
        r3[label] = point(us, n * 4, 2 * 3 * n * 4, peak, how, plan_form(P, L, L, "sum", "fp32", 3, sms))
        P.pl_layout_destroy(L)
        del ins, outs
    out["allreduce_r3_fp32_int"] = r3

    # ReduceScatter sweep, fp32 and bf16, out of place and in place
    rs = []
    for dt, tdt, S in (("fp32", torch.float32, 4), ("bf16", torch.bfloat16, 2)):
        ins = [synth.device_uniform_pm1(2, r, GiB // S, dev, tdt) for r in range(R)]
        outs = [torch.empty(GiB // S // R, dtype=tdt, device=dev) for _ in range(R)]
        for e in range(20, 31):
            T = 1 << e
            N = T // S
            lens = [N // R] * R
            lin = P.pl_layout_partitioned(R, lens)
            for variant in ("out_of_place", "in_place"):
                if variant == "in_place":
                    lout, po, cout = P.pl_layout_rank_owned_inplace(R, lens), P.ptrs(ins), [N] * R
                else:
                    lout, po, cout = P.pl_layout_rank_owned(R, lens), P.ptrs(outs), lens
                pi = P.ptrs(ins)
                call = lambda: P.pl_collective(ctx, lin, lout, "sum", dt, R, pi, [N] * R, po, cout, None, s)  # noqa: E731
                us, how = time_call(call, T, stream, torch)
                rs.append({"T": T, "dtype": dt, "variant": variant,
                           **point(us, T, (R + 1) * T, peak, how, plan_form(P, lin, lout, "sum", dt, R, sms))})
                P.pl_layout_destroy(lout)
            P.pl_layout_destroy(lin)
        del ins, outs
    out["reducescatter"] = rs

    # AllToAll: MoE token dispatch and the Ulysses swap
    a2a = {}
    n = 4096 * 7168
    m = [[n // R] * R for _ in range(R)]
    shapes = (("moe_4096x7168", P.pl_layout_alltoall_in(R, m), P.pl_layout_alltoall_out(R, m), n),
              ("ulysses_16384x32x128", P.pl_layout_ulysses_in(R, 16384, 32, 128),
               P.pl_layout_ulysses_out(R, 16384, 32, 128), 16384 * 32 * 128))
    for name, lin, lout, n in shapes:
        ins = [synth.device_normal_bf16(3, r, n, dev) for r in range(R)]
        outs = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        pi, po = P.ptrs(ins), P.ptrs(outs)
        call = lambda: P.pl_collective(ctx, lin, lout, "copy", "bf16", R, pi, [n] * R, po, [n] * R, None, s)  # noqa: E731
        us, how = time_call(call, n * 2, stream, torch)
        a2a[name] = point(us, n * 2, 2 * R * n * 2, peak, how, plan_form(P, lin, lout, "copy", "bf16", R, sms))
        P.pl_layout_destroy(lin)
        P.pl_layout_destroy(lout)
        del ins, outs
    out["alltoall"] = a2a

    # copy-engine AllGather against the kernel (the benchmark's AllGather buffers)
    ce = []
    for T in (64 << 20, wl.T):
        n = T // 2 // R
        ins, outs = wl.ag_in, wl.ag_out

        def by_memcpy():
            with torch.cuda.stream(stream):
                copy_engine_allgather(ins, outs, n)
        us_m, how_m = time_call(by_memcpy, T, stream, torch)
        us_k, how_k = time_call(lambda: wl.allgather(ctx, s, n), T, stream, torch)
        moved = (R + 1) * T
        ce.append({"T": T, "memcpy_per_pair": point(us_m, T, moved, peak, how_m),
                   "kernel": point(us_k, T, moved, peak, how_k, wl.sweep_form("allgather", T, sms))})
    out["copy_engine_allgather"] = ce

    # the AllReduce forms on the benchmark's AllReduce buffers
    forms = {"fused": P.PL_AR_FUSED, "composed": P.PL_AR_COMPOSED, "notified": P.PL_AR_NOTIFIED}
    arf = []
    for T in (64 << 20, 128 << 20, wl.T):
        n = T // 2
        L = P.pl_layout_partitioned(R, synth.equal_lengths(n, R))
        pi, po = P.ptrs(wl.ar_in), P.ptrs(wl.ar_out)
        for name, form in forms.items():
            pol = P.pl_policy_default(allreduce_form=form)
            us, how = time_call(lambda: P.pl_allreduce(ctx, "bf16", R, n, pi, po, pol, s), T, stream, torch)
            own = plan_bytes(P, L, L, "sum", "bf16", R, pol, sms, 0)
            arf.append({"T": T, "form": name, "plan_bytes": own, "own_frac": round(own / (us * 1e-6) / 1e9 / peak, 4),
                        **point(us, T, 2 * R * T, peak, how)})
        P.pl_layout_destroy(L)
    out["allreduce_forms"] = arf

    # the staged path, with a context that owns a scratch ring
    scratch = GiB
    sctx = P.pl_ctx_create(dev.index or 0, scratch)
    staged = []
    try:
        for T in (128 << 20, wl.T):
            n = T // 2
            lens = synth.equal_lengths(n, R)
            L = P.pl_layout_partitioned(R, lens)
            lo = P.pl_layout_rank_owned(R, lens)
            pi, po = P.ptrs(wl.ar_in), P.ptrs(wl.ar_out)
            cases = (("reducescatter", lo, P.pl_policy_default(path=P.PL_PATH_STAGED), (R + 1) * T),
                     ("allreduce_fused", L, P.pl_policy_default(path=P.PL_PATH_STAGED), 2 * R * T),
                     ("allreduce_composed", L, P.pl_policy_default(path=P.PL_PATH_STAGED,
                                                                   allreduce_form=P.PL_AR_COMPOSED), 2 * R * T))
            for name, lout, pol, alg in cases:
                cout = lens if lout is lo else [n] * R
                call = lambda: P.pl_collective(sctx, L, lout, "sum", "bf16", R, pi, [n] * R, po, cout, pol, s)  # noqa: E731
                us, how = time_call(call, T, stream, torch)
                own = plan_bytes(P, L, lout, "sum", "bf16", R, pol, sms, scratch)
                staged.append({"T": T, "collective": name, "plan_bytes": own,
                               "algorithmic_frac": round(alg / (us * 1e-6) / 1e9 / peak, 4),
                               **point(us, T, own, peak, how)})
            P.pl_layout_destroy(L)
            P.pl_layout_destroy(lo)
        torch.cuda.synchronize()
        assert P.pl_ctx_status(sctx, s) == P.PL_OK
    finally:
        P.pl_ctx_destroy(sctx)
    out["staged"] = staged
    out["note"] = ("points up to 64 MiB replay a CUDA graph on the same buffers back to back, so below the L2 size "
                   "(129 MB of working set) they measure latency and L2 bandwidth, and frac_of_peak can exceed 1; "
                   "from 128 MiB up, events around back-to-back calls on buffers larger than L2")
    torch.cuda.synchronize()
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    return out


def run_e2e(ctx, wl, stream, torch, steps):
    """The step through the C ABI with host (pinned) buffers: every step copies
    every input host->device and every output device->host, inside the timed
    region.  Copies in, collectives and copies out run on three streams, so the
    two directions of the host link overlap (within a step and across steps);
    events keep every buffer from being overwritten while it is still read."""
    pin = dict(dtype=torch.bfloat16, pin_memory=True)
    h_ag_in = [torch.empty(wl.n_ag, **pin) for _ in range(R)]
    h_ar_in = [torch.empty(wl.n_ar, **pin) for _ in range(R)]
    h_ag_out = [torch.empty(wl.n_ag * R, **pin) for _ in range(R)]
    h_ar_out = [torch.empty(wl.n_ar, **pin) for _ in range(R)]
    for h, d in zip(h_ag_in + h_ar_in, wl.ag_in + wl.ar_in):
        h.copy_(d)
    torch.cuda.synchronize()
    s_in, s_out, cmp = torch.cuda.Stream(), torch.cuda.Stream(), stream

    def step(prev):
        with torch.cuda.stream(s_in):
            if prev:
                s_in.wait_event(prev["ag_k"])  # the last AllGather has read its inputs
            for h, d in zip(h_ag_in, wl.ag_in):
                d.copy_(h, non_blocking=True)
            e_ag_in = s_in.record_event()
            if prev:
                s_in.wait_event(prev["ar_k"])
            for h, d in zip(h_ar_in, wl.ar_in):
                d.copy_(h, non_blocking=True)
            e_ar_in = s_in.record_event()
        cmp.wait_event(e_ag_in)
        if prev:
            cmp.wait_event(prev["ag_out"])  # the last AllGather output has reached the host
        wl.allgather(ctx, cmp.cuda_stream)
        e_ag_k = cmp.record_event()
        cmp.wait_event(e_ar_in)
        if prev:
            cmp.wait_event(prev["ar_out"])
        wl.allreduce(ctx, cmp.cuda_stream)
        e_ar_k = cmp.record_event()
        with torch.cuda.stream(s_out):
            s_out.wait_event(e_ag_k)
            for h, d in zip(h_ag_out, wl.ag_out):
                h.copy_(d, non_blocking=True)
            e_ag_out = s_out.record_event()
            s_out.wait_event(e_ar_k)
            for h, d in zip(h_ar_out, wl.ar_out):
                h.copy_(d, non_blocking=True)
            e_ar_out = s_out.record_event()
        return {"ag_k": e_ag_k, "ar_k": e_ar_k, "ag_out": e_ag_out, "ar_out": e_ar_out}

    step(None)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    prev = None
    for _ in range(steps):
        prev = step(prev)
    s_out.wait_event(prev["ar_out"])
    b.record(s_out)
    b.synchronize()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    h2d = R * (wl.n_ag + wl.n_ar) * 2
    d2h = R * (wl.n_ag * R + wl.n_ar) * 2
    return {"value": round(2 * wl.T / (ms * 1e-3) / 1e9, 2), "unit": UNIT, "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "buffers": "pinned host memory; copies in, collectives and copies out on three streams"}


def oracle_inputs_host(T_sample: int):
    """Bounded-sample inputs for the oracle, drawn on the host (reference arm)."""
    import numpy as np
    import torch
    import synth
    n_ag, n_ar = T_sample // 2 // R, T_sample // 2
    conv = lambda t: t.view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    ag = [conv(synth.host_normal_bf16_torch(SEED, r, n_ag)) for r in range(R)]
    ar = [conv(synth.host_normal_bf16_torch(SEED, 100 + r, n_ar)) for r in range(R)]
    return ag, ar


def oracle_inputs_from_device(wl, T_sample: int):
    """The first T_sample bytes' worth of the benchmark's own device inputs."""
    import numpy as np
    import torch
    n_ag, n_ar = T_sample // 2 // R, T_sample // 2
    conv = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    return [conv(x[:n_ag]) for x in wl.ag_in], [conv(x[:n_ar]) for x in wl.ar_in]


def oracle_time(ag, ar, threads=1):
    """Seconds the C oracle takes for one AllGather + AllReduce.  With threads > 1
    the element range is cut into that many slices and the unchanged oracle runs
    on each slice in its own thread (the C calls release the GIL): the same work,
    spread over the host cores."""
    import oracle
    if threads <= 1:
        t0 = time.perf_counter()
        oracle.allgather(ag, "bf16")
        oracle.allreduce(ar, "bf16")
        return time.perf_counter() - t0
    from concurrent.futures import ThreadPoolExecutor

    def cuts(n):
        return [(n * i // threads, n * (i + 1) // threads) for i in range(threads)]

    def work(i):
        a0, a1 = cuts(ag[0].size)[i]
        b0, b1 = cuts(ar[0].size)[i]
        oracle.allgather([x[a0:a1] for x in ag], "bf16")
        oracle.allreduce([x[b0:b1] for x in ar], "bf16")

    oracle.default()  # build and load before the clock starts
    with ThreadPoolExecutor(threads) as ex:
        t0 = time.perf_counter()
        list(ex.map(work, range(threads)))
        return time.perf_counter() - t0


def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def cpu_baseline_line(wl, T_sample):
    ag, ar = oracle_inputs_from_device(wl, T_sample)
    cores = host_cores()
    dt1 = oracle_time(ag, ar)
    dt = oracle_time(ag, ar, cores)
    return {"value": round(2 * T_sample / dt / 1e9, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "single_thread_value": round(2 * T_sample / dt1 / 1e9, 4),
            "sample": f"AllGather + AllReduce, R=8 bf16, T={T_sample >> 20} MiB each (the first "
                      f"{T_sample >> 20} MiB of the benchmark's own inputs; the workload is T=1 GiB), "
                      f"the C oracle on {cores} element-range slices in {cores} threads, {dt:.2f} s "
                      f"({dt1:.2f} s in one thread)"}


def run_ours(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    import __graft_entry__
    __graft_entry__.build()
    from copy_reduce_datapath_gb300 import purlin as P

    ctx = P.pl_ctx_create(local, 0)
    wl = Workload(args.T, device)
    stream = torch.cuda.Stream(device)
    s = stream.cuda_stream
    for _ in range(args.warmup):
        wl.allgather(ctx, s)
        wl.allreduce(ctx, s)
    torch.cuda.synchronize()
    assert P.pl_ctx_status(ctx, s) == P.PL_OK
    parity_ok = sampled_parity(wl, device)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    launches0 = P.pl_ctx_launches(ctx)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)  # let the sampler see the start of the timed region
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(args.steps):
        ev[k][0].record(stream)
        wl.allgather(ctx, s)
        ev[k][1].record(stream)
        wl.allreduce(ctx, s)
        ev[k][2].record(stream)
    end.record(stream)
    end.synchronize()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if ws > 1:
        torch.distributed.barrier()
    launches = P.pl_ctx_launches(ctx) - launches0
    ms_total = start.elapsed_time(end)
    ag_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    ar_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    assert P.pl_ctx_status(ctx, s) == P.PL_OK

    # CTAs and SMs each collective's launch used (the plan the library derived for this GPU)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    grid = {}
    lens_ar = [wl.n_ar // R] * (R - 1) + [wl.n_ar - (wl.n_ar // R) * (R - 1)]
    l_ar = P.pl_layout_partitioned(R, lens_ar)
    for name, lin, lout, op in (("allgather", wl.ag_lin, wl.ag_lout, "copy"), ("allreduce", l_ar, l_ar, "sum")):
        plan = P.pl_plan_create(lin, lout, op, "bf16", R, None, num_sms=sms)
        st = P.pl_plan_get_stats(plan)
        grid[name] = {"ctas": int(st.ctas), "sms_used": int(min(st.ctas, sms)), "sms": sms, "items": int(st.items)}
        P.pl_plan_destroy(plan)

    t_max = max_over_ranks(ms_total, ws, device)
    ms_step, value = replica_throughput(t_max, args.steps, args.T, ws)

    peak, peak_kind = measured_peaks()
    ar_bytes = 2 * R * wl.n_ar * 2        # read R*T, write R*T
    ag_bytes = (R * wl.n_ag + R * R * wl.n_ag) * 2  # read T, write R*T
    achieved = ar_bytes / (ar_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"AllGather + AllReduce over R=8 logical ranks in one GPU, bf16 N(0,1) seed 1, "
                               f"equal partitions, T={args.T >> 20} MiB per collective",
                   "R": R, "T_bytes": args.T, "parallelism": f"replicas x{ws} (no data-path collective)",
                   "l2": "inputs larger than L2 (every input buffer >= 128 MiB), no flush needed",
                   "policy": "automatic: zero-staging, fused AllReduce; AllGather on the bulk ring, "
                             "AllReduce on the 16-byte vector datapath"},
        "per_collective": {"allgather": {"ms": round(ag_ms, 4), "algbw_GBps": round(args.T / (ag_ms * 1e-3) / 1e9, 2),
                                         "hbm_GBps": round(ag_bytes / (ag_ms * 1e-3) / 1e9, 1), **grid["allgather"]},
                           "allreduce": {"ms": round(ar_ms, 4), "algbw_GBps": round(args.T / (ar_ms * 1e-3) / 1e9, 2),
                                         "hbm_GBps": round(achieved, 1), **grid["allreduce"]}},
        "roofline": {"bound": "hbm", "kernel": "snac_kernel (AllReduce, fused zero-staging)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} (copy bandwidth)",
                     "algorithmic_bytes_per_launch": ar_bytes,
                     "traffic": committed_traffic("allreduce_1GiB"),
                     "traffic_note": committed_traffic_note("allreduce_1GiB")},
        "gpu_launches": int(launches),
        "clocks": clocks,
        "parity_sampled": parity_ok,
    }
    if rank == 0 and not args.no_sweep:
        line["sweep"] = time_sweep(ctx, wl, stream, torch, peak)
        line["configs"] = time_configs(ctx, wl, stream, torch, peak)
    if rank == 0 and not args.no_e2e:
        e2e = run_e2e(ctx, wl, stream, torch, args.e2e_steps)
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu and ws == 1:
        line["cpu_baseline"] = cpu_baseline_line(wl, ORACLE_SAMPLE_T)
    P.pl_ctx_destroy(ctx)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------ single cases

CASES = {
    # name: (collective, dtype, reduction, description)
    "allgather": ("allgather", "bf16", "sum", "AllGather, R=8, bf16 N(0,1), equal partitions, T = output bytes per rank"),
    "allreduce": ("allreduce", "bf16", "sum", "AllReduce, R=8, bf16 N(0,1), T = bytes per rank"),
    "allreduce_r3_fp32": ("allreduce", "fp32", "sum", "AllReduce, R=3, fp32 integers in [-8, 8], T = bytes per rank"),
    "reducescatter_bf16": ("reducescatter", "bf16", "sum", "ReduceScatter, R=8, bf16 U(-1,1), T = input bytes per rank"),
    "reducescatter_fp32": ("reducescatter", "fp32", "sum", "ReduceScatter, R=8, fp32 U(-1,1), T = input bytes per rank"),
    "reducescatter_inplace_bf16": ("reducescatter_inplace", "bf16", "sum", "ReduceScatter in place, R=8, bf16 U(-1,1)"),
    "alltoall_moe": ("alltoall", "bf16", "sum", "AllToAll, R=8, per rank [4096 tokens, 7168] bf16, 8 token groups (T ignored)"),
    "ulysses": ("ulysses", "bf16", "sum", "Ulysses AllToAll, R=8, per rank [16384, 32, 128] bf16, seq->head (T ignored)"),
    "allgatherv": ("allgatherv", "bf16", "sum", "AllGatherV, R=8, bf16, Zipf s=0.125 lengths, T = output bytes per rank"),
    "reducescatterv": ("reducescatterv", "bf16", "sum", "ReduceScatterV, R=8, bf16, Zipf s=0.125, T = input bytes per rank"),
    "alltoallv": ("alltoallv", "bf16", "sum", "AllToAllV, R=8, bf16, Zipf s=0.125 rows, T = input bytes per rank"),
    # further element types and the maximum reduction
    "allreduce_fp16": ("allreduce", "fp16", "sum", "AllReduce, R=8, fp16 U(-1,1), T = bytes per rank"),
    "reducescatter_fp16": ("reducescatter", "fp16", "sum", "ReduceScatter, R=8, fp16 U(-1,1), T = input bytes per rank"),
    "allreduce_max_bf16": ("allreduce", "bf16", "max", "AllReduce (maximum), R=8, bf16 N(0,1), T = bytes per rank"),
    "allreduce_max_fp32": ("allreduce", "fp32", "max", "AllReduce (maximum), R=8, fp32 U(-1,1), T = bytes per rank"),
    "allgather_fp8": ("allgather", "fp8", "sum", "AllGather, R=8, one-byte elements, T = output bytes per rank"),
    "alltoall_moe_fp8": ("alltoall", "fp8", "sum", "AllToAll, R=8, per rank [4096 tokens, 7168] fp8, 8 token groups (T ignored)"),
    "allgatherv_fp8": ("allgatherv", "fp8", "sum", "AllGatherV, R=8, one-byte elements, Zipf s=0.125, T = output bytes per rank"),
}
TORCH_DT = {"bf16": "bfloat16", "fp32": "float32", "fp16": "float16", "fp8": "uint8"}
ELEM_BYTES = {"bf16": 2, "fp32": 4, "fp16": 2, "fp8": 1}


def run_case(args):
    """Times `warmup` + `steps` launches of one workload; prints latency, algbw and HBM bandwidth."""
    import torch
    import synth
    import __graft_entry__
    __graft_entry__.build()
    from copy_reduce_datapath_gb300 import purlin as P
    kind, dt, red, desc = CASES[args.case]
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    tdt = getattr(torch, TORCH_DT[dt])
    S = ELEM_BYTES[dt]
    pol = P.pl_policy_default()
    for kv in filter(None, args.policy.split(",")):
        k, v = kv.split("=")
        setattr(pol, k, int(v))
    Rr = 3 if args.case == "allreduce_r3_fp32" else R
    ctx = P.pl_ctx_create(0, args.scratch if pol.path == P.PL_PATH_STAGED else 0)
    T = args.T
    N = T // S

    def normal(seed, r, n):
        if dt == "bf16":
            return synth.device_normal_bf16(seed, r, n, dev)
        if dt == "fp8":
            return synth.device_bytes(seed, r, n, dev)
        return synth.device_uniform_pm1(seed, r, n, dev, tdt)

    if kind == "allgather":
        n = N // Rr
        ins = [normal(1, r, n) for r in range(Rr)]
        outs = [torch.empty(n * Rr, dtype=tdt, device=dev) for _ in range(Rr)]
        lin, lout, op = P.pl_layout_rank_owned(Rr, [n] * Rr), P.pl_layout_partitioned(Rr, [n] * Rr), "copy"
        moved = (n * Rr + Rr * n * Rr) * S
    elif kind == "allreduce":
        if args.case == "allreduce_r3_fp32":
            ins = [torch.from_numpy(synth.int_uniform_f32(0, r, N)).to(dev) for r in range(Rr)]
        else:
            ins = [normal(1, 100 + r, N) for r in range(Rr)]
        outs = [torch.empty(N, dtype=tdt, device=dev) for _ in range(Rr)]
        lin = lout = P.pl_layout_partitioned(Rr, synth.equal_lengths(N, Rr))
        op, moved = red, 2 * Rr * N * S
    elif kind in ("reducescatter", "reducescatter_inplace", "reducescatterv"):
        lens = synth.zipf_lengths(N, Rr, 0.125, seed=4) if kind == "reducescatterv" else [N // Rr] * Rr
        ins = [normal(2, r, N) for r in range(Rr)] if dt == "fp8" else \
            [synth.device_uniform_pm1(2, r, N, dev, tdt) for r in range(Rr)]
        lin = P.pl_layout_partitioned(Rr, lens)
        if kind == "reducescatter_inplace":
            outs, lout = ins, P.pl_layout_rank_owned_inplace(Rr, lens)
        else:
            outs = [torch.empty(lens[k], dtype=tdt, device=dev) for k in range(Rr)]
            lout = P.pl_layout_rank_owned(Rr, lens)
        op, moved = red, (Rr * N + N) * S
    elif kind == "allgatherv":
        lens = synth.zipf_lengths(N, Rr, 0.125, seed=4)
        ins = [normal(4, r, lens[r]) for r in range(Rr)]
        outs = [torch.empty(N, dtype=tdt, device=dev) for _ in range(Rr)]
        lin, lout, op = P.pl_layout_rank_owned(Rr, lens), P.pl_layout_partitioned(Rr, lens), "copy"
        moved = (N + Rr * N) * S
    elif kind in ("alltoall", "alltoallv", "ulysses"):
        if kind == "alltoall":
            n = 4096 * 7168
            m = [[n // Rr] * Rr for _ in range(Rr)]
            lin, lout = P.pl_layout_alltoall_in(Rr, m), P.pl_layout_alltoall_out(Rr, m)
        elif kind == "ulysses":
            n = 16384 * 32 * 128
            lin, lout = P.pl_layout_ulysses_in(Rr, 16384, 32, 128), P.pl_layout_ulysses_out(Rr, 16384, 32, 128)
            m = [[n // Rr] * Rr for _ in range(Rr)]
        else:
            m = synth.zipf_matrix(N, Rr, 0.125, seed=4)
            n = N
            lin, lout = P.pl_layout_alltoall_in(Rr, m), P.pl_layout_alltoall_out(Rr, m)
        ins = [normal(3, r, sum(m[r])) for r in range(Rr)]
        outs = [torch.empty(sum(m[r][j] for r in range(Rr)), dtype=tdt, device=dev) for j in range(Rr)]
        op, moved = "copy", 2 * Rr * n * S
        T = n * S
    stream = torch.cuda.current_stream()

    def call():
        P.pl_collective(ctx, lin, lout, op, dt, Rr, P.ptrs(ins), P.counts(ins), P.ptrs(outs), P.counts(outs), pol,
                        stream.cuda_stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        call()
    b.record(stream)
    torch.cuda.synchronize()
    assert P.pl_ctx_status(ctx, stream.cuda_stream) == P.PL_OK
    us = a.elapsed_time(b) * 1e3 / max(1, args.steps)
    peak, kind_peak = measured_peaks()
    # The plan's own bytes (staging included), from the derived work list.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    scratch = args.scratch if pol.path == P.PL_PATH_STAGED else 0
    plan = P.pl_plan_create(lin, lout, op, dt, Rr, pol, sms, scratch)
    st = P.pl_plan_get_stats(plan)
    own = int(st.bytes_read + st.bytes_written)
    P.pl_plan_destroy(plan)
    print(json.dumps({"case": args.case, "workload": desc, "T_bytes": T, "policy": args.policy or "default",
                      "scratch_bytes": scratch,
                      "steps": args.steps, "us": round(us, 2), "algbw_GBps": round(T / us / 1e3, 2),
                      "hbm_GBps": round(moved / us / 1e3, 1), "frac_of_peak": round(moved / us / 1e3 / peak, 4),
                      "plan_bytes": own, "plan_frac_of_peak": round(own / us / 1e3 / peak, 4),
                      "peak_GBps": peak, "peak_kind": kind_peak}), flush=True)
    P.pl_ctx_destroy(ctx)


def run_depth_sweep(args):
    """One 256 MiB copy (one source region to one destination region) through the
    Atom datapath: the vector path and the cp.async.bulk ring at depths 1..8,
    each at several CTA counts.  Reports read + write bandwidth."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from copy_reduce_datapath_gb300 import purlin as P
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    n = (256 << 20) // 2
    src = torch.randn(n, device=dev).to(torch.bfloat16)
    dst = torch.empty_like(src)
    ctx = P.pl_ctx_create(0, 0)
    L = P.pl_layout_rank_owned(1, [n])
    stream = torch.cuda.current_stream()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak, peak_kind = measured_peaks()
    rows = []
    for ctas in (8, 16, 32, 64, sms):
        for datapath, stages in [(P.PL_ATOM_VECTOR, 0)] + [(P.PL_ATOM_BULK, d) for d in range(1, 9)]:
            pol = P.pl_policy_default(datapath=datapath, stages=stages, ctas=ctas)

            def call():
                P.pl_collective(ctx, L, L, "copy", "bf16", 1, [src.data_ptr()], [n], [dst.data_ptr()], [n], pol,
                                stream.cuda_stream)
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(10):
                call()
            b.record(stream)
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / 10
            rows.append({"ctas": ctas, "datapath": "vector" if datapath == P.PL_ATOM_VECTOR else "bulk",
                         "stages": stages, "us": round(us, 1), "GBps": round(2 * n * 2 / us / 1e3, 1)})
    assert P.pl_ctx_status(ctx, stream.cuda_stream) == P.PL_OK
    torch.testing.assert_close(dst, src, rtol=0, atol=0)
    print(json.dumps({"sweep": "atom_copy_256MiB", "bytes_moved": 2 * n * 2, "peak_GBps": peak,
                      "peak_kind": peak_kind, "rows": rows}), flush=True)
    P.pl_ctx_destroy(ctx)


def run_policy_sweep(args):
    """The automatic chunk policy against fixed chunk sizes: AllGather and
    AllReduce of the benchmark workload (R=8, bf16) at T = 1 MiB .. 1 GiB, each
    with chunk_bytes = auto and 64 KiB .. 4 MiB (datapath automatic).  Prints,
    per (collective, T), the time of every chunk size, the chunk the automatic
    policy picked and its time relative to the best fixed size."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from copy_reduce_datapath_gb300 import purlin as P
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    wl = Workload(GiB, dev)
    ctx = P.pl_ctx_create(0, 0)
    stream = torch.cuda.Stream()  # graph capture needs a stream other than the default one
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    chunks = [0, 64 << 10, 256 << 10, 1 << 20, 4 << 20]
    rows = []
    for e in (20, 23, 26, 28, 30):
        T = 1 << e
        for name in ("allgather", "allreduce"):
            if name == "allgather":
                n = T // 2 // R
                lin, lout = wl._layouts(n)
                ins, outs, op = wl.ag_in, wl.ag_out, "copy"
                icount, ocount = [n] * R, [n * R] * R
            else:
                n = T // 2
                lens = [n // R] * (R - 1) + [n - (n // R) * (R - 1)]
                lin = lout = P.pl_layout_partitioned(R, lens)
                ins, outs, op = wl.ar_in, wl.ar_out, "sum"
                icount = ocount = [n] * R
            row = {"collective": name, "T": T, "us": {}}
            for cb in chunks:
                pol = P.pl_policy_default(chunk_bytes=cb)

                def call():
                    P.pl_collective(ctx, lin, lout, op, "bf16", R, P.ptrs(ins), icount, P.ptrs(outs), ocount, pol,
                                    stream.cuda_stream)
                us, _ = time_call(call, T, stream, torch)
                row["us"]["auto" if cb == 0 else str(cb)] = round(us, 2)
            plan = P.pl_plan_create(lin, lout, op, "bf16", R, None, num_sms=sms)
            row["auto_chunk_bytes"] = int(P.pl_plan_get_stats(plan).chunk_elems) * 2
            P.pl_plan_destroy(plan)
            fixed = {k: v for k, v in row["us"].items() if k != "auto"}
            best = min(fixed, key=fixed.get)
            row["best_fixed"] = int(best)
            row["auto_over_best"] = round(row["us"]["auto"] / fixed[best], 3)
            rows.append(row)
    assert P.pl_ctx_status(ctx, stream.cuda_stream) == P.PL_OK
    print(json.dumps({"sweep": "chunk_policy", "R": R, "dtype": "bf16", "rows": rows}), flush=True)
    P.pl_ctx_destroy(ctx)


def run_copy_engine(args):
    """AllGather (R=8, bf16, T bytes of output per rank) done by one contiguous
    device-to-device copy per (source, destination) pair -- the copy-engine
    route that launches no kernel -- timed beside the library's AllGather."""
    import torch
    import synth
    import __graft_entry__
    __graft_entry__.build()
    from copy_reduce_datapath_gb300 import purlin as P
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    T = args.T
    n = T // 2 // R
    ins = [synth.device_normal_bf16(SEED, r, n, dev) for r in range(R)]
    outs = [torch.empty(n * R, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    stream = torch.cuda.current_stream()

    def by_memcpy():
        for r in range(R):
            for j in range(R):
                outs[r][j * n:(j + 1) * n].copy_(ins[j], non_blocking=True)

    ctx = P.pl_ctx_create(0, 0)
    lin, lout = P.pl_layout_rank_owned(R, [n] * R), P.pl_layout_partitioned(R, [n] * R)

    def by_kernel():
        P.pl_collective(ctx, lin, lout, "copy", "bf16", R, P.ptrs(ins), P.counts(ins), P.ptrs(outs), P.counts(outs),
                        None, stream.cuda_stream)

    res = {}
    for name, fn in (("memcpy_per_pair", by_memcpy), ("snac_kernel", by_kernel)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(max(1, args.steps)):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / max(1, args.steps)
        res[name] = {"us": round(us, 2), "algbw_GBps": round(T / us / 1e3, 2),
                     "hbm_GBps": round((n * R + R * n * R) * 2 / us / 1e3, 1)}
        for r in range(R):
            for j in (0, R - 1):
                assert torch.equal(outs[r][j * n:(j + 1) * n], ins[j])
    print(json.dumps({"compare": "allgather_copy_engine_vs_kernel", "R": R, "T_bytes": T, "results": res}),
          flush=True)
    P.pl_ctx_destroy(ctx)


def run_reference(args):
    """The oracle on the host cores: the reference arm of this build (the pages
    ship no code).  Each step is a bounded sample of the workload (64 MiB per
    collective); the requested warm-up and timed steps all run unless the
    timed ones pass REFERENCE_BUDGET_S, so the run ends within a few minutes."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from oracle import build as ob
    ob.build()
    T_s = REFERENCE_SAMPLE_T
    ag, ar = oracle_inputs_host(T_s)
    cores = host_cores()
    for _ in range(args.warmup):
        oracle_time(ag, ar, cores)
    times, t0 = [], time.perf_counter()
    for _ in range(max(1, args.steps)):
        times.append(oracle_time(ag, ar, cores))
        if time.perf_counter() - t0 > REFERENCE_BUDGET_S:
            break
    steps = len(times)
    dt = statistics.median(times)
    value = 2 * T_s / dt / 1e9
    dt1 = oracle_time(ag, ar)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": ws,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "AllGather + AllReduce over R=8 logical ranks, bf16 N(0,1) seed 1, equal "
                               f"partitions; each step a bounded sample of T={T_s >> 20} MiB per collective "
                               "(the workload is T=1 GiB)", "R": R, "T_bytes": T_s, "workload_T_bytes": GiB},
        "steps_requested": args.steps,
        "steps_note": (f"all {steps} requested steps timed" if steps >= args.steps else
                       f"the CPU oracle stopped after {steps} of {args.steps} requested steps "
                       f"(a {REFERENCE_BUDGET_S:.0f} s bound, so that the run ends within a few minutes)"),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "single_thread_value": round(2 * T_s / dt1 / 1e9, 4),
                         "sample": f"T={T_s >> 20} MiB per collective, the C oracle on {cores} element-range "
                                   f"slices in {cores} threads, median of {steps} steps"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.depth_sweep:
        run_depth_sweep(args)
    elif args.copy_engine:
        run_copy_engine(args)
    elif args.policy_sweep:
        run_policy_sweep(args)
    elif args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
