#!/usr/bin/env python3
"""Benchmark: one step = layout -> dispatch (bf16) -> combine over one batch of
the DeepSeek-V3-shaped workload (4096 tokens, hidden 7168 bf16, 256 experts
over 8 logical ranks, top-8), synthetic inputs resident in HBM.

Prints ONE JSON line (rank 0). Default: 1 GPU, K timed steps (each after an
untimed L2 flush), then ~2 s of the same flushed step back to back under the
clock sampler, every variant and the skewed workload timed alone, the
end-to-end leg from pinned host buffers, and the CPU oracle timed on the host
cores (single-threaded and on every core) as a reported baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --profile-kernel combine     # one launch for an ncu capture

Under torchrun each rank runs an independent replica on its own GPU (the
path shards by tokens and has no exchange step): weak scaling, max-over-ranks
time, whole-job tokens/s. ``--impl reference`` times the CPU oracle (the only
reference implementation available for this path) on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from combine_moe_get_gb300 import workloads as wl  # noqa: E402

WORKLOAD = "dsv3"
HBM_SPEC_GBS = 7900.0   # nominal HBM3e bandwidth of a GB300, for context next to the measured peak
METRIC = "dispatch+combine tokens/s and achieved HBM GB/s (% of peak), DSv3 shape"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ measured peaks, clocks, profiles

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        target = str(device_index)
        try:
            bus = torch.cuda.get_device_properties(device_index).pci_bus_id
            if bus:
                target = bus
        except Exception:
            pass
        self.cmd = ["nvidia-smi", "-i", target, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "200"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        smax = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def profiled_traffic(kernel: str, source: str, workload: str = WORKLOAD):
    """DRAM traffic of one launch recorded in profiles/<kernel>_<workload>.md,
    if the kernel source has not changed since (its sha256 is recorded beside
    it): {"in_window": bytes ncu counted inside the kernel, "writeback": bytes
    of the kernel's output still dirty in L2 when it ended, counted as the
    writes of the L2-evicting read that follows it}, or None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    src = os.path.join(ROOT, "combine_moe_get_gb300", "csrc", source)
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except Exception:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256") != sha:
        return None
    try:
        return {"in_window": float(vals["dram_bytes_per_launch"]),
                "writeback": float(vals["writeback_bytes_after_launch"])}
    except Exception:
        return None


# ------------------------------------------------------------------ CPU oracle timing

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def time_oracle(inp, w, budget_s: float, min_steps: int = 1, threads: int = 1):
    """Whole oracle steps (layout, then bf16 dispatch, then combine) over the
    whole batch until `budget_s` elapses. With `threads` > 1 the dispatch and
    the combine run over token ranges on that many threads (the same per-token
    code and results); the layout, a serial scan, stays on one thread."""
    import oracle
    topk = inp.topk_idx.numpy()
    xb = inp.x.view(torch.int16).numpy().view(np.uint16)
    wts = inp.topk_weights.numpy()
    pb = inp.partial.view(torch.int16).numpy().view(np.uint16)
    cap = wl.recv_capacity(w.num_tokens, w.num_topk, w.num_ranks)
    steps, t0 = 0, time.perf_counter()
    while steps < min_steps or time.perf_counter() - t0 < budget_s:
        lay = oracle.layout(topk, w.num_experts, w.num_ranks)
        oracle.dispatch(xb, topk, wts, w.num_experts, w.num_ranks, lay["token_dst_row"], cap, threads=threads)
        oracle.combine(pb[: lay["num_recv"]], lay["token_dst_row"], threads=threads)
        steps += 1
    dt = time.perf_counter() - t0
    return steps, dt


def workload_config(w, recv_rows: int) -> dict:
    """The `config` of both arms' lines (identical, so the two are comparable)."""
    return {"workload": "DeepSeek-V3 prefill shape: T=4096, H=7168 bf16, E=256 over R=8 logical ranks, "
                        "top-8 uniform, softmax weights",
            "tokens": w.num_tokens, "hidden": w.hidden, "experts": w.num_experts, "ranks": w.num_ranks,
            "topk": w.num_topk, "recv_rows": recv_rows,
            "l2": "GPU arm: L2 flushed before every timed step (a buffer of twice the L2 size written, then another "
                  "read; untimed); CPU arm: the step's ~1.1 GB working set exceeds every host cache",
            "parallelism": "independent token shards, one per GPU; no collective"}


# ------------------------------------------------------------------ the GPU step

class Step:
    def __init__(self, moe, w, inp, device):
        self.moe, self.w = moe, w
        T, k, E, R, H = w.num_tokens, w.num_topk, w.num_experts, w.num_ranks, w.hidden
        self.cap = wl.recv_capacity(T, k, R)
        self.x = inp.x.to(device)
        self.topk = inp.topk_idx.to(device)
        self.wts = inp.topk_weights.to(device)
        self.partial = inp.partial.to(device)
        self.status = moe.new_status(device)
        self.bal = moe.new_balance_counter(device)     # the combine's
        self.bal_d = moe.new_balance_counter(device)   # the dispatch's
        self.lay = moe.Layout.empty(T, k, E, R, device)
        self.ws = torch.empty(moe.moe_get_layout_workspace_size(T, E, R), dtype=torch.uint8, device=device)
        self.disp = moe.Dispatched(
            recv_x=torch.empty(self.cap, H, dtype=torch.bfloat16, device=device), recv_x_scales=None,
            recv_topk_idx=torch.empty(self.cap, k, dtype=torch.int64, device=device),
            recv_topk_weights=torch.empty(self.cap, k, dtype=torch.float32, device=device),
            recv_src_idx=torch.empty(self.cap, dtype=torch.int32, device=device), x_scales=None)
        self.disp8 = moe.Dispatched(
            recv_x=torch.empty(self.cap, H, dtype=torch.uint8, device=device),
            recv_x_scales=torch.empty(self.cap, H // 128, dtype=torch.float32, device=device),
            recv_topk_idx=self.disp.recv_topk_idx, recv_topk_weights=self.disp.recv_topk_weights,
            recv_src_idx=self.disp.recv_src_idx, x_scales=torch.empty(T, H // 128, dtype=torch.float32, device=device))
        self.out = torch.empty(T, H, dtype=torch.bfloat16, device=device)
        # E4M3 rows + scales for the pass-through dispatch (codes of x; any bytes would do for a copy)
        self.x8 = (self.x.view(torch.int16) & 0xFF).to(torch.uint8).contiguous()
        self.x8_scales = torch.ones(T, H // 128, dtype=torch.float32, device=device)
        self.disp8in = moe.Dispatched(
            recv_x=self.disp8.recv_x, recv_x_scales=self.disp8.recv_x_scales,
            recv_topk_idx=self.disp.recv_topk_idx, recv_topk_weights=self.disp.recv_topk_weights,
            recv_src_idx=self.disp.recv_src_idx, x_scales=None)
        self.row_w = torch.rand(self.cap, generator=torch.Generator().manual_seed(w.seed + 2)).to(device)
        self.cw = torch.empty(T, k, dtype=torch.float32, device=device)
        # expand mode: one receive row per valid top-k entry, grouped by expert
        self.xcap = T * k
        self.xws = torch.empty(moe.moe_get_expand_layout_workspace_size(T, E), dtype=torch.uint8, device=device)
        self.xrows = torch.empty(T, k, dtype=torch.int32, device=device)
        self.dispx = moe.Dispatched(
            recv_x=torch.empty(self.xcap, H, dtype=torch.bfloat16, device=device), recv_x_scales=None,
            recv_topk_idx=torch.empty(self.xcap, k, dtype=torch.int64, device=device),
            recv_topk_weights=torch.empty(self.xcap, k, dtype=torch.float32, device=device),
            recv_src_idx=torch.empty(self.xcap, dtype=torch.int32, device=device), x_scales=None)
        self.partial_x = (self.partial if self.partial.shape[0] >= self.xcap else
                          wl.make_partial(torch.Generator().manual_seed(w.seed + 1), self.xcap, H).to(device))

    def layout(self):
        self.moe.moe_get_layout(self.topk, self.w.num_experts, self.w.num_ranks, out=self.lay, workspace=self.ws,
                                status=self.status)

    def dispatch(self, fp8=False):
        self.moe.moe_dispatch(self.x, self.topk, self.wts, self.w.num_experts, self.w.num_ranks,
                              self.lay.token_dst_row, self.cap, quantize_fp8=fp8,
                              out=self.disp8 if fp8 else self.disp, balance=self.bal_d, status=self.status)

    def dispatch_fp8_input(self):
        self.moe.moe_dispatch(self.x8, self.topk, self.wts, self.w.num_experts, self.w.num_ranks,
                              self.lay.token_dst_row, self.cap, x_scales=self.x8_scales, out=self.disp8in,
                              balance=self.bal_d, status=self.status)

    def combine_weighted(self):
        self.moe.moe_combine_ex(self.partial, self.lay.token_dst_row, row_weights=self.row_w,
                                recv_topk_weights=self.disp.recv_topk_weights, out=self.out,
                                combined_topk_weights=self.cw, balance=self.bal, status=self.status)

    def combine(self):
        # with a balance counter: the last 30% of the tokens go to whichever CTA is free first
        self.moe.moe_combine_ex(self.partial, self.lay.token_dst_row, out=self.out, balance=self.bal,
                                status=self.status)

    def combine_unbalanced(self):
        self.moe.moe_combine(self.partial, self.lay.token_dst_row, out=self.out, status=self.status)

    def combine_fp8(self):
        # E4M3 partial rows: the FP8 dispatch's own receive rows and scales (balance counter: used on long runs)
        self.moe.moe_combine_fp8(self.disp8.recv_x, self.disp8.recv_x_scales, self.lay.token_dst_row, out=self.out,
                                 balance=self.bal, status=self.status)

    def layout_dispatch(self):
        self.moe.moe_layout_dispatch(self.x, self.topk, self.wts, self.w.num_experts, self.w.num_ranks, self.cap,
                                     layout=self.lay, workspace=self.ws, out=self.disp, status=self.status)

    def expand_layout(self):
        self.moe.moe_get_expand_layout(self.topk, self.lay.expert_prefix, self.w.num_experts, out=self.xrows,
                                       workspace=self.xws, status=self.status)

    def dispatch_expand(self):
        self.moe.moe_dispatch(self.x, self.topk, self.wts, self.w.num_experts, self.w.num_ranks, self.xrows,
                              self.xcap, expand=True, out=self.dispx, balance=self.bal_d, status=self.status)

    def combine_expand(self):
        self.moe.moe_combine_ex(self.partial_x, self.xrows, out=self.out, balance=self.bal, status=self.status)

    def expand_step(self):
        self.layout()
        self.expand_layout()
        self.dispatch_expand()
        self.combine_expand()




class Flush:
    """The L2 flush between timed steps: write a buffer twice the size of L2,
    then read another one. The write evicts everything, and the read evicts the
    write's dirty lines (written back here, untimed), so the timed kernels start
    on a cold L2 that holds only clean lines and pay for no write-back but their
    own."""

    def __init__(self, device):
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.buf = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=device)
        self.src = torch.ones_like(self.buf)
        self.sum = torch.empty((), dtype=torch.int64, device=device)

    def __call__(self):
        self.buf.zero_()
        torch.sum(self.src.view(torch.int64), dim=0, out=self.sum)

    def evict(self):
        """A read of a clean buffer larger than L2: whatever the kernel before it
        left dirty in L2 is written back during this read."""
        torch.sum(self.buf.view(torch.int64), dim=0, out=self.sum)

    def describe(self) -> str:
        return (f"flushed between steps ({self.buf.numel() >> 20} MiB written, then {self.src.numel() >> 20} MiB "
                f"read; untimed)")


class Timer:
    """Times a callable alone: captured once in a CUDA graph with an event at
    each end and replayed after an L2 flush each time (eager calls bracketed by
    events when graphs are unavailable). Returns the per-call milliseconds."""

    def __init__(self, flush: Flush, stream, use_graph: bool):
        self.flush, self.stream, self.use_graph = flush, stream, use_graph

    def __call__(self, fn, reps: int):
        fn()                                    # first call outside any capture
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True, external=self.use_graph)
        b = torch.cuda.Event(enable_timing=True, external=self.use_graph)
        g = None
        if self.use_graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                a.record()
                fn()
                b.record()
        ms = []
        for i in range(reps + 2):
            self.flush()
            if g is not None:
                g.replay()
            else:
                a.record(self.stream)
                fn()
                b.record(self.stream)
            torch.cuda.synchronize()
            if i >= 2:
                ms.append(a.elapsed_time(b))
        return ms


def algorithmic_bytes(T: int, H: int, N: int, NX: int) -> dict:
    """Bytes each call must move at least (T tokens, hidden H, N receive rows,
    NX expand rows)."""
    row = H * 2
    nb = H // 128
    bf16 = T * row + N * row                            # x read once + one row per (token, rank)
    return {
        "dispatch": bf16, "combine": bf16,              # combine: the rows read, one bf16 row per token written
        "dispatch_fp8": T * row + N * H + N * nb * 4,   # x read + e4m3 rows + scales
        "dispatch_fp8_input": (T + N) * (H + nb * 4),   # e4m3 rows + scales read once, written per rank
        "combine_weighted": bf16 + N * 4,               # + one weight per receive row
        "dispatch_expand": T * row + NX * row,          # x read once + one row per valid entry
        "combine_fp8": N * (H + nb * 4) + T * row,      # e4m3 rows + scales read, bf16 out written
    }


def gbs(nbytes: float, ms: float) -> float:
    return nbytes / (ms * 1e-3) / 1e9


def run_ours(args, world, rank, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    from combine_moe_get_gb300 import binding as moe

    w = wl.CONFIGS[WORKLOAD]
    inp = wl.make_inputs(dataclass_replace_seed(w, w.seed + rank))
    st = Step(moe, w, inp, device)
    T, H = w.num_tokens, w.hidden
    flush_l2 = Flush(device)
    stream = torch.cuda.current_stream(device)

    def one(events=None):
        """The step through the public API: moe_layout_dispatch (the layout, then
        the dispatch, which starts loading input rows while the layout runs and
        balances its tail through the layout workspace), then moe_combine_ex with
        a balance counter. With events, the per-kernel breakdown: moe_get_layout,
        moe_dispatch and the same combine, with an event between each two."""
        if not events:
            st.layout_dispatch()
            st.combine()
            return
        events[0].record()
        st.layout()
        events[1].record()
        st.dispatch()
        events[2].record()
        st.combine()
        events[3].record()

    for _ in range(args.warmup):
        flush_l2()
        one()
    st.layout()   # the separate calls once before any capture
    st.dispatch()
    st.combine()
    torch.cuda.synchronize()
    moe.check_status(st.status, "warm-up")
    N = int(st.lay.rank_prefix[-1].item())

    # The step is captured once in a CUDA graph (after warm-up: no allocation or
    # attribute setting happens during capture) and replayed, so host-side
    # submission cost never leaves the GPU idle inside the timed events.
    timing = "cuda-graph replay"
    mean, med = statistics.fmean, statistics.median
    try:
        # the step alone: events only at its ends (an event between two kernels
        # adds its own gap to the step)
        ev_step = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            ev_step[0].record()
            one()
            ev_step[1].record()
        # the per-kernel breakdown: events between the kernels
        evs_k = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
        graph_k = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_k):
            one(evs_k)
        graph.replay()
        graph_k.replay()
        torch.cuda.synchronize()
    except Exception as exc:  # eager fallback (e.g. no external events in this torch)
        graph, graph_k, timing = None, None, f"eager ({type(exc).__name__})"

    def timed_step():
        """One step (after an untimed L2 flush): (step ms, [layout, dispatch, combine] ms or None)."""
        flush_l2()
        if graph is not None:
            graph.replay()
            torch.cuda.synchronize()
            return ev_step[0].elapsed_time(ev_step[1]), None
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        one(ev)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[3]), [ev[j].elapsed_time(ev[j + 1]) for j in (0, 1, 2)]

    def sustain(seconds: float):
        """The same step, L2 flushed before each, replayed back to back for about
        `seconds`, so that the clock sampler sees the GPU under this load: M
        flushed steps per graph replay, each bracketed by its own events."""
        if graph is None:
            return []
        M = 64
        evs = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True)) for _ in range(M)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for a, b in evs:
                flush_l2()
                a.record()
                one()
                b.record()
        ms, t0 = [], time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            g.replay()
            torch.cuda.synchronize()
            ms += [a.elapsed_time(b) for a, b in evs]
        del g
        return ms

    step_ms, parts = [], []
    with ClockSampler(device.index) as clk:
        barrier(world)
        torch.cuda.synchronize()
        for i in range(args.steps):
            ms, p = timed_step()
            step_ms.append(ms)
            if p:
                parts.append(p)
        torch.cuda.synchronize()
        barrier(world)
        # after the K timed steps, still under the clock sampler
        sus_ms = sustain(args.sustain_s)
    moe.check_status(st.status, "timed steps")
    clocks = clk.summary()
    clocks["window"] = f"the {args.steps} timed steps and the {len(sus_ms)} sustained steps after them"

    # per-kernel breakdown (outside the timed region): the graph with events between kernels
    if graph_k is not None:
        for i in range(args.steps):
            flush_l2()
            graph_k.replay()
            torch.cuda.synchronize()
            parts.append([evs_k[j].elapsed_time(evs_k[j + 1]) for j in (0, 1, 2)])
        moe.check_status(st.status, "kernel breakdown")
    lay_ms = [p[0] for p in parts]
    dis_ms = [p[1] for p in parts]
    com_ms = [p[2] for p in parts]
    ms_per_step = max_over_ranks(mean(step_ms), world, device)
    tokens_per_s = world * T / (ms_per_step / 1e3)
    ref_out = st.out.clone()     # the device-resident step's output, for the end-to-end leg's check

    # the other dispatch / combine variants, each timed alone with the same flush discipline
    timer = Timer(flush_l2, stream, graph is not None)
    reps = max(3, args.steps // 2)
    ld_ms = timer(st.layout_dispatch, reps)                              # the step's first call
    bcomb_ms = timer(st.combine, reps)                                   # the step's combine, alone
    ucomb_ms = timer(st.combine_unbalanced, reps)                        # moe_combine: static split only
    fp8_ms = timer(lambda: st.dispatch(fp8=True), reps)                  # fused E4M3 quantisation
    fp8in_ms = timer(st.dispatch_fp8_input, reps)                        # E4M3 rows + scales relayed
    wcomb_ms = timer(st.combine_weighted, reps)                          # weighted rows + combined weights
    st.dispatch(fp8=True)                                                # E4M3 rows for the FP8 combine
    fcomb_ms = timer(st.combine_fp8, reps)                               # E4M3 partial rows + scales
    xlay_ms = timer(st.expand_layout, reps)                              # expand mode, each kernel alone
    xdis_ms = timer(st.dispatch_expand, reps)
    xcom_ms = timer(st.combine_expand, reps)
    xstep_ms = timer(st.expand_step, reps)                               # the whole expand-mode step
    moe.check_status(st.status, "dispatch / combine variants")
    NX = int(st.lay.expert_prefix[-1].item())                            # expand rows: valid entries
    # the decode shape (T=128 over R=256): layout + dispatch as two launches and as one
    wd = wl.CONFIGS["decode"]
    sd = Step(moe, wd, wl.make_inputs(dataclass_replace_seed(wd, wd.seed + rank)), device)
    dec = {
        "decode_layout_dispatch_two_us": mean(timer(lambda: (sd.layout(), sd.dispatch()), reps)) * 1e3,
        "decode_layout_dispatch_fused_us": mean(timer(sd.layout_dispatch, reps)) * 1e3,
        "decode_step_two_us": mean(timer(lambda: (sd.layout(), sd.dispatch(), sd.combine()), reps)) * 1e3,
        "decode_step_fused_us": mean(timer(lambda: (sd.layout_dispatch(), sd.combine()), reps)) * 1e3,
    }
    moe.check_status(sd.status, "decode shape")
    del sd
    skewed = measure_skewed(moe, device, rank, timer, reps)
    small = measure_small_configs(moe, device, rank, timer, reps)
    # the fixed cost inside every event-timed figure: a one-kernel graph timed the same way
    tiny = torch.zeros(16, device=device)
    floor_ms = timer(lambda: tiny.add_(1), reps)
    pipelined = measure_pipelined(moe, st, w, device, rank, reps=max(3, min(20, args.steps)))

    peak, peak_kind = hbm_peak()
    ab = algorithmic_bytes(T, H, N, NX)
    bytes_bf16, bytes_fp8, bytes_fp8in = ab["dispatch"], ab["dispatch_fp8"], ab["dispatch_fp8_input"]
    bytes_wcomb, bytes_expand, bytes_fcomb = ab["combine_weighted"], ab["dispatch_expand"], ab["combine_fp8"]
    kern = {
        "layout_us": mean(lay_ms) * 1e3,
        "layout_median_us": med(lay_ms) * 1e3,
        "dispatch_median_us": med(dis_ms) * 1e3,
        "combine_median_us": med(com_ms) * 1e3,
        # dispatch + combine alone, T / (t_dispatch + t_combine)
        "dispatch_combine_tokens_per_s": T / ((mean(dis_ms) + mean(com_ms)) * 1e-3),
        "dispatch_us": mean(dis_ms) * 1e3,
        "combine_us": mean(com_ms) * 1e3,
        "layout_dispatch_us": mean(ld_ms) * 1e3,
        "combine_alone_us": mean(bcomb_ms) * 1e3,
        "combine_unbalanced_us": mean(ucomb_ms) * 1e3,
        "dispatch_fp8_us": mean(fp8_ms) * 1e3,
        "dispatch_fp8_input_us": mean(fp8in_ms) * 1e3,
        "combine_weighted_us": mean(wcomb_ms) * 1e3,
        "combine_fp8_us": mean(fcomb_ms) * 1e3,
        "expand_layout_us": mean(xlay_ms) * 1e3,
        "dispatch_expand_us": mean(xdis_ms) * 1e3,
        "combine_expand_us": mean(xcom_ms) * 1e3,
        "expand_step_us": mean(xstep_ms) * 1e3,
        "expand_step_tokens_per_s": T / (mean(xstep_ms) * 1e-3),
        "expand_rows": NX,
        **dec,
        "timing_floor_us": mean(floor_ms) * 1e3,
        "notes": {
            "timing_floor_us": "a graph holding one 16-element torch add, replayed after the same L2 flush and timed "
                               "the same way: the fixed launch and cold-start cost inside every event-timed figure",
            "dispatch_us, combine_us": "inside the step (the per-kernel breakdown graph); the in-step combine also "
                                       "writes back the dispatch's receive rows still dirty in L2",
            "combine_alone_us": "the step's balanced combine timed alone after an L2 flush",
            "combine_unbalanced_us": "moe_combine (static split, no balance counter) alone after an L2 flush",
        },
    }
    kern["dispatch_gbs"] = gbs(bytes_bf16, mean(dis_ms))
    kern["combine_gbs"] = gbs(bytes_bf16, mean(com_ms))
    kern["combine_alone_gbs"] = gbs(bytes_bf16, mean(bcomb_ms))
    kern["combine_unbalanced_gbs"] = gbs(bytes_bf16, mean(ucomb_ms))
    kern["dispatch_fp8_gbs"] = gbs(bytes_fp8, mean(fp8_ms))
    kern["dispatch_fp8_input_gbs"] = gbs(bytes_fp8in, mean(fp8in_ms))
    kern["combine_weighted_gbs"] = gbs(bytes_wcomb, mean(wcomb_ms))
    kern["combine_fp8_gbs"] = gbs(bytes_fcomb, mean(fcomb_ms))
    kern["dispatch_expand_gbs"] = gbs(bytes_expand, mean(xdis_ms))
    kern["combine_expand_gbs"] = gbs(bytes_expand, mean(xcom_ms))
    for key in ("dispatch", "combine", "combine_alone", "combine_unbalanced", "dispatch_fp8", "dispatch_fp8_input",
                "combine_weighted", "combine_fp8", "dispatch_expand", "combine_expand"):
        kern[f"{key}_frac"] = kern[f"{key}_gbs"] / peak
        kern[f"{key}_frac_of_spec"] = kern[f"{key}_gbs"] / HBM_SPEC_GBS
    skewed_bytes = skewed.pop("_bytes")
    for key, nbytes in skewed_bytes.items():
        skewed[f"{key}_gbs"] = gbs(nbytes, skewed[f"{key}_us"] * 1e-3)
        skewed[f"{key}_frac"] = skewed[f"{key}_gbs"] / peak
    kern["skewed"] = skewed
    kern.update(small)
    kern["pipelined"] = pipelined
    if sus_ms:
        kern["sustained"] = {"steps": len(sus_ms), "ms_per_step_mean": mean(sus_ms),
                             "ms_per_step_median": med(sus_ms), "tokens_per_s": T / (mean(sus_ms) * 1e-3),
                             "how": "the timed step, L2 flushed before each, replayed back to back for "
                                    f"~{args.sustain_s:g} s after the timed steps (64 steps per graph replay, "
                                    "each bracketed by its own events)"}
    dominant = "dispatch" if mean(dis_ms) >= mean(com_ms) else "combine"
    dom_ms = mean(dis_ms) if dominant == "dispatch" else mean(com_ms)
    achieved = gbs(bytes_bf16, dom_ms)
    prof = profiled_traffic(f"{dominant}_kernel", f"{dominant}.cu")
    step_gbs = gbs(2 * bytes_bf16, ms_per_step)

    e2e = run_e2e(moe, st, inp, w, device, args, ref_out, N)

    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 rows, uniform top-8 routing)",
        "config": workload_config(w, N),
        "step": "moe_layout_dispatch (layout, then bf16 dispatch) + moe_combine_ex (balance counter)",
        "timing": timing, "l2": flush_l2.describe(),
        "roofline": {"bound": "hbm", "kernel": f"{dominant}_kernel", "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None if prof is None else prof["in_window"] + prof["writeback"],
                     "traffic_in_window": None if prof is None else prof["in_window"],
                     "traffic_writeback": None if prof is None else prof["writeback"],
                     "traffic_scope": "one launch alone after an L2 flush: the DRAM bytes ncu counts inside the "
                                      "kernel plus the write-back of its output still dirty in L2 when it ends "
                                      "(the writes of the L2-evicting read that follows it, in the same ncu run)",
                     "algorithmic_bytes": bytes_bf16, "spec_peak": HBM_SPEC_GBS,
                     "frac_of_spec": achieved / HBM_SPEC_GBS,
                     "step_achieved": step_gbs, "step_frac": step_gbs / peak,
                     "step_bytes": 2 * bytes_bf16},
        "kernels": kern,
        "gpu_launches": 3 * args.steps,   # per step: the layout kernel (one cluster), the dispatch and the combine
        "clocks": clocks,
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu_baseline:
        cores = host_cores()
        s1, d1 = time_oracle(inp, w, args.cpu_budget)
        sn, dn = time_oracle(inp, w, args.cpu_budget / 2, threads=cores)
        line["cpu_baseline"] = {
            "value": sn * T / dn, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "single_thread_value": s1 * T / d1,
            "sample": f"{sn} full oracle steps of the same workload (layout on one thread; dispatch and combine "
                      f"over token ranges on {cores} threads) in {dn:.1f} s; single-threaded, {s1} steps in "
                      f"{d1:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_pipelined(moe, st, w, device, rank, rounds: int = 10, reps: int = 20):
    """Steps back to back, as a stream of batches runs: 3 * `rounds` steps in one
    CUDA graph, cycling over three full sets of buffers (the timed step's and two
    more with other seeds; a step touches ~0.74 GB of its set, so no step finds
    its inputs or its outputs' lines in the 129 MB L2 from the step before),
    no flush in between, events only at the graph's two ends. Each step
    is the timed one (moe_layout_dispatch + balanced moe_combine_ex); a step's
    launches overlap the previous step's tail as consecutive launches do."""
    sets = [st] + [Step(moe, w, wl.make_inputs(dataclass_replace_seed(w, w.seed + 1000 * (i + 1) + rank)), device)
                   for i in range(2)]
    for s_ in sets:
        s_.layout_dispatch()
        s_.combine()
    torch.cuda.synchronize()
    refs = [s_.out.clone() for s_ in sets]   # each set's step output, which every later run must reproduce
    a = torch.cuda.Event(enable_timing=True, external=True)
    b = torch.cuda.Event(enable_timing=True, external=True)
    M = 3 * rounds
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            a.record()
            for i in range(M):
                sets[i % 3].layout_dispatch()
                sets[i % 3].combine()
            b.record()
    except Exception as exc:   # no graph: nothing to report
        return {"unavailable": type(exc).__name__}
    ms = []
    for i in range(reps + 2):
        g.replay()
        torch.cuda.synchronize()
        if i >= 2:
            ms.append(a.elapsed_time(b) / M)
    for s_, ref in zip(sets, refs):
        moe.check_status(s_.status, "pipelined steps")
        if not torch.equal(s_.out.view(torch.int16), ref.view(torch.int16)):
            raise RuntimeError("pipelined steps: a step's output differs from its first run")
    del g, sets, refs
    torch.cuda.empty_cache()
    per = statistics.fmean(ms)
    return {"steps_per_graph": M, "graphs": reps, "ms_per_step_mean": per,
            "ms_per_step_median": statistics.median(ms), "tokens_per_s": w.num_tokens / (per * 1e-3),
            "how": "3 x 10 steps back to back in one CUDA graph over three sets of buffers (inputs and outputs "
                   "rotated; a step touches ~0.74 GB of its set, far above L2), no flush; events at the graph's "
                   "ends only"}


def measure_skewed(moe, device, rank, timer, reps):
    """The skewed workload (8192 tokens over 64 ranks, Zipf expert popularity)
    with the same kernels and flush discipline: the step and its kernels alone."""
    ws = wl.CONFIGS["skewed"]
    sk = Step(moe, ws, wl.make_inputs(dataclass_replace_seed(ws, ws.seed + rank)), device)
    sk.layout_dispatch()
    sk.combine()
    torch.cuda.synchronize()
    moe.check_status(sk.status, "skewed workload")
    T, H = ws.num_tokens, ws.hidden
    N = int(sk.lay.rank_prefix[-1].item())
    mean = statistics.fmean
    out = {"tokens": T, "hidden": H, "experts": ws.num_experts, "ranks": ws.num_ranks, "topk": ws.num_topk,
           "routing": "Zipf(s=1) expert popularity over a random permutation", "recv_rows": N}
    out["step_us"] = mean(timer(lambda: (sk.layout_dispatch(), sk.combine()), reps)) * 1e3
    out["layout_us"] = mean(timer(sk.layout, reps)) * 1e3
    out["layout_dispatch_us"] = mean(timer(sk.layout_dispatch, reps)) * 1e3
    out["dispatch_us"] = mean(timer(sk.dispatch, reps)) * 1e3
    out["dispatch_fp8_us"] = mean(timer(lambda: sk.dispatch(fp8=True), reps)) * 1e3
    out["combine_us"] = mean(timer(sk.combine, reps)) * 1e3
    out["combine_unbalanced_us"] = mean(timer(sk.combine_unbalanced, reps)) * 1e3
    out["combine_fp8_us"] = mean(timer(sk.combine_fp8, reps)) * 1e3
    moe.check_status(sk.status, "skewed workload")
    out["step_tokens_per_s"] = T / (out["step_us"] * 1e-6)
    row = H * 2
    b = T * row + N * row
    out["_bytes"] = {"step": 2 * b, "dispatch": b, "combine": b, "combine_unbalanced": b,
                     "dispatch_fp8": T * row + N * H + N * (H // 128) * 4,
                     "combine_fp8": N * (H + (H // 128) * 4) + T * row}
    out["notes"] = "every kernel timed alone after an L2 flush (dispatch and combine with balance counters)"
    del sk
    torch.cuda.empty_cache()
    return out


def expected_distinct_ranks(E: int, R: int, k: int) -> float:
    """The pages' closed form for the expected number of distinct ranks a token
    reaches with k experts drawn uniformly without replacement from E experts
    spread evenly over R ranks: R * (1 - C(E - E/R, k) / C(E, k))."""
    import math
    return R * (1.0 - math.comb(E - E // R, k) / math.comb(E, k))


def measure_small_configs(moe, device, rank, timer, reps):
    """The tiny workload's step (two launches and moe_layout_dispatch) and the
    layout-only 2048-expert / 256-rank runs (128 and 2^20 tokens), each timed
    alone with the same flush, with the realised mean number of distinct
    destination ranks per token beside the closed form."""
    mean = statistics.fmean
    out = {}
    wt = wl.CONFIGS["tiny"]
    st = Step(moe, wt, wl.make_inputs(dataclass_replace_seed(wt, wt.seed + rank)), device)
    out["tiny"] = {
        "tokens": wt.num_tokens, "hidden": wt.hidden, "experts": wt.num_experts, "ranks": wt.num_ranks,
        "topk": wt.num_topk,
        "step_two_us": mean(timer(lambda: (st.layout(), st.dispatch(), st.combine()), reps)) * 1e3,
        "step_fused_us": mean(timer(lambda: (st.layout_dispatch(), st.combine()), reps)) * 1e3,
    }
    moe.check_status(st.status, "tiny workload")
    n = int(st.lay.rank_prefix[-1].item())
    out["tiny"]["mean_distinct_ranks"] = n / wt.num_tokens
    out["tiny"]["expected_distinct_ranks"] = expected_distinct_ranks(wt.num_experts, wt.num_ranks, wt.num_topk)
    out["tiny"]["step_fused_tokens_per_s"] = wt.num_tokens / (out["tiny"]["step_fused_us"] * 1e-6)
    del st
    for name in ("layout_2048", "layout_2048_1m"):
        w = wl.CONFIGS[name]
        topk = wl.make_inputs(dataclass_replace_seed(w, w.seed + rank), with_partial=False).topk_idx.to(device)
        lay = moe.Layout.empty(w.num_tokens, w.num_topk, w.num_experts, w.num_ranks, device)
        ws = torch.empty(max(1, moe.moe_get_layout_workspace_size(w.num_tokens, w.num_experts, w.num_ranks)),
                         dtype=torch.uint8, device=device)
        status = moe.new_status(device)
        ms = timer(lambda: moe.moe_get_layout(topk, w.num_experts, w.num_ranks, out=lay, workspace=ws,
                                              status=status), reps)
        moe.check_status(status, name)
        n = int(lay.rank_prefix[-1].item())
        out[name] = {"tokens": w.num_tokens, "experts": w.num_experts, "ranks": w.num_ranks, "topk": w.num_topk,
                     "layout_us": mean(ms) * 1e3, "tokens_per_s": w.num_tokens / (mean(ms) * 1e-3),
                     "mean_distinct_ranks": n / w.num_tokens,
                     "expected_distinct_ranks": expected_distinct_ranks(w.num_experts, w.num_ranks, w.num_topk)}
        del topk, lay, ws
    torch.cuda.empty_cache()
    return out


def run_e2e(moe, st, inp, w, device, args, ref_out, ref_rows):
    """Same step through the public API from pinned host buffers: H2D of the
    step's inputs, a 4-byte read of the receive count, H2D of the partial rows,
    D2H of the combined output -- every step's copies inside the timed region.
    Two steps are in flight on two sets of device buffers: step i's output D2H
    (its own stream) overlaps step i+1's input H2D, since the host link carries
    both directions at once; the host waits only for each step's receive count.
    After the timed steps the last output read back to the host is compared bit
    for bit with the device-resident step's output on the same inputs."""
    T, H = w.num_tokens, w.hidden
    hx = inp.x.pin_memory()
    htopk = inp.topk_idx.pin_memory()
    hw = inp.topk_weights.pin_memory()
    hpart = inp.partial.pin_memory()
    bufs = [st, Step(moe, w, inp, device)]
    houts = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    hcount = [torch.empty(1, dtype=torch.int32).pin_memory() for _ in range(2)]
    s_in, s_comp, s_out = (torch.cuda.Stream(device) for _ in range(3))
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("free", "inp", "cnt", "part", "comb")}
    used = [False, False]

    def step(i):
        b = i % 2
        s = bufs[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev["free"][b])        # the buffer's previous step has been read back
            s.x.copy_(hx, non_blocking=True)
            s.topk.copy_(htopk, non_blocking=True)
            s.wts.copy_(hw, non_blocking=True)
            ev["inp"][b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev["inp"][b])
            s.layout_dispatch()
            hcount[b].copy_(s.lay.rank_prefix[-1:], non_blocking=True)
            ev["cnt"][b].record(s_comp)
        ev["cnt"][b].synchronize()
        n = int(hcount[b].item())
        with torch.cuda.stream(s_in):
            s.partial[:n].copy_(hpart[:n], non_blocking=True)
            ev["part"][b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev["part"][b])
            s.combine()
            ev["comb"][b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comb"][b])
            houts[b].copy_(s.out, non_blocking=True)
            ev["free"][b].record(s_out)
        used[b] = True
        return n

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    K = max(4, args.steps // 2)
    t0 = time.perf_counter()
    ns = [step(args.warmup + i) for i in range(K)]
    torch.cuda.synchronize()
    sec = (time.perf_counter() - t0) / K
    for s in bufs:
        moe.check_status(s.status, "e2e")
    last = houts[(args.warmup + K - 1) % 2]
    same = ns[-1] == ref_rows and torch.equal(last.view(torch.int16), ref_out.cpu().view(torch.int16))
    if not same:
        raise RuntimeError("end-to-end leg: the output read back differs from the device-resident step's")
    n = ns[-1]
    h2d = hx.numel() * 2 + htopk.numel() * 8 + hw.numel() * 4 + n * H * 2
    d2h = 4 + houts[0].numel() * 2
    del bufs[1]
    return {"value": T / sec, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": sec * 1e3, "in_flight": "2 steps: step i's output read-back overlaps step i+1's input copies",
            "output_check": "the last step's output read back to the host equals the device-resident step's "
                            "output on the same inputs, bit for bit (and the same receive-row count)"}


def dataclass_replace_seed(w, seed):
    import dataclasses
    return dataclasses.replace(w, seed=seed)


# ------------------------------------------------------------------ one kernel for an ncu capture

PROFILE_KERNELS = ("layout", "dispatch", "combine", "dispatch_fp8", "combine_fp8", "layout_dispatch", "expand_layout",
                   "step")


def run_profile(args):
    """A small run for ncu: the DeepSeek-V3 workload on cuda:0 (about 2.5 GB
    on the device), a few untimed calls, then, inside the NVTX range
    "profile", ONE call of the chosen kernel(s) after an L2 flush followed by
    an L2-evicting read of a clean buffer larger than L2 (whose DRAM writes are
    the kernel's output left dirty in L2). Capture with
    `ncu --nvtx --nvtx-include "profile/" ...`. No timing is printed: a
    number taken under a profiler is not a measurement."""
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    from combine_moe_get_gb300 import binding as moe
    w = wl.CONFIGS[args.profile_workload]
    st = Step(moe, w, wl.make_inputs(w), device)
    flush_l2 = Flush(device)
    st.layout()
    st.dispatch(fp8=True)                       # E4M3 rows and scales for the FP8 combine's input
    fn = {"layout": st.layout, "dispatch": st.dispatch, "combine": st.combine,
          "dispatch_fp8": lambda: st.dispatch(fp8=True), "combine_fp8": st.combine_fp8,
          "layout_dispatch": st.layout_dispatch, "expand_layout": st.expand_layout,
          "step": lambda: (st.layout_dispatch(), st.combine())}[args.profile_kernel]
    for _ in range(2):
        flush_l2()
        fn()
    flush_l2()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("profile")
    fn()
    flush_l2.evict()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    moe.check_status(st.status, "profile run")
    N = int(st.lay.rank_prefix[-1].item())
    print(json.dumps({"profile_kernel": args.profile_kernel, "workload": w.name, "recv_rows": N}), flush=True)


def _traced(moe, fn, flush_l2, buf, count, what):
    """Records (`what`) of one call of `fn`: captured in a CUDA graph with
    tracing on (the launches keep the trace buffer they were captured with),
    then replayed once after an L2 flush, as the benchmark times it."""
    fn()
    torch.cuda.synchronize()
    moe.trace_enable(buf, count, what)
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
    finally:
        moe.trace_enable(None, None)
    count.zero_()
    flush_l2()
    graph.replay()
    torch.cuda.synchronize()
    return moe.trace_read(buf, count)


def _timeline(moe, rec, rec_phases) -> list:
    """Per kernel, in launch order: CTAs, warps per CTA, SMs, first warp start
    and last warp end (us from the first warp of `rec`), warp lifetimes, CTA
    end times and, where the kernel records them, its phases from `rec_phases`
    (a replay recording phases only): median and longest duration over the
    CTAs, and when the last CTA ended each (us from that replay's first
    stamp)."""
    warps, _ = moe.trace_split(rec)
    _, phases = moe.trace_split(rec_phases)
    t0 = int(warps["start_ns"].min())
    us = lambda ns: round((int(ns) - t0) / 1e3, 2)
    p0 = int(phases["start_ns"].min()) if len(phases) else 0
    pus = lambda ns: round((int(ns) - p0) / 1e3, 2)
    out = []
    for kid in sorted(np.unique(warps["kernel"]), key=lambda k: int(warps["start_ns"][warps["kernel"] == k].min())):
        r = warps[warps["kernel"] == kid]
        life = (r["end_ns"] - r["start_ns"]) / 1e3
        cta_end = np.array([r["end_ns"][r["cta"] == c].max() for c in np.unique(r["cta"])])
        k = {
            "kernel": moe.TRACE_KERNELS.get(int(kid), str(int(kid))), "ctas": int(len(cta_end)),
            "warps_per_cta": int(r["warp"].max()) + 1, "sms": int(len(np.unique(r["sm"]))),
            "first_start_us": us(r["start_ns"].min()), "last_end_us": us(r["end_ns"].max()),
            "warp_life_us": {"median": round(float(np.median(life)), 2), "max": round(float(life.max()), 2)},
            "cta_end_us": {q: us(np.percentile(cta_end, p)) for q, p in (("min", 0), ("p50", 50), ("max", 100))},
        }
        ph = phases[phases["kernel"] == kid]
        names = moe.TRACE_PHASE_NAMES.get(int(kid), ())
        if len(ph) and names:
            k["phases"] = []
            for i, name in enumerate(names, start=1):
                q = ph[ph["warp"] == moe.TRACE_PHASE + i]
                if not len(q):
                    continue
                d = (q["end_ns"] - q["start_ns"]) / 1e3
                k["phases"].append({"phase": name, "median_us": round(float(np.median(d)), 2),
                                    "max_us": round(float(d.max()), 2), "last_end_us": pus(q["end_ns"].max())})
        out.append(k)
    return out


def run_trace(args):
    """Timelines from the tracing build of the library (compiled with
    MOE_PROFILE): one step (moe_layout_dispatch, then moe_combine_ex with a
    balance counter) and the dispatch, combine, quantising dispatch and FP8
    combine called alone, each replayed from a CUDA graph after an L2 flush.
    Per kernel: CTAs, warps per CTA, SMs used, when its first warp started and
    its last warp ended, how long its warps lived, when its CTAs finished and,
    for the cluster layout, dispatch and combine, the phases of its CTAs.
    Per lone call also its span (first warp start to last warp end), and its
    algorithmic bytes over the span as a fraction of the measured copy
    bandwidth. The warps' records come from one replay and the phases from
    another that records nothing else (a warp record costs its warp an
    atomic, which slows the layout). These are a timeline; the event-timed
    figures of the benchmark are the measurement."""
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    from combine_moe_get_gb300 import binding as moe
    from combine_moe_get_gb300 import build as moe_build
    w = wl.CONFIGS[args.profile_workload]
    tl = moe.load_library(moe_build.build_trace())
    peak, peak_kind = hbm_peak()
    with moe.using(tl):
        st = Step(moe, w, wl.make_inputs(w), device)
        flush_l2 = Flush(device)
        for _ in range(3):
            flush_l2()
            st.layout_dispatch()
            st.combine()
        st.dispatch(fp8=True)       # E4M3 rows and scales for the FP8 combine's input
        torch.cuda.synchronize()
        N = int(st.lay.rank_prefix[-1].item())
        ab = algorithmic_bytes(w.num_tokens, w.hidden, N, 0)
        buf = torch.zeros((1 << 20) * moe.TRACE_RECORD.itemsize, dtype=torch.uint8, device=device)
        count = torch.zeros(1, dtype=torch.int32, device=device)
        step = lambda: (st.layout_dispatch(), st.combine())
        rec = _traced(moe, step, flush_l2, buf, count, moe.TRACE_WARPS)
        n_step = int(count.item())
        rec_ph = _traced(moe, step, flush_l2, buf, count, moe.TRACE_PHASES)
        calls = {}
        for name, fn in (("dispatch", st.dispatch), ("combine", st.combine),
                         ("dispatch_fp8", lambda: st.dispatch(fp8=True)), ("combine_fp8", st.combine_fp8)):
            r = _traced(moe, fn, flush_l2, buf, count, moe.TRACE_WARPS)
            r_ph = _traced(moe, fn, flush_l2, buf, count, moe.TRACE_PHASES)
            span_us = (int(r["end_ns"].max()) - int(r["start_ns"].min())) / 1e3
            calls[name] = {"span_us": round(span_us, 2), "algorithmic_bytes": ab[name],
                           "gbs_over_span": round(gbs(ab[name], span_us * 1e-3), 1),
                           "frac_over_span": round(gbs(ab[name], span_us * 1e-3) / peak, 3),
                           "kernels": _timeline(moe, r, r_ph)}
        moe.check_status(st.status, "traced calls")
    stamps = np.unique(np.concatenate([rec["start_ns"], rec["end_ns"]]))
    print(json.dumps({"trace": w.name, "records": n_step, "recv_rows": N,
                      "step_us": round((int(rec["end_ns"].max()) - int(rec["start_ns"].min())) / 1e3, 2),
                      "timer_step_ns": int(np.diff(stamps).min()) if len(stamps) > 1 else None,
                      "kernels": _timeline(moe, rec, rec_ph), "calls": calls,
                      "peak": {"gbs": peak, "kind": peak_kind}}), flush=True)


# ------------------------------------------------------------------ reference arm (CPU oracle)

def run_reference(args, world, rank):
    """The CPU oracle on the same workload: each step is the oracle's layout,
    bf16 dispatch and combine over all 4096 tokens, the dispatch and the
    combine over token ranges on every host core (the same per-token code and
    results as single-threaded). Under torchrun only rank 0 runs it."""
    if rank != 0:
        return
    import oracle
    w = wl.CONFIGS[WORKLOAD]
    inp = wl.make_inputs(w)
    cores = host_cores()
    time_oracle(inp, w, 0.0, min_steps=args.warmup, threads=cores)
    steps, dt = time_oracle(inp, w, 0.0, min_steps=args.steps, threads=cores)
    value = steps * w.num_tokens / dt
    N = oracle.layout(inp.topk_idx.numpy(), w.num_experts, w.num_ranks)["num_recv"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 rows, uniform top-8 routing)",
        "config": workload_config(w, N),
        "step": "layout + bf16 dispatch + combine (CPU oracle; dispatch and combine over token ranges on every "
                "host core)",
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{steps} full oracle steps over all {w.num_tokens} tokens of the workload "
                                   f"(layout on one thread; dispatch and combine on {cores} threads)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of single-threaded oracle work for cpu_baseline (half that threaded)")
    ap.add_argument("--sustain-s", type=float, default=2.0,
                    help="seconds of back-to-back flushed steps after the timed ones, under the clock sampler")
    ap.add_argument("--profile-kernel", choices=PROFILE_KERNELS, default=None,
                    help="run one call of this kernel for an ncu capture instead of the benchmark")
    ap.add_argument("--profile-workload", choices=["dsv3", "skewed", "decode"], default=WORKLOAD)
    ap.add_argument("--trace", action="store_true",
                    help="print one step's per-kernel timeline from the tracing build instead of the benchmark")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.profile_kernel:
        run_profile(args)
        return
    if args.trace:
        run_trace(args)
        return
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
