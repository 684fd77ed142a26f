"""Benchmark of the HiSA decode step (score + select + attend) on GB300.

Workload: R independent V4-Flash-shaped decode queries per step (each: Np = 32768
pooled rows of a 131072-token prefix, H_i = 64 x D_i = 128 indexer, index_block = 64,
keep = 16, index_topk = 512, 64 query heads x Dh = 512, window 128, bf16 keys / KV,
f32 indexer q). One step = the newest block mean of every sequence appended to the
block-mean cache, the coarse block filter, the fine top-k and the sparse combine: three
C-ABI calls (hisa_block_filter_append, hisa_select_topk, hisa_sparse_attend). The headline
replays the K timed steps as one CUDA graph (two batches alternating, each kernel chained to
the one before it by programmatic dependent launch); the stage times come from one graph per
call.

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from deepseek_sparse_attention_hisa_gb300 import inputs  # noqa: E402

METRIC = "HiSA decode queries/s (score+select+attend) and HBM GB/s vs GB300 peak"
UNIT = "queries/s"
L2_FLUSH_BYTES = 256 << 20


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ----------------------------------------------------------------------------
# algorithmic bytes per decode query (V4-Flash shape), by stage
# ----------------------------------------------------------------------------
def stage_bytes(wl, nb):
    H_i, D_i, b, keep, k, H, Dh, W = (wl.H_i, wl.D_i, wl.index_block, wl.index_keep,
                                      wl.index_topk, wl.H, wl.Dh, wl.window)
    q_idx = H_i * D_i * 4
    w = H_i * 4
    means = b * D_i * 2 + D_i * 4                        # newest block: read b keys, write 1 mean
    filt = q_idx + w + nb * D_i * 4 + keep * 4           # q, w, all block means, top_blk
    sel = q_idx + w + keep * b * D_i * 2 + keep * 4 + k * 4   # q, w, kept blocks' keys, top_blk, I
    att = H * Dh * 2 + W * Dh * 2 + k * Dh * 2 + k * 4 + H * 4 + H * Dh * 4  # q, local, gathered, I, sinks, out
    # unique bytes of the whole step: q/w and I/top_blk counted once
    step = means + q_idx + w + nb * D_i * 4 + keep * b * D_i * 2 + H * Dh * 2 + W * Dh * 2 + \
        k * Dh * 2 + H * 4 + H * Dh * 4 + k * 4 + keep * 4
    return dict(block_filter_append=means + filt, select_topk=sel, sparse_attend=att), step


def step_bytes_rows(wl, nb, L):
    """Unique algorithmic bytes of one sequence's step with L query rows (decode: L = 1):
    per sequence the newest block's keys in and its mean out, all nb block means, the local
    rows (window + L - 1) and the sinks; per row q, w, the kept blocks' keys, top_blk, I,
    the attention q, the gathered rows and the output (rows select their own sets)."""
    H_i, D_i, b, keep, k, H, Dh, W = (wl.H_i, wl.D_i, wl.index_block, wl.index_keep,
                                      wl.index_topk, wl.H, wl.Dh, wl.window)
    per_seq = b * D_i * 2 + D_i * 4 + nb * D_i * 4 + (W + L - 1) * Dh * 2 + H * 4
    per_row = (H_i * D_i * 4 + H_i * 4 + keep * b * D_i * 2 + keep * 4 + k * 4 +
               H * Dh * 2 + k * Dh * 2 + H * Dh * 4)
    return per_seq + L * per_row


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    """SM clock, power and clock-event reasons of one GPU, polled every ~1 ms through NVML
    (read-only queries) while the timed region runs; nvidia-smi at 20 ms if NVML is not
    loadable. Only samples taken between mark_start() and mark_stop() are summarised."""
    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index: int):
        self.cuda_index = cuda_index
        self.samples = []          # (time, sm_mhz, reasons set)
        self.sm_max = None
        self.source = None
        self.t0 = self.t1 = None
        self._stop = threading.Event()
        self.proc = None
        self.thread = None

    # -- device handle ---------------------------------------------------------
    def _nvml_handle(self, nv):
        import ctypes
        h = ctypes.c_void_p()
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.cuda_index).uuid)
            key = ("GPU-" + uuid if not uuid.startswith("GPU-") else uuid).encode()
            if nv.nvmlDeviceGetHandleByUUID(key, ctypes.byref(h)) == 0:
                return h
        except Exception:
            pass
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        idx = self.cuda_index
        if ids and self.cuda_index < len(ids):
            if ids[self.cuda_index].isdigit():
                idx = int(ids[self.cuda_index])
            elif nv.nvmlDeviceGetHandleByUUID(ids[self.cuda_index].encode(),
                                              ctypes.byref(h)) == 0:
                return h
        if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(h)) == 0:
            return h
        return None

    def _nvml_loop(self, nv, h):
        import ctypes
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.perf_counter()
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                    nv.nvmlDeviceGetCurrentClocksThrottleReasons(h, ctypes.byref(rs)) == 0:
                names = {n for bit, n in self.REASONS.items() if rs.value & bit}
                self.samples.append((t, float(clk.value), names))
            time.sleep(0.001)

    def _smi_loop(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.proc.stdout:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            self.sm_max = smax
            rs = {n for n, v in zip(names, parts[4:8]) if v.lower().startswith("active")}
            self.samples.append((time.perf_counter(), sm, rs))

    def __enter__(self):
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = self._nvml_handle(nv)
            if h is None:
                raise OSError("no NVML handle")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.sm_max = float(mx.value)
            self.source = "nvml 1 ms"
            self.thread = threading.Thread(target=self._nvml_loop, args=(nv, h), daemon=True)
            self.thread.start()
        except Exception:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.cuda_index), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi 20 ms"
                self.thread = threading.Thread(target=self._smi_loop, daemon=True)
                self.thread.start()
                deadline = time.perf_counter() + 5.0   # wait for the first sample
                while not self.samples and time.perf_counter() < deadline:
                    time.sleep(0.01)
            except Exception:
                self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_stop(self):
        self.t1 = time.perf_counter()

    def __exit__(self, *a):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        t0 = self.t0 if self.t0 is not None else -1e30
        t1 = self.t1 if self.t1 is not None else 1e30
        inside = [(sm, rs) for t, sm, rs in self.samples if t0 <= t <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.sm_max, "reasons": ["unsampled"],
                    "samples": 0, "source": self.source}
        reasons = set()
        for _, rs in inside:
            reasons |= rs
        return {"sm_mhz": statistics.median(sm for sm, _ in inside), "sm_max_mhz": self.sm_max,
                "reasons": sorted(reasons), "samples": len(inside), "source": self.source}


# ----------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)
# ----------------------------------------------------------------------------
def host_copy_of_sequence(data, b):
    """Host numpy copy of sequence b of a device-drawn batch (bf16 -> uint16 bits)."""
    import torch

    def h(t):
        t = t.detach().cpu()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()
    k0, k1 = int(data["key_off"][b]), int(data["key_off"][b + 1])
    return dict(q_idx=h(data["q_idx"][b, 0]), w=h(data["w"][b, 0]), keys=h(data["keys"][k0:k1]),
                q_attn=h(data["q_attn"][b]), local_kv=h(data["local_kv"][b]),
                local_pos0=int(data["local_pos0"][b]), pooled_kv=h(data["pooled_kv"][k0:k1]),
                sinks=h(data["sinks"]), t0=int(data["t0"][b]))


def oracle_query(wl, s):
    from oracle import hisa_oracle as O
    d = O.hisa_select_decode(s["q_idx"], s["w"], s["keys"], wl.index_block, wl.index_keep,
                             wl.index_topk)
    O.sparse_combine(s["q_attn"], s["local_kv"], s["local_pos0"], s["pooled_kv"], d["I"][None],
                     s["sinks"], s["t0"], wl.r, wl.window)


def time_oracle(wl, samples, budget_s):
    n = 0
    t_start = time.perf_counter()
    while True:
        oracle_query(wl, samples[n % len(samples)])
        n += 1
        el = time.perf_counter() - t_start
        if el >= budget_s:
            break
    return n, el


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def host_samples(wl, n):
    """n sequences drawn on the host (the oracle's input), same recipe as the batch."""
    one = wl.replace(B=n)
    data = inputs.generate(one)
    out = []
    for b in range(n):
        k0, k1 = int(data["key_off"][b]), int(data["key_off"][b + 1])
        out.append(dict(q_idx=data["q_idx"][b, 0], w=data["w"][b, 0], keys=data["keys"][k0:k1],
                        q_attn=data["q_attn"][b], local_kv=data["local_kv"][b],
                        local_pos0=int(data["local_pos0"][b]),
                        pooled_kv=data["pooled_kv"][k0:k1], sinks=data["sinks"],
                        t0=int(data["t0"][b])))
    return out


def run_reference(args, wl, R):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    samples = host_samples(wl, 2)
    per_step = max(1, int(args.ref_queries))
    for _ in range(args.warmup):
        oracle_query(wl, samples[0])
    t0 = time.perf_counter()
    for s in range(args.steps):
        for q in range(per_step):
            oracle_query(wl, samples[(s * per_step + q) % len(samples)])
    el = time.perf_counter() - t0
    value = args.steps * per_step / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"v4flash_decode (Np=32768, H_i=64x128, H=64x512, W=128); "
                               f"each step {per_step} of the R={R} queries, CPU oracle",
                   "queries_per_step": per_step},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores_used(), "kind": "oracle",
                         "sample": f"{args.steps * per_step} queries over 2 host-drawn sequences"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def traffic_from_profile(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu capture, or None once the
    kernel's sources have changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        ent = t.get(kernel)
        if not ent:
            return None
        from deepseek_sparse_attention_hisa_gb300 import build
        if ent.get("source_stamp") != build.kernel_stamp(kernel):
            return None
        return ent.get("bytes_per_launch")
    except Exception:
        return None


def max_over_ranks(ms, device):
    """The slowest rank's time (every rank gets it); the value itself at world size 1."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, R, K, total_ms):
    """Whole-job queries/s: every rank runs R independent queries per step (weak scaling)."""
    return world * R * K / (total_ms / 1e3)


def run_gpu(args, wl, R):
    import torch
    import torch.distributed as dist

    from deepseek_sparse_attention_hisa_gb300 import binding as hb
    from deepseek_sparse_attention_hisa_gb300 import build
    from deepseek_sparse_attention_hisa_gb300.problem import Problem

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    build.build_library()
    hb.lib()

    bwl = wl.replace(B=R, Np=(int(args.Np),))
    data = inputs.generate_device(bwl, device=dev, seed=1000 + rank)
    prob = Problem(data, device=dev)
    nb = int(prob.nb[0])
    newest = torch.as_tensor(np.full(R, nb - 1, dtype=np.int32), device=dev)
    prob.block_means()                               # cache of completed blocks
    # a second, disjoint batch of R sequences: the headline alternates the two, so that
    # a step's inputs were last touched two steps (2 x ~430 MB) earlier
    prob_b = Problem(inputs.generate_device(bwl, device=dev, seed=1100 + rank), device=dev)
    prob_b.block_means()
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)
    # the newest block's mean is appended every step (a new block completes every
    # r * index_block = 256 tokens in a real decode loop: this recomputes it each step)
    stages = ["block_filter_append", "select_topk", "sparse_attend"]

    def calls_for(pr):
        return {
            "block_filter_append": lambda s: pr.block_filter_append(first_block=newest, stream=s),
            "select_topk": lambda s: pr.select_topk(stream=s, chained=True),
            "sparse_attend": lambda s: pr.attend(stream=s, chained=True),
        }
    calls = calls_for(prob)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for name in stages:                          # eager warm-up: attributes, lazy init
            calls[name](stream)
    stream.synchronize()
    graphs = {}
    for name in stages:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            calls[name](stream)
        graphs[name] = g
    # the whole step as one graph (the headline), and one graph per stage (stage times)
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        for name in stages:
            calls[name](stream)
    # headline graph: a step of batch A then a step of batch B, chained kernel to kernel
    calls_b = calls_for(prob_b)
    with torch.cuda.stream(stream):
        for name in stages:
            calls_b[name](stream)
    stream.synchronize()
    g_rot = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_rot, stream=stream):
        for cl in (calls, calls_b):
            for name in stages:
                cl[name](stream)

    def chain_graph(n, names):
        """n rounds of the given calls, batch A then batch B alternating, as ONE graph: each
        kernel is programmatically chained to the one before it, as inside g_rot, and no graph
        launch (which nothing overlaps: ~6 us each, measured) falls between two of them."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                cl = calls if i % 2 == 0 else calls_b
                for name in names:
                    cl[name](stream)
        return g

    # headline graph: the K timed steps themselves, A, B, A, ... chained kernel to kernel
    g_head = chain_graph(args.steps, stages)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    scrub = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2(write_only=False):
        """Evict the step's inputs from L2: write a buffer larger than L2, then read another
        one, so that L2 holds clean lines of neither (a step does not write back the flush's
        dirty lines). write_only keeps the dirty lines, for the comparison line."""
        flush.zero_()
        if not write_only:
            torch.sum(scrub, dim=0, out=sink)

    def step(evs=None):
        """One step from the per-stage graphs, with an event after every stage."""
        if evs is not None:
            evs[0].record(stream)
        for i, name in enumerate(stages):
            graphs[name].replay()
            if evs is not None:
                evs[i + 1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_l2()
            g_step.replay()
            flush_l2()
            step()
        for _ in range((args.warmup + 1) // 2):
            g_rot.replay()
        g_head.replay()                              # untimed: the graph's first launch
    stream.synchronize()
    assert prob.status(stream) == 0 and prob_b.status(stream) == 0, \
        "device status flags set during warm-up"

    K = args.steps
    # ---- headline: K steps back to back, batches A and B alternating (no flush: the step
    # inputs, ~430 MB per batch, are over 3x the L2; each batch is reused every other step)
    rot_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.mark_start()
        t_wall = time.perf_counter()
        with torch.cuda.stream(stream):
            rot_ev[0].record(stream)
            g_head.replay()
            rot_ev[1].record(stream)
        stream.synchronize()
        t_wall = time.perf_counter() - t_wall
        clk.mark_stop()
    torch.cuda.synchronize()
    rot_total_ms = max_over_ranks(rot_ev[0].elapsed_time(rot_ev[1]), dev)
    assert prob.status(stream) == 0 and prob_b.status(stream) == 0, \
        "device status flags set during the timed region"
    del g_head
    # the same K steps from graphs of two steps (A then B) replayed K / 2 times: a graph launch
    # between every second step (reported beside the value, not as it)
    two_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    with torch.cuda.stream(stream):
        two_ev[0].record(stream)
        for _ in range(K // 2):
            g_rot.replay()
        if K % 2:
            g_step.replay()
        two_ev[1].record(stream)
    stream.synchronize()
    two_step_ms = max_over_ranks(two_ev[0].elapsed_time(two_ev[1]), dev) / K
    # each stage's kernel back to back the same way (batch A, batch B, A, ...): its average
    # launch duration in steady state, the roofline's denominator
    stage_rot_ms = {}
    n_launch = 2 * max(K // 2, 1)
    for name in stages:
        g2 = chain_graph(n_launch, [name])
        ev2 = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        with torch.cuda.stream(stream):
            g2.replay()
            ev2[0].record(stream)
            g2.replay()
            ev2[1].record(stream)
        stream.synchronize()
        stage_rot_ms[name] = max_over_ranks(ev2[0].elapsed_time(ev2[1]), dev) / n_launch
        del g2
    assert prob.status(stream) == 0 and prob_b.status(stream) == 0
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(K)]
    wo_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(K)]
    # ---- the same step with the L2 flushed before each one (timed one by one), per stage,
    # and after a write-only flush
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk_f:
        clk_f.mark_start()
        with torch.cuda.stream(stream):
            for i in range(K):                      # whole-step graph
                flush_l2()                          # L2 flush outside the step's events
                step_ev[i][0].record(stream)
                g_step.replay()
                step_ev[i][1].record(stream)
            for i in range(K):                      # stage times: per-stage graphs
                flush_l2()
                step(evs[i])
            for i in range(K):                      # the same step after a write-only flush
                flush_l2(write_only=True)
                wo_ev[i][0].record(stream)
                g_step.replay()
                wo_ev[i][1].record(stream)
        stream.synchronize()
        clk_f.mark_stop()
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    wo_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in wo_ev), dev) / K
    stage_ms = {name: [evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K)]
                for j, name in enumerate(stages)}
    flushed_ms = max_over_ranks(sum(step_ms), dev) / K
    ms_per_step = rot_total_ms / K
    value = job_value(world, R, K, rot_total_ms)

    # e2e: the same step through the public API from pinned host buffers, with the
    # per-step query inputs copied in and the results (out, I) copied back.
    host_in = {n: data[n].detach().cpu().pin_memory() for n in ("q_idx", "w", "q_attn")}
    host_out = {"out": torch.empty_like(prob.out, device="cpu").pin_memory(),
                "I": torch.empty_like(prob.I, device="cpu").pin_memory()}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
    with torch.cuda.stream(stream):
        for i in range(K):
            flush_l2()
            e2e_ev[i][0].record(stream)
            prob.q_idx.copy_(host_in["q_idx"], non_blocking=True)
            prob.w.copy_(host_in["w"], non_blocking=True)
            prob.q_attn.copy_(host_in["q_attn"], non_blocking=True)
            g_step.replay()
            host_out["out"].copy_(prob.out, non_blocking=True)
            host_out["I"].copy_(prob.I, non_blocking=True)
            e2e_ev[i][1].record(stream)
    stream.synchronize()
    e2e_serial_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev) / K, dev)
    assert prob.status(stream) == 0, "device status flags set during the timed region"
    e2e_ms = e2e_pipelined(prob, host_in, host_out, calls_for, K, dev)
    e2e_direct_ms = e2e_pipelined(prob, host_in, host_out, calls_for, K, dev, direct_out=True)
    # the same, with the combine's output rounded to bf16 (hisa_attn_desc.out_dtype): half the
    # bytes copied back; reported beside the f32 figures, never as the value
    prob16 = prob.with_out("bf16")
    host_out16 = {"out": torch.empty_like(prob16.out, device="cpu").pin_memory(),
                  "I": host_out["I"]}
    d2h16 = sum(t.numel() * t.element_size() for t in host_out16.values())
    e2e_b16_ms = e2e_pipelined(prob16, host_in, host_out16, calls_for, K, dev)

    per_stage_bytes, step_bytes = stage_bytes(wl, nb)
    peak, peak_src = peaks()
    stage_avg = {n: statistics.mean(v) for n, v in stage_ms.items()}
    dom = max(stage_rot_ms, key=stage_rot_ms.get)
    achieved = per_stage_bytes[dom] * R / (stage_rot_ms[dom] / 1e3) / 1e9
    kernel_of = {"block_filter_append": "k_score_pipe", "select_topk": "k_score_pipe",
                 "sparse_attend": "k_attend_tc"}
    traffic = traffic_from_profile(kernel_of[dom]) if dom == "sparse_attend" else None

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"v4flash_decode x R={R} independent sequences per GPU "
                               f"(Np={args.Np} each, H_i=64x128, b=64, keep=16, k=512, "
                               f"H=64x512 bf16, W=128)",
                   "R": R, "Np": int(args.Np),
                   "l2": "inputs larger than L2: K steps back to back alternating two disjoint "
                         f"batches of R sequences ({step_bytes * R / 1e6:.0f} MB touched per step, "
                         f"{2 * step_bytes * R / 1e6:.0f} MB between two uses of a batch, L2 129 MB); "
                         "'flushed' has the same step timed one by one after an L2 flush"},
        "flushed": {"ms_per_step": flushed_ms, "value": job_value(world, R, 1, flushed_ms),
                    "step_hbm_gbs": step_bytes * R / (flushed_ms / 1e3) / 1e9,
                    "how": "before each step (outside its events): 256 MiB written, then 256 MiB "
                           "read, so no step input and no dirty flush line is in L2",
                    "clocks": clk_f.summary()},
        "ms_per_step_after_write_only_flush": wo_ms,
        "ms_per_step_two_step_graphs": two_step_ms,
        "ms_per_step_how": "the K timed steps as one graph, batches A and B alternating, every kernel "
                           "programmatically chained to the one before; ms_per_step_two_step_graphs: "
                           "the same steps from a graph of two (A, B) replayed K / 2 times, a graph "
                           "launch between every second step",
        "step_hbm_gbs": step_bytes * R / (ms_per_step / 1e3) / 1e9,
        "step_bytes_per_query": step_bytes,
        "stages_us": {n: v * 1e3 for n, v in stage_rot_ms.items()},
        "stages_us_how": "each stage's kernel launched back to back over the two batches (A, B, A, "
                         "..., one graph of 2 x (K / 2) launches, each chained to the one before), "
                         "average per launch; stages_us_flushed: one launch at a time after an L2 "
                         "flush",
        "stages_us_flushed": {n: v * 1e3 for n, v in stage_avg.items()},
        "roofline": {"bound": "hbm", "kernel": kernel_of[dom], "stage": dom, "achieved": achieved, "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic},
        # headline, two-step graphs, flushed whole-step, per-stage and write-only passes,
        # back-to-back stages
        "gpu_launches": 6 * K * launches_per_step(prob),
        "e2e": {"value": job_value(world, R, 1, min(e2e_ms, e2e_direct_ms)), "unit": UNIT,
                "copied_out_value": job_value(world, R, 1, e2e_ms),
                "direct_out_value": job_value(world, R, 1, e2e_direct_ms),
                "serial_value": job_value(world, R, 1, e2e_serial_ms),
                "bf16_out_value": job_value(world, R, 1, e2e_b16_ms),
                "bf16_out_d2h_bytes_per_step": d2h16,
                "how": "two buffer sets: step i's inputs copied in and step i-1's results copied "
                       "out on their own streams while step i computes; every step's copies are "
                       "in the timed region. value = the better of copied_out_value (out and I "
                       "copied back by cudaMemcpy) and direct_out_value (the combine writes out "
                       "straight into page-locked host memory, I copied back); serial_value: copy "
                       "in, step, copy out, one after the other, L2 flushed before each; "
                       "bf16_out_value: as copied_out_value with out rounded to bf16 by the "
                       "combine (out_dtype = HISA_BF16), not part of value",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "wall_s": t_wall,
    }
    clocks = clk.summary()
    line["clocks"] = clocks
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        samples = [host_copy_of_sequence(data, 0)]
        n, el = time_oracle(wl, samples, args.cpu_seconds)
        line["cpu_baseline"] = {"value": n / el, "unit": UNIT, "cores": cores_used(),
                                "kind": "oracle",
                                "sample": f"{n} queries of sequence 0 of the batch, {el:.1f} s"}
    # single-GPU side legs (a multi-GPU run reports the scaling line only)
    if not args.no_prefill and world == 1:
        line["prefill_scoring"] = run_prefill_scoring(args, dev, stream)
    if not args.no_extra and world == 1:
        line["latency_one_query"] = run_latency(wl, dev, stream)
        line["long_context_selection"] = run_long_context(dev, stream)
        line["prefill_hisa_step"] = run_prefill_hisa(dev, stream)
        line["ragged_decode_b32"] = run_ragged(dev, stream)
        line["verify_L4"] = run_verify(dev, stream)
        line["compressor_append"] = run_compress(dev, stream, R)
        line["r_sweep"] = run_r_sweep(dev, stream)
        line["per_step_means"] = run_per_step_means(dev, stream, R)
    if not args.no_np_sweep and world == 1:
        line["decode_np_sweep"] = run_np_sweep(dev, stream, R)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def prefill_flops(wl):
    """Unmasked flops of the dense prefill scoring: sum over rows j of V(t0 + j) keys x
    H_i heads x D_i dims x 2 (multiply and add)."""
    Np = int(wl.Np[0])
    V = np.minimum(Np, (wl.t0 + np.arange(wl.L) + 1) // wl.r)
    return int(V.sum()) * wl.H_i * wl.D_i * 2


def run_prefill_scoring(args, dev, stream):
    """hisa_index_scores on the batched-prefill workload (L = 4096 rows, Np = 16384 bf16
    keys, bf16 q): the dense L x Np x (H_i * D_i) contraction, timed with CUDA events."""
    import torch

    from deepseek_sparse_attention_hisa_gb300.problem import Problem
    wl = inputs.WORKLOADS["prefill"].replace(with_attention=False)
    data = inputs.generate_device(wl, device=dev, seed=3000)
    prob = Problem(data, device=dev)
    scores = torch.empty((wl.L, int(wl.Np[0])), dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            prob.index_scores(scores, stream=stream)
    stream.synchronize()
    n = 10
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            a.record(stream)
            prob.index_scores(scores, stream=stream)
            b.record(stream)
    stream.synchronize()
    assert prob.status(stream) == 0
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    flops = prefill_flops(wl)
    peak = bf16_peak()
    return {"workload": "prefill L=4096 x Np=16384 x (64 x 128), bf16 q and keys, causal",
            "ms": ms, "flops": flops, "tflops": flops / ms / 1e9, "peak_tflops": peak[0],
            "peak_source": peak[1], "frac": flops / ms / 1e9 / peak[0]}


class L2Flush:
    """Evicts every input from L2 between timed iterations: a 256 MiB write, then a 256 MiB
    read, so that L2 holds clean lines of neither (a timed region does not write back the
    flush's own dirty lines)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self, write_only=False):
        import torch
        self.w.zero_()
        if not write_only:
            torch.sum(self.r, dim=0, out=self.sink)


def timed_graph(g, stream, flush, n):
    """Mean and median ms of n replays of CUDA graph g, each after an L2 flush (outside the
    events), timed with events on the launching stream."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            flush()
            a.record(stream)
            g.replay()
            b.record(stream)
    stream.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    return statistics.mean(ms), statistics.median(ms)


def capture(fn, stream):
    import torch
    with torch.cuda.stream(stream):
        fn(stream)                                   # eager warm-up
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn(stream)
    return g


def decode_leg(wl, dev, stream, flush, n, seed, what):
    """One step over wl's batch (newest block means appended, coarse filter, fine top-k,
    combine; the last two chained), captured as one graph and timed after an L2 flush.
    Bytes are the step's unique algorithmic bytes (step_bytes_rows) summed over sequences."""
    import torch

    from deepseek_sparse_attention_hisa_gb300.problem import Problem
    data = inputs.generate_device(wl, device=dev, seed=seed)
    prob = Problem(data, device=dev)
    newest = torch.as_tensor((prob.nb - 1).astype(np.int32), device=dev)
    prob.block_means()
    torch.cuda.synchronize()

    stages = {"block_filter_append": lambda s: prob.block_filter_append(first_block=newest, stream=s),
              "select_topk": lambda s: prob.select_topk(stream=s, chained=True),
              "sparse_attend": lambda s: prob.attend(stream=s, chained=True)}

    def step(s):
        for fn in stages.values():
            fn(s)
    g = capture(step, stream)
    mean, med = timed_graph(g, stream, flush, n)
    stage_us = {k: timed_graph(capture(fn, stream), stream, flush, n)[0] * 1e3
                for k, fn in stages.items()}
    assert prob.status(stream) == 0, f"device status flags set in the {what} leg"
    nbytes = sum(step_bytes_rows(wl, int(nb), wl.L) for nb in prob.nb)
    peak, src = peaks()
    rows = wl.B * wl.L
    out = {"us_per_step": mean * 1e3, "us_median": med * 1e3, "stages_us": stage_us,
           "rows_per_step": rows,
           "rows_per_s": rows / (mean / 1e3), "ns_per_row": mean * 1e6 / rows,
           "bytes_per_step": nbytes, "hbm_gbs": nbytes / (mean / 1e3) / 1e9,
           "frac": nbytes / (mean / 1e3) / 1e9 / peak, "peak_source": src}
    del prob, data, g
    torch.cuda.empty_cache()
    return out


def run_per_step_means(dev, stream, R, n=10):
    """The decode step with every block mean recomputed from the keys each step
    (hisa_block_means over all blocks, then the coarse filter, fine top-k and combine)
    instead of the cached means with the newest block appended: the reading of the
    pages' step that keeps no cache. Reported beside the headline, never as it; its
    bytes add every sequence's Np keys (8 MiB at Np = 32768)."""
    import torch

    from deepseek_sparse_attention_hisa_gb300.problem import Problem
    wl = inputs.WORKLOADS["v4flash_decode"].replace(B=R, Np=(32768,))
    data = inputs.generate_device(wl, device=dev, seed=7000)
    prob = Problem(data, device=dev)
    def step(s):
        prob.block_means(stream=s)                       # every block of every sequence
        prob.block_filter(stream=s)
        prob.select_topk(stream=s, chained=True)
        prob.attend(stream=s, chained=True)
    g = capture(step, stream)
    flush = L2Flush(dev)
    mean, med = timed_graph(g, stream, flush, n)
    gm = capture(lambda s: prob.block_means(stream=s), stream)
    means_ms, _ = timed_graph(gm, stream, flush, n)
    assert prob.status(stream) == 0
    nb = int(prob.nb[0])
    keys = int(wl.Np[0]) * wl.D_i * 2
    # step_bytes_rows counts the newest block's keys and mean; here all keys are read and
    # all nb means written (and read back by the coarse filter)
    per_seq = step_bytes_rows(wl, nb, 1) - (wl.index_block * wl.D_i * 2 + wl.D_i * 4) + keys + nb * wl.D_i * 4
    nbytes = R * per_seq
    peak, src = peaks()
    out = {"workload": f"v4flash_decode, R = {R} queries per step, Np = 32768, block means recomputed each step",
           "us_per_step": mean * 1e3, "us_median": med * 1e3, "rows_per_s": R / (mean / 1e3),
           "bytes_per_step": nbytes, "hbm_gbs": nbytes / (mean / 1e3) / 1e9,
           "frac": nbytes / (mean / 1e3) / 1e9 / peak, "peak_source": src,
           "block_means_us": means_ms * 1e3,
           "block_means_frac": R * (keys + nb * wl.D_i * 4) / (means_ms / 1e3) / 1e9 / peak}
    del prob, data, g, gm
    torch.cuda.empty_cache()
    return out


def run_np_sweep(dev, stream, R, n=10):
    """Decode step time against context length: R independent V4-Flash decode queries per
    step at Np = 4K .. 256K pooled rows (16K .. 1M tokens). HiSA's work per query is
    O(nb + keep * b + k), so only the coarse stage's nb * 512 B of block means grows."""
    wl = inputs.WORKLOADS["v4flash_decode"]
    flush = L2Flush(dev)
    out = {"workload": f"v4flash_decode, R = {R} queries per step, keep = 16, k = 512", "points": []}
    for Np in (4096, 16384, 32768, 65536, 131072, 262144):
        r = decode_leg(wl.replace(B=R, Np=(Np,)), dev, stream, flush, n, 5000 + Np, f"Np={Np}")
        r["Np"] = Np
        r["bytes_per_query"] = r.pop("bytes_per_step") // R
        out["points"].append(r)
    return out


def run_r_sweep(dev, stream, n=10):
    """The decode step with more independent queries per step (4 and 6 per SM instead of 2),
    each step timed after an L2 flush: the step's per-CTA start and end costs are paid once per
    CTA, so more queries per CTA amortise them."""
    wl = inputs.WORKLOADS["v4flash_decode"]
    flush = L2Flush(dev)
    out = {"workload": "v4flash_decode, R queries per step, Np = 32768", "points": []}
    for R in (608, 912):
        r = decode_leg(wl.replace(B=R, Np=(32768,)), dev, stream, flush, n, 8000 + R, f"R={R}")
        r["R"] = R
        out["points"].append(r)
    return out


def run_ragged(dev, stream, n=20):
    """The batched ragged decode workload itself: B = 32 sequences with Np_b drawn uniformly
    from [4096, 65536] (the workload's own seed-2 draw), one step per batch of 32."""
    wl = inputs.WORKLOADS["ragged_decode"]
    r = decode_leg(wl, dev, stream, L2Flush(dev), n, wl.seed, "ragged")
    r["workload"] = "ragged_decode: B = 32, Np_b ~ U[4096, 65536] (seed 2), one batch per step"
    return r


def run_verify(dev, stream, L=4, R=304, n=10):
    """Multi-token verify on the HiSA batched path: R / L sequences of Np = 32768 pooled rows,
    L draft tokens each at t0 .. t0 + L - 1 = 4 Np - L .. 4 Np - 1 (the first rows see one
    pooled row fewer), so the step holds R query rows like the decode step."""
    wl = inputs.WORKLOADS["v4flash_decode"]
    B = R // L
    r = decode_leg(wl.replace(B=B, L=L, Np=(32768,), t0=4 * 32768 - L), dev, stream, L2Flush(dev),
                   n, 6000 + L, "verify")
    r["workload"] = f"verify: B = {B} sequences x L = {L} draft tokens, Np = 32768"
    return r


def run_compress(dev, stream, R, n=20):
    """The indexer compressor (hisa_compress_append; DeepSeek-V4 indexer shape: D_i = 128,
    r = 4, overlap, RoPE on 64 dims, bf16 cache, block means of 64 rows): (a) decode, R
    sequences appending one pooled row each, the row that completes block 511 (so each
    also writes a block mean from the 64 stored rows); (b) prefill, one sequence appending
    1024 pooled rows (4096 tokens, 16 blocks). Projected token rows drawn on the device."""
    import torch

    from deepseek_sparse_attention_hisa_gb300 import binding as hb
    flush = L2Flush(dev)
    out = {}
    for name, B, p0, nn in (("decode", R, 32767, 1), ("prefill", 1, 0, 1024)):
        D, r, C = 128, 4, 256
        cap = p0 + nn
        T = (nn + 1) * r
        g = torch.Generator(device=dev)
        g.manual_seed(7000 + B)
        kv = torch.randn((B * T, C), generator=g, device=dev)
        gate = torch.randn((B * T, C), generator=g, device=dev)
        ape = torch.randn((r, C), generator=g, device=dev)
        norm_w = 1.0 + 0.1 * torch.randn((D,), generator=g, device=dev)
        keys = torch.randn((B * cap, D), generator=g, device=dev).to(torch.bfloat16)
        tok_off = torch.arange(B + 1, device=dev, dtype=torch.int64) * T
        key_off = torch.arange(B + 1, device=dev, dtype=torch.int64) * cap
        nb = cap // 64
        means_off = torch.arange(B + 1, device=dev, dtype=torch.int64) * nb
        means = torch.zeros((B * nb, D), device=dev)
        p_first = torch.full((B,), p0, dtype=torch.int32, device=dev)
        n_new = torch.full((B,), nn, dtype=torch.int32, device=dev)
        desc = hb.CompressDesc(B=B, D_i=D, r=r, overlap=1, rope_dims=64, index_block=64,
                               n_new_max=nn, k_dtype=hb.HISA_BF16, rope_theta=160000.0,
                               eps=1e-6, tok_rows=B * T, keys_rows=B * cap, means_rows=B * nb)
        ws = hb.alloc_workspace(hb.workspace_bytes(hb.OP_COMPRESS, desc), dev)

        def call(s, desc=desc, kv=kv, gate=gate, tok_off=tok_off, p_first=p_first, n_new=n_new,
                 ape=ape, norm_w=norm_w, keys=keys, key_off=key_off, means=means,
                 means_off=means_off, ws=ws):
            hb.compress_append(desc, kv, gate, tok_off, p_first, n_new, ape, norm_w, keys,
                               key_off, means, means_off, ws, s)
        gr = capture(call, stream)
        mean, med = timed_graph(gr, stream, flush, n)
        assert hb.device_status(ws, stream) == 0
        # bytes: the token rows (kv and gate of the previous and new windows), ape and norm
        # weight, the new rows out, and per completed block its 64 rows in and its mean out
        blocks = B * ((p0 + nn) // 64 - p0 // 64)
        nbytes = (B * T * C * 4 * 2 + r * C * 4 + D * 4 + B * nn * D * 2 +
                  blocks * (64 * D * 2 + D * 4))
        peak, src = peaks()
        out[name] = {"sequences": B, "new_rows_each": nn, "us": mean * 1e3, "us_median": med * 1e3,
                     "bytes": nbytes, "hbm_gbs": nbytes / (mean / 1e3) / 1e9,
                     "frac": nbytes / (mean / 1e3) / 1e9 / peak, "peak_source": src}
        del kv, gate, keys, means, gr
        torch.cuda.empty_cache()
    return out


def run_prefill_hisa(dev, stream, n=10):
    """The HiSA batched path on the prefill workload (one sequence, L = 4096 new rows,
    Np = 16384 pooled rows, bf16 q and keys): block means once, then per step the coarse
    filter with per-row eligibility, the fine top-k with the causal re-mask and the sparse
    combine over each row's window and selected rows; each stage timed as a graph after an
    L2 flush."""
    import torch

    from deepseek_sparse_attention_hisa_gb300.problem import Problem
    wl = inputs.WORKLOADS["prefill"]
    data = inputs.generate_device(wl, device=dev, seed=4000)
    prob = Problem(data, device=dev)
    prob.block_means()
    torch.cuda.synchronize()
    flush = L2Flush(dev)
    out = {"workload": "prefill: L = 4096 rows x Np = 16384 (64 x 128 indexer, bf16 q and keys), "
                       "64 x 512 attention over 128 cached + 4096 new local rows, window 128, k = 512"}
    total = 0.0
    for name, fn in (("block_filter", lambda s: prob.block_filter(stream=s)),
                     ("select_topk", lambda s: prob.select_topk(stream=s)),
                     ("sparse_attend", lambda s: prob.attend(stream=s))):
        g = capture(fn, stream)
        ms, _ = timed_graph(g, stream, flush, n)
        out[name + "_us"] = ms * 1e3
        total += ms
    assert prob.status(stream) == 0
    out["step_us"] = total * 1e3
    out["rows_per_s"] = wl.L / (total / 1e3)
    # per-stage tensor-core work (plain multiply-add counts; masked work included) against
    # the bf16 peak: coarse L x nb x H_i x D_i, fine L x keep*b x H_i x D_i, combine
    # L x (window + k) x H x Dh for S and again for PV
    Lr, nb = wl.L, int(wl.Np[0]) // wl.index_block
    flops = {"block_filter": Lr * nb * wl.H_i * wl.D_i * 2,
             "select_topk": Lr * wl.index_keep * wl.index_block * wl.H_i * wl.D_i * 2,
             "sparse_attend": Lr * (wl.window + wl.index_topk) * wl.H * wl.Dh * 4}
    peak, src = bf16_peak()
    out["tensor_frac"] = {k: v / (out[k + "_us"] * 1e-6) / 1e12 / peak for k, v in flops.items()}
    out["tensor_peak_tflops"] = peak
    out["tensor_peak_source"] = src
    return out


def e2e_pipelined(prob, host_in, host_out, calls_for, K, dev, direct_out=False):
    """ms per step of the whole step through the public API with host buffers, copies
    overlapped with compute: two sets of device buffers; step i's inputs go in on one stream
    and step i-1's out and I come back on another while step i runs on a third. Every step's
    copies and compute lie inside the timed region, which spans all K steps (the 434 MB a
    step touches exceed L2, so no flush is inserted). With direct_out the combine writes out
    straight into page-locked host memory (one host buffer per set) and only I is copied."""
    import torch

    from deepseek_sparse_attention_hisa_gb300 import binding as hb
    sets = [prob, prob.io_clone()]
    s_in, s_c, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    host_outs = [torch.empty_like(host_out["out"]).pin_memory() for _ in sets] if direct_out else None
    graphs = []
    for b, pr in enumerate(sets):
        cl = calls_for(pr)
        if direct_out:
            dptr = hb.DevicePointer(hb.device_pointer_of_pinned(host_outs[b]), host_outs[b].numel())
            cl = dict(cl, sparse_attend=lambda s, pr=pr, dptr=dptr: pr.attend(out=dptr, stream=s,
                                                                              chained=True))

        def step(s, cl=cl):
            for name in ("block_filter_append", "select_topk", "sparse_attend"):
                cl[name](s)
        graphs.append(capture(step, s_c))
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event()
    in_done, c_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e in c_done + out_done:
        e.record(s_c)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(s_in)
    for i in range(K):
        b = i % 2
        pr = sets[b]
        s_in.wait_event(c_done[b])                   # step i-2 is done with this set
        s_in.wait_event(out_done[b])                 # and its results are back
        with torch.cuda.stream(s_in):
            pr.q_idx.copy_(host_in["q_idx"], non_blocking=True)
            pr.w.copy_(host_in["w"], non_blocking=True)
            pr.q_attn.copy_(host_in["q_attn"], non_blocking=True)
        in_done[b].record(s_in)
        s_c.wait_event(in_done[b])
        with torch.cuda.stream(s_c):
            graphs[b].replay()
        c_done[b].record(s_c)
        s_out.wait_event(c_done[b])
        with torch.cuda.stream(s_out):
            if not direct_out:
                host_out["out"].copy_(pr.out, non_blocking=True)
            host_out["I"].copy_(pr.I, non_blocking=True)
        out_done[b].record(s_out)
    s_in.wait_stream(s_out)
    t1.record(s_in)
    torch.cuda.synchronize()
    for pr in sets:
        assert pr.status() == 0, "device status flags set during the pipelined end-to-end run"
    return max_over_ranks(t0.elapsed_time(t1) / K, dev)


def run_latency(wl, dev, stream, n=50):
    """One V4-Flash decode query (B = 1): the same three calls as the throughput step, as one
    graph, L2 flushed before each replay."""
    import torch

    from deepseek_sparse_attention_hisa_gb300.problem import Problem
    data = inputs.generate_device(wl.replace(B=1), device=dev, seed=2000)
    prob = Problem(data, device=dev)
    newest = torch.as_tensor(np.array([int(prob.nb[0]) - 1], dtype=np.int32), device=dev)
    prob.block_means()
    torch.cuda.synchronize()

    def step(s):
        prob.block_filter_append(first_block=newest, stream=s)
        prob.select_topk(stream=s, chained=True)
        prob.attend(stream=s, chained=True)
    g = capture(step, stream)
    mean, med = timed_graph(g, stream, L2Flush(dev), n)
    assert prob.status(stream) == 0
    return {"workload": "v4flash_decode, one query (B = 1, Np = 32768)", "us_mean": mean * 1e3,
            "us_median": med * 1e3, "replays": n}


def run_long_context(dev, stream, n=20):
    """The long-context selection (Np = 262144, 1% of keys planted along q, selection only):
    flat top-k against HiSA at keep 16 and 64 (block means cached), each timed as a graph
    after an L2 flush; recall = |I_HiSA and I_flat| / k."""
    import torch

    from deepseek_sparse_attention_hisa_gb300.problem import Problem
    data = inputs.generate("long_context")
    flush = L2Flush(dev)
    k = data["wl"].index_topk
    flat = Problem(data, device=dev)
    I_flat = torch.full((1, k), -1, dtype=torch.int32, device=dev)
    g = capture(lambda s: flat.flat_topk(I=I_flat, stream=s), stream)
    flat_ms, _ = timed_graph(g, stream, flush, n)
    assert flat.status(stream) == 0
    ref = set(int(x) for x in I_flat.cpu().numpy().ravel() if x >= 0)
    out = {"workload": "long_context: Np = 262144 bf16 keys, f32 q, 1% planted, selection only",
           "flat_us": flat_ms * 1e3, "hisa_us": {}, "recall": {}}
    for keep in (16, 64):
        prob = Problem(data, device=dev, index_keep=keep)
        prob.block_means()
        torch.cuda.synchronize()

        def sel(s, prob=prob):
            prob.block_filter(stream=s)
            prob.select_topk(stream=s)
        g = capture(sel, stream)
        ms, _ = timed_graph(g, stream, flush, n)
        assert prob.status(stream) == 0
        got = set(int(x) for x in prob.I.cpu().numpy().ravel() if x >= 0)
        out["hisa_us"][str(keep)] = ms * 1e3
        out["recall"][str(keep)] = len(got & ref) / k
    return out


def launches_per_step(prob):
    """Kernels this library launches per step for the V4 decode shape: the coarse filter
    with the newest block means appended 1 and the fine top-k 1 (each scores and selects
    in one tcgen05 kernel), the combine 1, plus the split-K merge when it is split."""
    from deepseek_sparse_attention_hisa_gb300 import binding as hb
    ws_need = hb.workspace_bytes(hb.OP_SPARSE_ATTEND, prob.adesc)
    attend = 2 if ws_need > 256 else 1
    return 1 + 1 + attend


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--R", type=int, default=304,
                    help="independent decode queries per step (2 x 152 SMs)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-queries", type=int, default=4, help="oracle queries per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill scoring leg")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the one-query latency and long-context selection legs")
    ap.add_argument("--no-np-sweep", action="store_true",
                    help="skip the decode step time at Np = 4K .. 256K (R queries each)")
    ap.add_argument("--Np", type=int, default=32768,
                    help="pooled rows per sequence (32768 = the V4-Flash 131072-token prefix)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    wl = inputs.WORKLOADS["v4flash_decode"]
    if args.impl == "reference":
        run_reference(args, wl, args.R)
    else:
        run_gpu(args, wl, args.R)


if __name__ == "__main__":
    main()
