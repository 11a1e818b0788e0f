"""Benchmark of the packed variable-length masked-attention hot path on GB300.

One step = the whole path over one packed batch, every call through the
C ABI (libpvl.so) on one stream:
    pack_build_seq_ids -> tile_map_build -> masked_attn_fwd -> masked_attn_bwd
Workload: the 64k concatenated pack (one row of 7 episodes with latent F
drawn from U{103..362} rounded up to multiples of 8, 38 tokens per frame,
tail padded with seq_id -1 to 65,536 tokens), H = 12, D = 128, bf16.
Metric: effective TFLOP/s = 14 * D * H * (unmasked pairs) / step time, where
a pair (i, j) is unmasked iff seq_id[i] == seq_id[j] >= 0 (forward 4 D and
backward 10 D flops per pair and head).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

`--workload adaln64k` measures the fused LayerNorm-Modulate forward and
backward, `--workload loss64k` the frame_valid-masked loss with its gradient
(both HBM bound, in GB/s).

`--workload bucket_sweep` runs the same path over the 40 length-bucketed
batches of 4 (160 episodes) in one step.

`--workload cross_concat64k` (or cross_padded) measures cross attention
instead: the same episodes as queries at 38 tokens per frame and as keys at 16
tokens per frame, each side with its own seq_ids (9 launches per step: one
seq_id build per side).

Under torchrun (N > 1) every rank runs an independent replica of the step on
its own GPU (the path has no exchange step); rank 0 prints one JSON line.
`--impl reference` times the fp64 CPU oracle on this host's cores instead
(rank 0 only), on bounded samples of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective masked-attn fwd+bwd TFLOP/s and tokens/s at 1 GB300; % of bf16 peak"
FLOPS_PER_PAIR_FWD = 4
FLOPS_PER_PAIR_BWD = 10
# kernels per step: seq_ids 1, tile map 3 (both levels), forward 1, backward 3
LAUNCHES_PER_STEP = 8


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def unmasked_pairs(lay, tokens_per_frame_k=None) -> int:
    """Pairs per head: every segment's real tokens form one id (distinct ids per
    segment); for cross attention queries at the layout's tokens per frame and
    keys at tokens_per_frame_k."""
    T = lay.tokens_per_frame
    Tk = T if tokens_per_frame_k is None else tokens_per_frame_k
    return int(sum(int(v) * T * int(v) * Tk for row in lay.seg_valid for v in row))


# ------------------------------------------------------------------ clocks
class NvmlClockSampler:
    """Samples the SM clock, the power draw and the active clock-event reasons
    every 10 ms through NVML's read-only queries (libnvidia-ml.so.1 through
    ctypes), so that a timed region of a fraction of a second still gets a
    clock record.  The GPU is found by the PCI address torch reports for the
    CUDA device.  Raises OSError where NVML is not usable."""

    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    PERIOD_S = 0.01

    def __init__(self, cuda_index: int):
        import ctypes
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        props = torch.cuda.get_device_properties(cuda_index)
        bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0".encode()
        self.handle = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(self.handle)) != 0:
            raise OSError(f"no NVML device at {bus.decode()}")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.lib, self.ct = lib, ctypes
        self.samples: list[tuple[float, float, float, int]] = []
        self.stop_flag = threading.Event()
        self.thread = None

    def _one(self):
        ct, lib, h = self.ct, self.lib, self.handle
        sm, smax, mw, bits = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(sm)) != 0:      # NVML_CLOCK_SM
            return
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ct.byref(smax))
        lib.nvmlDeviceGetPowerUsage(h, ct.byref(mw))
        self.reasons_fn(h, ct.byref(bits))
        self.samples.append((float(sm.value), float(smax.value), mw.value / 1000.0, int(bits.value)))

    def _loop(self):
        while not self.stop_flag.is_set():
            self._one()
            time.sleep(self.PERIOD_S)

    def start(self):
        self._one()
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    def stop(self) -> dict:
        self.stop_flag.set()
        if self.thread:
            self.thread.join(timeout=5)
        self._one()
        sm = [x[0] for x in self.samples]
        reasons = sorted({name for x in self.samples for bit, name in self.REASON_BITS.items() if x[3] & bit})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(x[1] for x in self.samples) if sm else None,
                "reasons": reasons, "samples": len(sm),
                "power_w_max": round(max(x[2] for x in self.samples), 1) if sm else None,
                "source": "NVML every 10 ms over the timed region"}


def clock_sampler(cuda_index: int):
    """NVML sampler where NVML answers, else nvidia-smi at 200 ms."""
    try:
        return NvmlClockSampler(cuda_index)
    except (OSError, AttributeError, RuntimeError):
        return ClockSampler(cuda_index)


def choose_peak(peaks: dict, clk: dict, region_s: float):
    """The bf16 peak that applies to a timed region.  The burst figure
    (cuBLAS timed alone, at full clock) applies unless the region lasts a
    second or more, its clock record shows the power cap, and the cap held
    the median SM clock below 97 % of its maximum; then the sustained figure
    (cuBLAS back to back for seconds under the power cap, at a lower clock)
    applies.  Returns (peak, kind, why)."""
    capped = "sw_power_cap" in (clk.get("reasons") or [])
    sm, smax = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    slowed = bool(sm and smax and sm < 0.97 * smax)
    clock = f"median SM clock {sm} of {smax} MHz over {clk.get('samples')} samples"
    if region_s >= 1.0 and capped and slowed and peaks.get("bf16_tflops_sustained"):
        return peaks["bf16_tflops_sustained"], "sustained", \
            f"timed region {region_s:.2f} s under sw_power_cap, {clock}"
    if region_s < 1.0:
        why = f"timed region {region_s:.2f} s, shorter than 1 s"
    elif not capped:
        why = f"timed region {region_s:.2f} s, no sw_power_cap sample"
    else:
        why = f"timed region {region_s:.2f} s, sw_power_cap seen but the clock held"
    return peaks["bf16_tflops"], "burst", f"{why} ({clock})"


def blas_info() -> str:
    """The BLAS library numpy calls and its thread count, read from the
    running process (threadpoolctl where installed, else numpy's build
    configuration and the library's own thread query)."""
    try:
        from threadpoolctl import threadpool_info
        libs = [d for d in threadpool_info() if d.get("user_api") == "blas"]
        if libs:
            return "; ".join(f"{d.get('internal_api')} {d.get('version')} ({os.path.basename(d.get('filepath', ''))}), "
                             f"{d.get('num_threads')} threads" for d in libs)
    except ImportError:
        pass
    name = "unknown"
    try:
        cfg = np.show_config(mode="dicts")
        name = cfg["Build Dependencies"]["blas"].get("name", "unknown")
    except Exception:  # noqa: BLE001 - best effort description
        pass
    threads = None
    try:
        import ctypes
        with open("/proc/self/maps") as fh:
            paths = sorted({ln.split()[-1] for ln in fh if "openblas" in ln.lower() and ln.split()[-1].startswith("/")})
        for path in paths:
            lib = ctypes.CDLL(path)
            for sym in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_", "openblas_get_num_threads"):
                fn = getattr(lib, sym, None)
                if fn is not None:
                    threads = int(fn())
                    break
            if threads is not None:
                break
    except OSError:
        pass
    env = {k: os.environ[k] for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS") if k in os.environ}
    return f"{name}, {threads if threads is not None else 'unknown'} threads" + (f" (env {env})" if env else "")


class ClockSampler:
    """Samples nvidia-smi every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi every 200 ms"}


def pipelined_e2e(n_steps, h2d, compute, d2h):
    """Times n_steps end to end with the copies of neighbouring steps
    overlapped: step i's inputs go in on one stream while step i-1 computes,
    its results come back on a third while step i+1 computes.  Buffers are
    double-buffered (b = i % 2): h2d(b) fills input set b, compute(b) reads
    set b and writes output set b, d2h(b) reads output set b back; events
    keep a set from being reused before its previous user is done.  Returns
    milliseconds from the first copy in to the last copy out."""
    import torch
    cur = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
    in_ready = [ev(), ev()]
    done = [ev(), ev()]       # compute of the set finished (inputs free, outputs written)
    out_read = [ev(), ev()]   # results of the set copied back (outputs free)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(cur)
    s_in.wait_stream(cur)
    s_out.wait_stream(cur)
    for i in range(n_steps):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(done[b])
            h2d(b)
            in_ready[b].record(s_in)
        cur.wait_event(in_ready[b])
        if i >= 2:
            cur.wait_event(out_read[b])
        compute(b)
        done[b].record(cur)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[b])
            d2h(b)
            out_read[b].record(s_out)
    cur.wait_stream(s_out)
    cur.wait_stream(s_in)
    t1.record(cur)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1)


# -------------------------------------------------------------- GPU arm
def dist_setup(n_gpus: int):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest of the ranks' values (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, ms_per_step_max: float, world: int) -> float:
    """Whole-job throughput of weak-scaled replicas: every rank processes the
    same units per step, the job's step lasts as long as the slowest rank's."""
    return world * units_per_rank / (ms_per_step_max * 1e-3)


def traffic_record(kernel_file: str, workload: str, kernel: str | None = None):
    """DRAM bytes per launch from the committed ncu summary, if it still
    matches the source: of the file's whole call, or of one kernel of it."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh)
    src = os.path.join(ROOT, "packed_variable_length_gb300", "csrc", kernel_file)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    entry = rec.get(kernel_file)
    if not entry or entry.get("source_sha") != sha or entry.get("workload") != workload:
        return None
    if kernel is not None:
        rw = entry.get("kernels", {}).get(kernel)
        return None if rw is None else int(sum(rw))
    return entry.get("dram_bytes_per_launch")


# name -> (workload number, cross attention?)
WORKLOADS = {"concat64k": (4, False), "padded": (3, False), "same_length": (2, False),
             "cross_concat64k": (4, True), "cross_padded": (3, True)}


def describe(lay, valid_tokens: int, cl=None) -> str:
    if cl is not None:
        return (describe(lay, valid_tokens) + f"; cross attention: queries as above, keys and values the same "
                f"episodes at {cl.tokens_per_frame_k} tokens/frame (Lk = {cl.Lk}), each side with its own seq_ids")
    if lay.name == "concat64k":
        return (f"concat64k: one packed row of {lay.K} episodes (latent F = {lay.seg_frames[0].tolist()}, "
                f"{lay.tokens_per_frame} tokens/frame, {valid_tokens} valid tokens) padded with seq_id -1 to "
                f"L = {lay.L}; H = {lay.H}, D = {lay.D}")
    return (f"{lay.name}: B = {lay.B} episodes of valid F = {lay.seg_valid[:, 0].tolist()} padded to "
            f"F = {int(lay.seg_frames[0, 0])} ({lay.tokens_per_frame} tokens/frame, L = {lay.L}); "
            f"H = {lay.H}, D = {lay.D}")


def cpu_baseline(lay, tensors, budget_heads=1, cl=None):
    """The fp64 oracle as it stands on this host's cores: fwd + bwd of one head
    over every episode of the workload."""
    import oracle
    sid = oracle.build_seq_ids(lay.seg_frames, lay.seg_valid, lay.tokens_per_frame, lay.L)
    ksid, Tk = None, None
    if cl is not None:
        Tk = cl.tokens_per_frame_k
        ksid = oracle.build_seq_ids(lay.seg_frames, lay.seg_valid, Tk, cl.Lk)
    heads = list(range(budget_heads))
    t0 = time.perf_counter()
    oracle.attention_fwd(tensors["q"], tensors["k"], tensors["v"], sid, heads=heads, k_seq_id=ksid)
    oracle.attention_bwd(tensors["q"], tensors["k"], tensors["v"], tensors["do"], sid, heads=heads, k_seq_id=ksid)
    dt = time.perf_counter() - t0
    flops = (FLOPS_PER_PAIR_FWD + FLOPS_PER_PAIR_BWD) * lay.D * len(heads) * unmasked_pairs(lay, Tk)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"fp64 numpy oracle, fwd+bwd of {len(heads)} of {lay.H} heads over all {lay.B * lay.K} episodes "
                      f"({lay.B} x {lay.L} tokens), {dt:.1f} s; BLAS: {blas_info()}"}


def run_gpu(args):
    import torch
    import packed_variable_length_gb300 as pvl
    import workloads as wl

    rank, world, local = dist_setup(args.gpus)
    number, cross = WORKLOADS[args.workload]
    cl = wl.cross_config_layout(number) if cross else None
    lay = cl.q if cross else wl.config_layout(number)
    host = wl.make_cross_tensors(cl) if cross else wl.make_tensors(lay)  # bf16 CPU tensors, seeded
    dev = {k: v.cuda() for k, v in host.items()}
    B, L, H, D = lay.B, lay.L, lay.H, lay.D
    T = lay.tokens_per_frame
    Tk, Lk = (cl.tokens_per_frame_k, cl.Lk) if cross else (T, L)
    pairs = unmasked_pairs(lay, Tk)
    valid_tokens = int(lay.seg_valid.sum()) * T
    launches = LAUNCHES_PER_STEP + (1 if cross else 0)
    flops_fwd = FLOPS_PER_PAIR_FWD * D * H * pairs
    flops_bwd = FLOPS_PER_PAIR_BWD * D * H * pairs
    flops = flops_fwd + flops_bwd

    sid = torch.empty((B, L), dtype=torch.int32, device="cuda")
    ksid = torch.empty((B, Lk), dtype=torch.int32, device="cuda") if cross else None
    tm_ws = torch.empty(pvl.tile_map_ws_bytes(B, L, Lk=Lk), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(dev["q"])
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    dq = torch.empty_like(dev["q"])
    dk, dv = (torch.empty_like(dev["k"]) for _ in range(2))
    bws = torch.empty(pvl.masked_attn_bwd_ws_bytes(B, L, H, D, Lk=Lk), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step(timers=None):
        pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, T, L, out=sid)
        if cross:
            pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, Tk, Lk, out=ksid)
        tm = pvl.tile_map_build(sid, ws=tm_ws, k_seq_id=ksid)
        if timers is not None:
            timers[0].record(stream)
        pvl.masked_attn_fwd(dev["q"], dev["k"], dev["v"], sid, tm, o=o, lse=lse, k_seq_id=ksid)
        if timers is not None:
            timers[1].record(stream)
            pvl.mark_next_bwd_main(timers[3], timers[4])   # the main backward kernel alone
        pvl.masked_attn_bwd(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, sid, tm, dq=dq, dk=dk, dv=dv, ws=bws,
                            k_seq_id=ksid)
        if timers is not None:
            timers[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    pvl.device_error()

    timers = [[ev() for _ in range(5)] for _ in range(args.steps)]
    for t in timers:                # the library records [3], [4]: their CUDA events must exist
        t[3].record(stream)
        t[4].record(stream)
    torch.cuda.synchronize()
    clocks = clock_sampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start, t_end = ev(), ev()
    t_start.record(stream)
    for i in range(args.steps):
        step(timers[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    pvl.device_error()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), world)
    ms_step = ms_total / args.steps
    fwd_ms = sum(t[0].elapsed_time(t[1]) for t in timers) / args.steps
    bwd_ms = sum(t[1].elapsed_time(t[2]) for t in timers) / args.steps
    main_ms = sum(t[3].elapsed_time(t[4]) for t in timers) / args.steps

    # end to end: every step copies its inputs in from pinned host memory and
    # its results back, inside the timed region; neighbouring steps' copies
    # overlap the compute (two buffer sets, three streams)
    pin = {k: v.pin_memory() for k, v in host.items()}
    sets_in = [dev, {k: torch.empty_like(v) for k, v in dev.items()}]
    sets_out = [{"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv},
                {n: torch.empty_like(t) for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}]
    out_host = [{n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in so.items()} for so in sets_out]

    def e2e_h2d(bi):
        for k in ("q", "k", "v", "do"):
            sets_in[bi][k].copy_(pin[k], non_blocking=True)

    def e2e_compute(bi):
        di, do_ = sets_in[bi], sets_out[bi]
        pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, T, L, out=sid)
        if cross:
            pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, Tk, Lk, out=ksid)
        tm = pvl.tile_map_build(sid, ws=tm_ws, k_seq_id=ksid)
        pvl.masked_attn_fwd(di["q"], di["k"], di["v"], sid, tm, o=do_["o"], lse=do_["lse"], k_seq_id=ksid)
        pvl.masked_attn_bwd(di["q"], di["k"], di["v"], do_["o"], di["do"], do_["lse"], sid, tm, dq=do_["dq"],
                            dk=do_["dk"], dv=do_["dv"], ws=bws, k_seq_id=ksid)

    def e2e_d2h(bi):
        for n, t in sets_out[bi].items():
            out_host[bi][n].copy_(t, non_blocking=True)

    # enough steps that the pipeline's fill (the first step's copy in) and
    # drain (the last step's copy out) are a small part of the timed region
    e2e_steps = max(4, min(args.steps, 50))
    pipelined_e2e(2, e2e_h2d, e2e_compute, e2e_d2h)
    barrier(world)
    e2e_ms = max_over_ranks(pipelined_e2e(e2e_steps, e2e_h2d, e2e_compute, e2e_d2h), world) / e2e_steps
    pvl.device_error()
    h2d = sum(pin[k].numel() * pin[k].element_size() for k in ("q", "k", "v", "do"))
    d2h = sum(t.numel() * t.element_size() for t in out_host[0].values())

    # tile efficiency: unmasked pairs / pairs inside the tiles the kernels
    # compute (FULL + PARTIAL), forward on 256 x 128 tiles, backward on 128 x 128
    tmh = pvl.tile_map_build(sid, ws=tm_ws, k_seq_id=ksid)
    tile_eff = {}
    for name, level, area in (("fwd", 1, 256 * 128), ("bwd", 0, 128 * 128)):
        cls = tmh.to_host(level)["cls"]
        tile_eff[name] = round(pairs / (int((cls > 0).sum()) * area), 4)

    peaks = load_peaks()
    peak, peak_kind, peak_why = choose_peak(peaks, clk, ms_total * 1e-3)
    value = aggregate(flops, ms_step, world) / 1e12
    bwd_achieved = flops_bwd / (bwd_ms * 1e-3) / 1e12
    main_achieved = flops_bwd / (main_ms * 1e-3) / 1e12
    traffic = traffic_record("attn_bwd.cu", args.workload)
    main_traffic = traffic_record("attn_bwd.cu", args.workload, f"bwd_main_kernel<{D}>")
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": describe(lay, valid_tokens, cl),
            "B": B, "L": L, "H": H, "D": D, "tokens_per_frame": T,
            **({"Lk": Lk, "tokens_per_frame_k": Tk} if cross else {}),
            "unmasked_pairs_per_head": pairs,
            "tile_efficiency": tile_eff,
            "step": "pack_build_seq_ids + tile_map_build + masked_attn_fwd + masked_attn_bwd",
            "l2": (f"inputs larger than L2 (Q, dO {dev['q'].numel() * 2 / 1e6:.0f} MB each, K, V "
                   f"{dev['k'].numel() * 2 / 1e6:.0f} MB each); no flush"),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "tokens_per_s": round(world * valid_tokens / (ms_step * 1e-3), 1),
        "padded_tokens_per_s": round(world * B * L / (ms_step * 1e-3), 1),
        "pct_of_peak": round(100.0 * (value / world) / peak, 2),
        "peak_tflops": peak,
        "peak_kind": f"bf16 dense, {peaks['source']} {peak_kind}: {peak_why}",
        "fwd_ms": round(fwd_ms, 4),
        "bwd_ms": round(bwd_ms, 4),
        "bwd_main_ms": round(main_ms, 4),
        "fwd_tflops": round(flops_fwd / (fwd_ms * 1e-3) / 1e12, 2),
        "bwd_tflops": round(bwd_achieved, 2),
        "bwd_main_tflops": round(main_achieved, 2),
        "clocks": clk,
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "every step copies its Q, K, V, dO in from pinned host memory and O, LSE, dQ, dK, dV back; "
                        "neighbouring steps' copies overlap the compute (two buffer sets, three streams)"},
        "gpu_launches": launches * args.steps,
        "roofline": {
            "kernel": f"bwd_main_kernel<{D}> (the main backward launch alone, timed by its own CUDA events "
                      "on the launching stream)",
            "bound": "tensor", "achieved": round(main_achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(main_achieved / peak, 4), "traffic": main_traffic,
            "peak_note": f"of {peaks['source']} (bf16 cuBLAS, {peak_kind})",
            "algorithmic": "10 * D * H * unmasked pairs per launch",
        },
        "roofline_bwd_call": {
            "kernel": "masked_attn_bwd (bwd_pre + bwd_main + bwd_convert launches, timed together)",
            "bound": "tensor", "achieved": round(bwd_achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(bwd_achieved / peak, 4), "traffic": traffic,
            "peak_note": f"of {peaks['source']} (bf16 cuBLAS, {peak_kind})",
            "algorithmic": "10 * D * H * unmasked pairs per call",
        },
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(lay, host, cl=cl)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------ bucket sweep workload
def run_bucket_sweep(args):
    """Workload 5: the 40 batches of 4 that the length-bucketing sampler cuts
    from 160 episode lengths (F ~ U{103..362}, padded to multiples of 8, 38
    tokens per frame, L = 38 F_pad per batch).  One step is the whole path
    (seq_ids, tile map, forward, backward) over all 40 batches, in the
    sampler's order; the metric is the headline's, over the sweep's unmasked
    pairs.  Inputs: one seeded draw at the largest batch's size, each batch
    reading its [4, L, H, D] prefix (values do not change the work)."""
    import torch
    import packed_variable_length_gb300 as pvl
    import workloads as wl

    rank, world, local = dist_setup(args.gpus)
    layouts, batches, lengths = wl.bucket_sweep_layouts()
    big = max(layouts, key=lambda la: la.B * la.L)
    H, D, T = big.H, big.D, big.tokens_per_frame
    host = wl.make_tensors(big)                               # bf16 CPU tensors, seeded
    dev = {k: v.cuda().view(-1) for k, v in host.items()}
    n_max = big.B * big.L * H * D
    outs = {n: torch.empty(n_max, dtype=torch.bfloat16, device="cuda") for n in ("o", "dq", "dk", "dv")}
    lse_pool = torch.empty(big.B * H * big.L, dtype=torch.float32, device="cuda")
    sid_pool = torch.empty(big.B * big.L, dtype=torch.int32, device="cuda")
    tm_pool = torch.empty(max(pvl.tile_map_ws_bytes(la.B, la.L) for la in layouts), dtype=torch.uint8, device="cuda")
    bws_pool = torch.empty(max(pvl.masked_attn_bwd_ws_bytes(la.B, la.L, H, D) for la in layouts),
                           dtype=torch.uint8, device="cuda")
    pairs = [unmasked_pairs(la) for la in layouts]
    flops_fwd = FLOPS_PER_PAIR_FWD * D * H * sum(pairs)
    flops_bwd = FLOPS_PER_PAIR_BWD * D * H * sum(pairs)
    flops = flops_fwd + flops_bwd
    valid_tokens = sum(int(la.seg_valid.sum()) * T for la in layouts)
    padded_tokens = sum(la.B * la.L for la in layouts)
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def views(la, ins, outs_):
        shp = (la.B, la.L, H, D)
        n = la.B * la.L * H * D
        i = {k: ins[k][:n].view(shp) for k in ("q", "k", "v", "do")}
        o = {k: outs_[k][:n].view(shp) for k in ("o", "dq", "dk", "dv")}
        o["lse"] = outs_["lse"][: la.B * H * la.L].view(la.B, H, la.L)
        return i, o

    def batch_step(la, ins, outs_, timers=None):
        i, o = views(la, ins, outs_)
        sid = sid_pool[: la.B * la.L].view(la.B, la.L)
        pvl.pack_build_seq_ids(la.seg_frames, la.seg_valid, T, la.L, out=sid)
        tm = pvl.tile_map_build(sid, ws=tm_pool[: pvl.tile_map_ws_bytes(la.B, la.L)])
        if timers is not None:
            timers[0].record(stream)
        pvl.masked_attn_fwd(i["q"], i["k"], i["v"], sid, tm, o=o["o"], lse=o["lse"])
        if timers is not None:
            timers[1].record(stream)
        pvl.masked_attn_bwd(i["q"], i["k"], i["v"], o["o"], i["do"], o["lse"], sid, tm, dq=o["dq"], dk=o["dk"],
                            dv=o["dv"], ws=bws_pool[: pvl.masked_attn_bwd_ws_bytes(la.B, la.L, H, D)])
        if timers is not None:
            timers[2].record(stream)

    dev_out = {**outs, "lse": lse_pool}

    def step(timers=None):
        for bi, la in enumerate(layouts):
            batch_step(la, dev, dev_out, None if timers is None else timers[bi])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    pvl.device_error()
    n_steps = max(1, min(args.steps, 10))     # one step is ~0.3 s of GPU work
    timers = [[[ev(), ev(), ev()] for _ in layouts] for _ in range(n_steps)]
    clocks = clock_sampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start, t_end = ev(), ev()
    t_start.record(stream)
    for i in range(n_steps):
        step(timers[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    pvl.device_error()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), world)
    ms_step = ms_total / n_steps
    fwd_ms = sum(t[0].elapsed_time(t[1]) for st in timers for t in st) / n_steps
    bwd_ms = sum(t[1].elapsed_time(t[2]) for st in timers for t in st) / n_steps

    # end to end: each batch's inputs copied in from pinned host memory and its
    # results copied back, neighbouring batches' copies overlapping the compute
    pin = {k: v.view(-1).pin_memory() for k, v in host.items()}
    sets_in = [dev, {k: torch.empty_like(v) for k, v in dev.items()}]
    sets_out = [dev_out, {k: torch.empty_like(v) for k, v in dev_out.items()}]
    out_host = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in so.items()} for so in sets_out]
    cursor = {"h2d": 0, "compute": 0, "d2h": 0}

    def nxt(kind):
        la = layouts[cursor[kind] % len(layouts)]
        cursor[kind] += 1
        return la

    def e2e_h2d(b):
        la = nxt("h2d")
        n = la.B * la.L * H * D
        for k in ("q", "k", "v", "do"):
            sets_in[b][k][:n].copy_(pin[k][:n], non_blocking=True)

    def e2e_compute(b):
        batch_step(nxt("compute"), sets_in[b], sets_out[b])

    def e2e_d2h(b):
        la = nxt("d2h")
        n = la.B * la.L * H * D
        for k in ("o", "dq", "dk", "dv"):
            out_host[b][k][:n].copy_(sets_out[b][k][:n], non_blocking=True)
        m = la.B * H * la.L
        out_host[b]["lse"][:m].copy_(sets_out[b]["lse"][:m], non_blocking=True)

    pipelined_e2e(2, e2e_h2d, e2e_compute, e2e_d2h)
    for kind in cursor:
        cursor[kind] = 0
    barrier(world)
    e2e_passes = 2
    e2e_ms = max_over_ranks(pipelined_e2e(e2e_passes * len(layouts), e2e_h2d, e2e_compute, e2e_d2h), world) / e2e_passes
    pvl.device_error()
    h2d = sum(8 * la.B * la.L * H * D for la in layouts)
    d2h = sum(8 * la.B * la.L * H * D + 4 * la.B * H * la.L for la in layouts)

    # tile efficiency over the sweep: unmasked pairs / pairs inside computed tiles
    tiles = {"fwd": 0, "bwd": 0}
    for la in layouts:
        sid = pvl.pack_build_seq_ids(la.seg_frames, la.seg_valid, T, la.L)
        tmh = pvl.tile_map_build(sid)
        for name, level, area in (("fwd", 1, 256 * 128), ("bwd", 0, 128 * 128)):
            tiles[name] += int((tmh.to_host(level)["cls"] > 0).sum()) * area
    tile_eff = {k: round(sum(pairs) / v, 4) for k, v in tiles.items()}
    f_valid = sum(int(la.seg_valid.sum()) for la in layouts)
    f_padded = sum(la.B * int(la.seg_frames[0, 0]) for la in layouts)

    peaks = load_peaks()
    peak, peak_kind, peak_why = choose_peak(peaks, clk, ms_total * 1e-3)
    value = aggregate(flops, ms_step, world) / 1e12
    bwd_achieved = flops_bwd / (bwd_ms * 1e-3) / 1e12
    n_launch = LAUNCHES_PER_STEP * len(layouts)
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": n_steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": (f"bucket_sweep: {len(layouts)} batches of 4 from the length-bucketing sampler over "
                         f"{len(lengths)} episodes (F ~ U{{103..362}}, padded to multiples of 8, {T} tokens/frame), "
                         f"L = {T} x F_pad per batch ({min(la.L for la in layouts)}..{max(la.L for la in layouts)}); "
                         f"H = {H}, D = {D}; one step = all {len(layouts)} batches"),
            "H": H, "D": D, "tokens_per_frame": T, "batches": len(layouts),
            "distinct_shapes": len({la.L for la in layouts}),
            "waste_pct": round(100.0 * (1 - f_valid / f_padded), 2),
            "unmasked_pairs_per_head": sum(pairs), "tile_efficiency": tile_eff,
            "step": "per batch: pack_build_seq_ids + tile_map_build + masked_attn_fwd + masked_attn_bwd",
            "inputs": "one seeded draw at the largest batch's size; each batch reads its prefix",
            "l2": "every batch's fwd + bwd touches more than L2 (Q, K, V, dO >= 52 MB each, fp32 dQ accumulator); "
                  "no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "tokens_per_s": round(world * valid_tokens / (ms_step * 1e-3), 1),
        "padded_tokens_per_s": round(world * padded_tokens / (ms_step * 1e-3), 1),
        "pct_of_peak": round(100.0 * (value / world) / peak, 2), "peak_tflops": peak,
        "peak_kind": f"bf16 dense, {peaks['source']} {peak_kind}: {peak_why}",
        "fwd_ms": round(fwd_ms, 4), "bwd_ms": round(bwd_ms, 4),
        "fwd_tflops": round(flops_fwd / (fwd_ms * 1e-3) / 1e12, 2), "bwd_tflops": round(bwd_achieved, 2),
        "clocks": clk,
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "passes": e2e_passes, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "every batch copies its Q, K, V, dO in from pinned host memory and O, LSE, dQ, dK, dV back; "
                        "neighbouring batches' copies overlap the compute (two buffer sets, three streams)"},
        "gpu_launches": n_launch * n_steps,
        "roofline": {
            "kernel": "masked_attn_bwd (bwd_pre + bwd_main + bwd_convert launches, timed together), summed over "
                      "the 40 batches",
            "bound": "tensor", "achieved": round(bwd_achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(bwd_achieved / peak, 4), "traffic": None,
            "peak_note": f"of {peaks['source']} (bf16 cuBLAS, {peak_kind})",
            "algorithmic": "10 * D * H * unmasked pairs per launch",
        },
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        small = min(layouts, key=lambda la: la.B * la.L)
        result["cpu_baseline"] = cpu_baseline(small, wl.make_tensors(small), budget_heads=4)
        result["cpu_baseline"]["sample"] += f" (batch {small.name}, the sweep's smallest)"
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------ AdaLN workload
ADALN_SHAPE = (1, 64000, 5120)  # B, N (the page's 64k sequence), D (a 14B-class DiT width)


def run_adaln(args):
    """Fused LayerNorm-Modulate forward + backward ("AdaptiveLoad" §2.B) at
    B = 1, N = 64,000, D = 5120; HBM bound, so the metric is algorithmic
    bytes per second: forward reads x and writes y (4 N D bytes plus the
    modulation vectors), backward reads x and dy and writes dx (6 N D bytes
    plus the modulation vectors and their gradients)."""
    import torch
    import packed_variable_length_gb300 as pvl

    rank, world, local = dist_setup(args.gpus)
    B, N, D = ADALN_SHAPE
    g = torch.Generator().manual_seed(2605)
    host = {"x": (torch.randn(B, N, D, generator=g) * 2).to(torch.bfloat16),
            "dy": torch.randn(B, N, D, generator=g).to(torch.bfloat16),
            "shift": torch.randn(B, D, generator=g), "scale": torch.randn(B, D, generator=g) * 0.3}
    dev = {k: v.cuda() for k, v in host.items()}
    y = torch.empty_like(dev["x"])
    dx = torch.empty_like(dev["x"])
    dshift = torch.empty(B, D, device="cuda")
    dscale = torch.empty(B, D, device="cuda")
    ws = torch.empty(pvl.adaln_bwd_ws_bytes(B, N, D), dtype=torch.uint8, device="cuda")
    bytes_fwd = 4 * N * D * B + 8 * B * D
    bytes_bwd = 6 * N * D * B + 12 * B * D
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step(timers=None):
        if timers is not None:
            timers[0].record(stream)
        pvl.adaln_fwd(dev["x"], dev["shift"], dev["scale"], 1e-6, y=y)
        if timers is not None:
            timers[1].record(stream)
        pvl.adaln_bwd(dev["x"], dev["scale"], dev["dy"], 1e-6, dx=dx, dshift=dshift, dscale=dscale, ws=ws)
        if timers is not None:
            timers[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    pvl.device_error()
    timers = [[ev(), ev(), ev()] for _ in range(args.steps)]
    clocks = clock_sampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = ev(), ev()
    t0.record(stream)
    for i in range(args.steps):
        step(timers[i])
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    pvl.device_error()
    ms_step = max_over_ranks(t0.elapsed_time(t1), world) / args.steps
    fwd_ms = sum(t[0].elapsed_time(t[1]) for t in timers) / args.steps
    bwd_ms = sum(t[1].elapsed_time(t[2]) for t in timers) / args.steps

    pin = {k: v.pin_memory() for k, v in host.items()}
    sets_in = [dev, {k: torch.empty_like(v) for k, v in dev.items()}]
    sets_out = [{"y": y, "dx": dx, "dshift": dshift, "dscale": dscale},
                {n: torch.empty_like(t) for n, t in (("y", y), ("dx", dx), ("dshift", dshift), ("dscale", dscale))}]
    out_host = [{n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in so.items()} for so in sets_out]

    def e2e_h2d(bi):
        for k in host:
            sets_in[bi][k].copy_(pin[k], non_blocking=True)

    def e2e_compute(bi):
        di, do_ = sets_in[bi], sets_out[bi]
        pvl.adaln_fwd(di["x"], di["shift"], di["scale"], 1e-6, y=do_["y"])
        pvl.adaln_bwd(di["x"], di["scale"], di["dy"], 1e-6, dx=do_["dx"], dshift=do_["dshift"],
                      dscale=do_["dscale"], ws=ws)

    def e2e_d2h(bi):
        for n, t in sets_out[bi].items():
            out_host[bi][n].copy_(t, non_blocking=True)

    e2e_steps = max(4, min(args.steps, 10))
    pipelined_e2e(2, e2e_h2d, e2e_compute, e2e_d2h)
    barrier(world)
    e2e_ms = pipelined_e2e(e2e_steps, e2e_h2d, e2e_compute, e2e_d2h)
    pvl.device_error()
    e2e_ms = max_over_ranks(e2e_ms, world) / e2e_steps
    peaks = load_peaks()
    hbm = peaks["hbm_gbs"]
    value = aggregate(bytes_fwd + bytes_bwd, ms_step, world) / 1e9
    bwd_gbs = bytes_bwd / (bwd_ms * 1e-3) / 1e9
    result = {
        "metric": "fused LayerNorm-Modulate fwd+bwd algorithmic GB/s and tokens/s at 1 GB300",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in/out, fp32 arithmetic", "data": "synthetic",
        "config": {"workload": f"adaln64k: B = {B}, N = {N}, D = {D}, x ~ N(0, 4), scale ~ N(0, 0.09), shift ~ N(0, 1)",
                   "B": B, "N": N, "D": D, "l2": "x, y, dy, dx are 655 MB each (larger than L2); no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "tokens_per_s": round(world * B * N / (ms_step * 1e-3), 1),
        "fwd_ms": round(fwd_ms, 4), "bwd_ms": round(bwd_ms, 4),
        "fwd_gbs": round(bytes_fwd / (fwd_ms * 1e-3) / 1e9, 1), "bwd_gbs": round(bwd_gbs, 1),
        "clocks": clk,
        "e2e": {"value": round(world * (bytes_fwd + bytes_bwd) / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in pin.values()),
                "d2h_bytes_per_step": sum(v.numel() * v.element_size() for v in out_host[0].values()),
                "note": "every step copies x, dy, shift, scale in and y, dx, dshift, dscale back; neighbouring "
                        "steps' copies overlap the compute (two buffer sets, three streams)"},
        "gpu_launches": 3 * args.steps,
        "roofline": {"kernel": "adaln_bwd (row kernel + tile-sum kernel, timed together)", "bound": "hbm",
                     "achieved": round(bwd_gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(bwd_gbs / hbm, 4),
                     "traffic": traffic_record("adaln.cu", "adaln64k"),
                     "peak_note": f"of {peaks['source']} (STREAM-style copy)",
                     "algorithmic": "6 N D + 12 B D bytes per launch"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        n = 2000
        t = time.perf_counter()
        oracle.adaln_fwd(host["x"][:, :n], host["shift"], host["scale"])
        oracle.adaln_bwd(host["x"][:, :n], host["shift"], host["scale"], host["dy"][:, :n])
        dt = time.perf_counter() - t
        result["cpu_baseline"] = {"value": round((10 * n * D * B) / dt / 1e9, 3), "unit": "GB/s",
                                  "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                                  "sample": f"fp64 numpy oracle, fwd+bwd of the first {n} of {N} tokens, {dt:.1f} s"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


LOSS_GRID = 128     # latent positions per frame (8 x 16)
LOSS_C = 48         # latent channels


def run_loss(args):
    """The frame_valid-masked squared-error loss with its gradient in the same
    pass ("lingbot_va_packing" §2.1, compute_loss) on the 64k pack's episodes
    at the latent's own grid: 8 x 16 positions and 48 channels per frame
    (the latent shape (48, F, 8, 16) of the attention profiling report), over
    the pack's frame capacity (65,536 // 38 frames).  HBM bound: the metric is
    algorithmic bytes per second (pred and target read on valid positions,
    the gradient written everywhere, the ids read once).  The tensors are
    about 21 MB each, inside L2, so L2 is flushed before every timed call."""
    import torch
    import packed_variable_length_gb300 as pvl
    import workloads as wl

    rank, world, local = dist_setup(args.gpus)
    lay = wl.config_layout(4)
    frames = lay.L // lay.tokens_per_frame
    B, L, C = lay.B, frames * LOSS_GRID, LOSS_C
    host = wl.make_loss_tensors(B, L, C, 2606)
    dev = {k: v.cuda() for k, v in host.items()}
    sid = pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, LOSS_GRID, L)
    n_valid = int((sid >= 0).sum().item())
    grad = torch.empty_like(dev["pred"])
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(pvl.masked_mse_ws_bytes(B, L, C), dtype=torch.uint8, device="cuda")
    flush = torch.ones(64 << 20, dtype=torch.float32, device="cuda")    # 256 MB > L2
    sink = torch.empty((), dtype=torch.float32, device="cuda")
    bytes_step = 4 * n_valid * C + 2 * B * L * C + 4 * B * L + 4
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step():
        pvl.masked_mse_loss(dev["pred"], dev["target"], sid, grad=grad, loss=loss, ws=ws)

    # L2 is flushed by reading the buffer (clean lines): a written flush would
    # leave 129 MB of dirty lines whose write-back lands inside the next call
    for _ in range(args.warmup):
        torch.sum(flush, dim=0, out=sink)
        step()
    torch.cuda.synchronize()
    pvl.device_error()
    pairs = [(ev(), ev()) for _ in range(args.steps)]
    clocks = clock_sampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    for a, b in pairs:
        torch.sum(flush, dim=0, out=sink)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    pvl.device_error()
    ms_step = max_over_ranks(sum(a.elapsed_time(b) for a, b in pairs), world) / args.steps
    value = aggregate(bytes_step, ms_step, world) / 1e9

    pin = {k: v.pin_memory() for k, v in host.items()}
    sets_in = [dev, {k: torch.empty_like(v) for k, v in dev.items()}]
    sets_out = [(grad, loss, ws, sid), (torch.empty_like(grad), torch.empty_like(loss), torch.empty_like(ws),
                                        torch.empty_like(sid))]
    loss_host = [torch.empty(1, dtype=torch.float32, pin_memory=True) for _ in range(2)]

    def e2e_h2d(bi):
        for k in host:
            sets_in[bi][k].copy_(pin[k], non_blocking=True)

    def e2e_compute(bi):
        g_, l_, w_, s_ = sets_out[bi]
        pvl.pack_build_seq_ids(lay.seg_frames, lay.seg_valid, LOSS_GRID, L, out=s_)
        pvl.masked_mse_loss(sets_in[bi]["pred"], sets_in[bi]["target"], s_, grad=g_, loss=l_, ws=w_)

    def e2e_d2h(bi):
        loss_host[bi].copy_(sets_out[bi][1], non_blocking=True)

    e2e_steps = max(4, min(args.steps, 20))
    pipelined_e2e(2, e2e_h2d, e2e_compute, e2e_d2h)
    e2e_ms = pipelined_e2e(e2e_steps, e2e_h2d, e2e_compute, e2e_d2h)
    pvl.device_error()
    e2e_ms = max_over_ranks(e2e_ms, world) / e2e_steps
    peaks = load_peaks()
    hbm = peaks["hbm_gbs"]
    result = {
        "metric": "frame_valid-masked loss + gradient algorithmic GB/s at 1 GB300",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in/out, fp32 arithmetic, cross-CTA sum in fp32 pairs", "data": "synthetic",
        "config": {"workload": (f"loss64k: the 64k pack's {lay.K} episodes (latent F = {lay.seg_frames[0].tolist()}) "
                                f"on the latent grid, {LOSS_GRID} positions x {C} channels per frame, "
                                f"{frames} frames of capacity (L = {L}, {n_valid} valid positions)"),
                   "B": B, "L": L, "C": C, "valid_positions": n_valid,
                   "l2": "pred, target, grad are 21 MB each (inside L2): a 256 MB buffer is read before every "
                         "timed call, outside its events (a read leaves clean lines, so no write-back lands in the call)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "clocks": clk,
        "e2e": {"value": round(world * bytes_step / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in pin.values()),
                "d2h_bytes_per_step": 4,
                "note": "per step: pred and target copied in, seq_ids built from the host segment table, the "
                        "loss call, the loss read back; neighbouring steps' copies overlap the compute (two buffer "
                        "sets, three streams)"},
        "gpu_launches": args.steps,
        "roofline": {"kernel": "masked_mse_loss (the 64-byte workspace clear and the loss kernel, timed together)",
                     "bound": "hbm",
                     "achieved": round(bytes_step / (ms_step * 1e-3) / 1e9, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(bytes_step / (ms_step * 1e-3) / 1e9 / hbm, 4),
                     "traffic": traffic_record("masked_loss.cu", "loss64k"),
                     "peak_note": f"of {peaks['source']} (STREAM-style copy)",
                     "algorithmic": "4 C per valid position + 2 C per position + 4 per id, bytes per call"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        valid = oracle.valid_from_seq_id(oracle.build_seq_ids(lay.seg_frames, lay.seg_valid, LOSS_GRID, L))
        t = time.perf_counter()
        reps = 0
        while reps < 3 or time.perf_counter() - t < 5.0:
            oracle.masked_mse(host["pred"], host["target"], valid)
            oracle.masked_mse_grad(host["pred"], host["target"], valid)
            reps += 1
        dt = (time.perf_counter() - t) / reps
        result["cpu_baseline"] = {"value": round(bytes_step / dt / 1e9, 3), "unit": "GB/s",
                                  "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                                  "sample": f"fp64 numpy oracle, loss and gradient of the whole workload, "
                                            f"{reps} repetitions, {dt:.2f} s each"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


ADAPTIVE_M_MEM = 65536        # token budget per GPU batch (the 64k pack)
ADAPTIVE_HIDDEN = 1536        # H * D: the AdaLN width of the timed layer step
ADAPTIVE_RANKS = 8            # simulated synchronous data-parallel ranks
ADAPTIVE_EPISODES = 1000      # episode pool: enough that the 33 padded shapes fill their batches


def run_adaptive(args):
    """AdaptiveLoad's dual-constraint bucketing ("AdaptiveLoad" §2.A, §4) on
    the library's own kernels.  The timed unit ("layer step") for a batch of B
    episodes padded to F_pad frames (S = 38 F_pad tokens each) is masked
    attention forward + backward (H = 12, D = 128) plus AdaLN forward +
    backward at width 1536 over the batch's tokens, 11 launches.
      1. Shape benchmarking: the layer step is timed over a (B, F_pad) grid
         and step_time ~ a + b B S^p is fitted; M_comp = the fitted load of a
         memory-bound batch at the shortest bucket (S = 38 * 104).
      2. 1000 episode lengths drawn like workload 5's (F ~ U{103..362}; with
         33 padded shapes, 160 would leave most buckets short of one
         memory-bound batch) are batched three ways:
         equal-token (B = floor(M_mem / S)), dual-constraint (B_shape), and
         the fixed batch of 4 of the packing report's sampler.
      3. Every batch's layer step is timed; reported per arm, under the
         page's names ("AdaptiveLoad" §4, load-balance results): the
         compute imbalance rate, the coefficient of variation of the batches'
         compute load (here the fitted cost model's load B S^p), and the
         synchronisation overhead, the coefficient of variation of the step
         time (here the measured batch step times); plus the valid tokens/s
         of 8 simulated synchronous data-parallel ranks taking the batches
         round-robin (each step as long as its slowest)."""
    import torch
    import packed_variable_length_gb300 as pvl
    from packed_variable_length_gb300 import adaptive_load as al
    import workloads as wl

    rank, world, local = dist_setup(args.gpus)
    H, D, T = 12, 128, wl.TOKENS_PER_FRAME
    C = ADAPTIVE_HIDDEN
    n_max = ADAPTIVE_M_MEM
    g = torch.Generator().manual_seed(2607)
    flat = {k: (torch.randn(n_max * C, generator=g)).to(torch.bfloat16).cuda() for k in ("q", "k", "v", "do")}
    outs = {k: torch.empty(n_max * C, dtype=torch.bfloat16, device="cuda") for k in ("o", "dq", "dk", "dv", "y", "dx")}
    shift = torch.randn(64, C, generator=g).cuda()
    scale = (torch.randn(64, C, generator=g) * 0.3).cuda()
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def layer_step(frames, f_pad):
        """Returns a callable running the layer step for one pad-collated batch."""
        B = len(frames)
        L = T * f_pad
        v = lambda t: t[: B * L * C].view(B, L, H, D)  # noqa: E731
        q, k, vv, do = v(flat["q"]), v(flat["k"]), v(flat["v"]), v(flat["do"])
        o, dq, dk, dv = v(outs["o"]), v(outs["dq"]), v(outs["dk"]), v(outs["dv"])
        x, dy = q.view(B, L, C), do.view(B, L, C)
        y, dx = outs["y"][: B * L * C].view(B, L, C), outs["dx"][: B * L * C].view(B, L, C)
        sid = torch.empty((B, L), dtype=torch.int32, device="cuda")
        tm_ws = torch.empty(pvl.tile_map_ws_bytes(B, L), dtype=torch.uint8, device="cuda")
        lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
        bws = torch.empty(pvl.masked_attn_bwd_ws_bytes(B, L, H, D), dtype=torch.uint8, device="cuda")
        aws = torch.empty(pvl.adaln_bwd_ws_bytes(B, L, C), dtype=torch.uint8, device="cuda")
        dshift = torch.empty((B, C), dtype=torch.float32, device="cuda")
        dscale = torch.empty((B, C), dtype=torch.float32, device="cuda")
        seg_f = np.full((B, 1), f_pad, np.int32)
        seg_v = np.asarray(frames, np.int32).reshape(B, 1)

        def run():
            pvl.pack_build_seq_ids(seg_f, seg_v, T, L, out=sid)
            tm = pvl.tile_map_build(sid, ws=tm_ws)
            pvl.masked_attn_fwd(q, k, vv, sid, tm, o=o, lse=lse)
            pvl.masked_attn_bwd(q, k, vv, o, do, lse, sid, tm, dq=dq, dk=dk, dv=dv, ws=bws)
            pvl.adaln_fwd(x, shift[:B], scale[:B], 1e-6, y=y)
            pvl.adaln_bwd(x, scale[:B], dy, 1e-6, dx=dx, dshift=dshift, dscale=dscale, ws=aws)
        return run

    def time_step(run, reps):
        run()
        pairs = [(ev(), ev()) for _ in range(reps)]
        for a, b in pairs:
            a.record(stream)
            run()
            b.record(stream)
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) for a, b in pairs])) * 1e-3

    clocks = clock_sampler(local)
    clocks.start()
    # 1. shape benchmarking and the cost-model fit
    shapes = [(Bn, fp) for fp in (104, 168, 232, 296, 360) for Bn in (1, 2, 4, 8, 16) if Bn * T * fp <= n_max]
    samp = []
    for Bn, fp in shapes:
        samp.append((Bn, T * fp, time_step(layer_step([fp] * Bn, fp), max(3, args.steps // 10))))
    Bs, Ss, ts = (np.array(c, dtype=np.float64) for c in zip(*samp))
    model = al.fit_cost_model(Bs, Ss, ts)
    s_min = T * 104
    m_comp = al.m_comp_for(n_max, s_min, model.p)
    # 2. three ways to batch the same 160 episodes
    lengths = wl.bucket_sweep_lengths(1005, ADAPTIVE_EPISODES)
    arms = {
        "equal_token": al.DualConstraintBatchSampler(lengths, T, n_max, math.inf, model.p, seed=1005).all_batches(),
        "dual_constraint": al.DualConstraintBatchSampler(lengths, T, n_max, m_comp, model.p, seed=1005).all_batches(),
        "fixed_batch_4": wl.bucket_sweep_layouts(1005, ADAPTIVE_EPISODES, 4)[1],
    }
    # 3. every batch's layer step
    results = {}
    n_launch = 0
    for name, batches in arms.items():
        times, tokens, loads = [], [], []
        for bt in batches:
            frames = [int(lengths[i]) for i in bt]
            fp = int(al.padded_frames(max(frames), 8))
            times.append(time_step(layer_step(frames, fp), 3))
            tokens.append(T * sum(frames))
            loads.append(len(bt) * (T * fp) ** model.p)
            n_launch += (LAUNCHES_PER_STEP + 3) * 4  # the attention step plus AdaLN forward (1) and backward (2)
        tps, step_t, idle = al.simulate_data_parallel(times, tokens, ADAPTIVE_RANKS)
        results[name] = {"batches": len(batches),
                         "compute_imbalance_rate_cv_modelled_load": round(al.coefficient_of_variation(loads), 4),
                         "sync_overhead_cv_step_time": round(al.coefficient_of_variation(times), 4),
                         "sim_dp8_tokens_per_s": round(tps, 1), "sim_dp8_idle_fraction": round(idle, 4),
                         "sim_dp8_cv_step": round(al.coefficient_of_variation(step_t), 4),
                         "batch_sizes": sorted(set(len(b) for b in batches)),
                         "total_step_time_s": round(float(sum(times)), 4)}
    clk = clocks.stop()
    pvl.device_error()
    dual, base = results["dual_constraint"], results["equal_token"]
    value = world * dual["sim_dp8_tokens_per_s"]
    result = {
        "metric": "valid tokens/s of 8 simulated synchronous data-parallel ranks under dual-constraint bucketing "
                  "(layer step: masked attention fwd+bwd + AdaLN fwd+bwd, timed per batch on 1 GB300)",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": len(arms["dual_constraint"]),
        "warmup": 1, "ms_per_step": round(1e3 * dual["total_step_time_s"] / len(arms["dual_constraint"]), 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": (f"adaptive_load: {ADAPTIVE_EPISODES} episode lengths drawn like workload 5's (F ~ U{{103..362}}, padded to "
                                f"multiples of 8, 38 tokens/frame), M_mem = {n_max} tokens, H = {H}, D = {D}, "
                                f"AdaLN width {C}; each batch's layer step timed (median of 3) after one warm-up"),
                   "l2": "batches up to 65,536 tokens x 1536 (201 MB per tensor, larger than L2); no flush",
                   "cost_model": {"a_s": model.a, "b": model.b, "p": round(model.p, 5), "r2": round(model.r2, 6),
                                  "shapes": len(shapes)},
                   "m_comp": m_comp, "s_ref": s_min, "arms": results,
                   "dual_vs_equal_token_throughput": round(dual["sim_dp8_tokens_per_s"] / base["sim_dp8_tokens_per_s"], 4),
                   "page_measures": {
                       "compute imbalance rate (CV of compute load)": {
                           "here_equal_token_to_dual": [base["compute_imbalance_rate_cv_modelled_load"],
                                                        dual["compute_imbalance_rate_cv_modelled_load"]],
                           "page": "39% -> 18.9% (its corpus and cluster)"},
                       "synchronisation overhead (CV of step time)": {
                           "here_equal_token_to_dual": [base["sync_overhead_cv_step_time"],
                                                        dual["sync_overhead_cv_step_time"]],
                           "page": "18.7% -> 10.4% (16 GPUs)"}},
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "clocks": clk,
        "gpu_launches": n_launch,
    }
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ----------------------------------------------------------- reference arm
def run_reference(args):
    """The fp64 oracle on the host cores, one bounded sample per step: fwd + bwd
    of one block of at most 2048 queries of one (episode, head) of the same
    workload against all of that episode's keys (the oracle's separate
    query / key id form), the blocks taken in a seeded order over every
    episode and head, so that any --steps K ends within minutes."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    import workloads as wl
    lay = wl.config_layout(4)
    host = wl.make_tensors(lay)
    T = lay.tokens_per_frame
    starts = np.concatenate([[0], np.cumsum(lay.seg_frames[0]) * T])
    block = 2048
    samples = []
    for h in range(lay.H):
        for e in range(lay.K):
            lo, hi = int(starts[e]), int(starts[e] + lay.seg_valid[0, e] * T)
            samples += [(e, h, a, min(a + block, hi), lo, hi) for a in range(lo, hi, block)]
    order = np.random.default_rng(0).permutation(len(samples))
    done_flops = 0.0
    done_time = 0.0
    for it in range(args.warmup + args.steps):
        e, h, a, b, lo, hi = samples[order[it % len(samples)]]
        q, do = host["q"][:, a:b], host["do"][:, a:b]
        k, v = host["k"][:, lo:hi], host["v"][:, lo:hi]
        sid_q = np.zeros((1, b - a), np.int32)
        sid_k = np.zeros((1, hi - lo), np.int32)
        t0 = time.perf_counter()
        oracle.attention_fwd(q, k, v, sid_q, heads=[h], k_seq_id=sid_k)
        oracle.attention_bwd(q, k, v, do, sid_q, heads=[h], k_seq_id=sid_k)
        dt = time.perf_counter() - t0
        if it >= args.warmup:
            done_flops += (FLOPS_PER_PAIR_FWD + FLOPS_PER_PAIR_BWD) * lay.D * (b - a) * (hi - lo)
            done_time += dt
    value = done_flops / done_time / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = (f"fp64 numpy oracle: each step is fwd+bwd of one block of <= {block} queries of one (episode, head) "
              f"of the concat64k workload against all of that episode's keys ({len(samples)} blocks over {lay.K} "
              f"episodes x {lay.H} heads, seeded order); {args.steps} timed steps, {done_time:.1f} s; "
              f"BLAS: {blas_info()}")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * done_time / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "concat64k (same as the GPU arm), sampled per 2048-query block of one (episode, head)",
                   "B": lay.B, "L": lay.L, "H": lay.H, "D": lay.D},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # 200 steps of the headline step time ~1.7 s, long enough for ~9 clock samples
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="concat64k", choices=sorted(WORKLOADS) + ["adaln64k", "loss64k", "adaptive_load", "bucket_sweep"],
                    help="concat64k is the headline workload; the others are smaller cases for profiling")
    args = ap.parse_args()
    if args.warmup < 3:
        print("bench.py: raising --warmup to 3 (the minimum for a valid timing)", file=sys.stderr)
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "adaln64k":
        run_adaln(args)
    elif args.workload == "loss64k":
        run_loss(args)
    elif args.workload == "adaptive_load":
        run_adaptive(args)
    elif args.workload == "bucket_sweep":
        run_bucket_sweep(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
