"""Benchmark of the absorbed MLA decode step on B300.

One step = append the B*Q new tokens' rows (RMSNorm + RoPE + paged write)
+ decode all B sequences (plan, attend, combine), on the full-width workload
B=64, S=4096, H=128, d_c=512, d_r=64, bf16, one query token per sequence.
Inputs are seeded synthetic draws resident in HBM before timing starts.

Prints one JSON line.  `value` = decode tokens/s (B*Q query tokens per
step) over all ranks; the attention kernel's roofline fraction, the e2e
figure through host buffers and the fp64 oracle's CPU throughput are
reported alongside.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python bench.py --profile-attend N   # build, plan once, N attention launches, no timing (for ncu)
  python bench.py --workload long_split # another configuration (default: full_width, the headline)
  python bench.py --absorb              # the absorption GEMMs either side of the decode (own JSON line)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode tokens/s, cache-read GB/s and TFLOP/s vs B300 roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def algorithmic_counts(w, lowp: bool = False):
    """Bytes the method must move and flops it must do (per decode); `lowp`:
    the low-precision cache rows (656 bytes per token instead of 1152)."""
    import numpy as np
    elt = 2 if w.dtype == "bf16" else 4
    width = w.d_c + w.d_r
    row_bytes = 656 if lowp else width * elt
    cache_bytes = int(np.sum(w.lens.astype(np.int64))) * row_bytes
    q_bytes = w.B * w.Q * w.H * width * elt
    out_bytes = w.B * w.Q * w.H * w.d_c * elt
    visible = 0
    for b in range(w.B):
        for j in range(w.Q):
            visible += max(0, int(w.lens[b]) - w.Q + j + 1)
    flops = 2 * w.H * (width + w.d_c) * visible
    return cache_bytes + q_bytes + out_bytes, flops, cache_bytes


def kernel_traffic(profile_name: str, src_file: str):
    """ncu DRAM bytes per launch from the committed summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"kernel_source_sha256:\s*([0-9a-f]{16,64})", text)
    if not m or not h:
        return None
    with open(os.path.join(ROOT, src_file), "rb") as f:
        cur = hashlib.sha256(f.read()).hexdigest()
    if not cur.startswith(h.group(1)):
        return None
    return float(m.group(1))


class _Nvml:
    """Read-only NVML queries through ctypes (libnvidia-ml.so.1 ships with
    the driver; the Python NVML wheel may be absent)."""

    CLOCK_SM = 1
    REASONS = (("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20), ("hw_thermal_slowdown", 0x40),
               ("sw_power_cap", 0x4))

    def __init__(self, device):
        import ctypes
        import torch
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        p = torch.cuda.get_device_properties(device)
        bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0".encode()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(self.h)) != 0:
            idx = int(getattr(device, "index", 0) or 0)
            if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(self.h)) != 0:
                raise RuntimeError("no NVML handle")
        self._u = ctypes.c_uint()
        self._ull = ctypes.c_ulonglong()

    def max_sm_mhz(self):
        if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, self.ct.byref(self._u)) != 0:
            return None
        return float(self._u.value)

    def sample(self):
        ct = self.ct
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, ct.byref(self._u)) != 0:
            raise RuntimeError("nvmlDeviceGetClockInfo failed")
        mhz = float(self._u.value)
        watts = float("nan")
        if self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(self._u)) == 0:
            watts = self._u.value / 1000.0
        reasons = []
        if self.lib.nvmlDeviceGetCurrentClocksThrottleReasons(self.h, ct.byref(self._ull)) == 0:
            r = self._ull.value
            reasons = [n for n, m in self.REASONS if r & m]
        return mhz, watts, reasons


class ClockSampler:
    """SM clock, power and clock-event (throttle) reasons sampled about every
    millisecond during the timed region, by read-only NVML queries from a
    background thread (the timed region of a short run lasts a few
    milliseconds, so an nvidia-smi loop at 100 ms would see mostly idle
    samples)."""

    def __init__(self, device):
        self.device = device
        self.rows = []
        self.max_mhz = None
        self._stop = None
        self._thread = None
        self.error = None

    def __enter__(self):
        import threading
        try:
            nv = _Nvml(self.device)
            self.max_mhz = nv.max_sm_mhz()
        except Exception as e:  # pragma: no cover - no NVML on this machine
            self.error = f"NVML unavailable: {e}"
            return self
        self._stop = threading.Event()

        def loop():
            while not self._stop.is_set():
                try:
                    mhz, watts, reasons = nv.sample()
                except Exception as e:  # pragma: no cover
                    self.error = str(e)
                    return
                self.rows.append((time.perf_counter(), mhz, watts, reasons))
                time.sleep(0.0005)

        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()
        time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)

    def summary(self, t0=None, t1=None):
        """Median SM clock over the samples taken between t0 and t1
        (perf_counter times; all samples when none fall inside)."""
        rows = self.rows
        if t0 is not None and t1 is not None:
            inside = [r for r in rows if t0 <= r[0] <= t1]
            rows = inside or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [self.error or "no samples"]}
        reasons = sorted({n for r in rows for n in r[3]})
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(r[1] for r in rows), "power_w_max": max(r[2] for r in rows),
                "samples": len(rows), "sampler": "NVML about every 1 ms, timed region only", "reasons": reasons}


# ------------------------------------------------------------------ oracle --

class OracleStep:
    """The fp64 oracle on the host cores over sampled sequences of the
    workload.  The history cache (all but the newest Q tokens) is built once;
    a step appends each sampled sequence's newest tokens and decodes it."""

    def __init__(self, w, seqs):
        import numpy as np
        import oracle as O
        self.w, self.seqs, self.O, self.np = w, list(seqs), O, np
        first_new = {b: max(0, int(w.lens[b]) - w.Q) for b in self.seqs}
        self.caches = {b: O.sequence_cache(w, b, 0, first_new[b]) for b in self.seqs}
        self.raw_new = {b: w.raw_rows(b, first_new[b], int(w.lens[b])) for b in self.seqs}
        self.first_new = first_new
        try:
            from threadpoolctl import threadpool_info
            self.cores = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
        except Exception:  # pragma: no cover
            self.cores = os.cpu_count() or 1

    def run(self) -> int:
        w, O, np = self.w, self.O, self.np
        for b in self.seqs:
            c_raw, k_raw = self.raw_new[b]
            L = int(w.lens[b])
            rows = O.append_rows(O.widen(c_raw, w.raw_dtype), O.widen(k_raw, w.raw_dtype), np.arange(self.first_new[b], L),
                                 np.ones(w.d_c), w.eps, w.rope_base, O.append_flags(w), w.dtype)
            C = np.concatenate([self.caches[b][0], rows[:, :w.d_c]])
            R = np.concatenate([self.caches[b][1], rows[:, w.d_c:]])
            O.decode_sequence(w, b, cache=(C, R))
        return len(self.seqs) * w.Q


def oracle_throughput(w, seqs, budget_s: float = 10.0):
    """Tokens/s of the oracle, repeating steps for about `budget_s` seconds."""
    st = OracleStep(w, seqs)
    t0 = time.perf_counter()
    tokens, passes = 0, 0
    while True:
        tokens += st.run()
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return tokens / el, st.cores, el, passes


REFERENCE_BUDGET_S = 150.0   # the reference arm's timed steps end within a few minutes


def run_reference(args, w):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    # sample: up to 4 sequences per step, fewer when K steps of 4 would run
    # past the budget (one pass over one sequence is timed first)
    probe = OracleStep(w, [0])
    t0 = time.perf_counter()
    probe.run()
    per_seq = time.perf_counter() - t0
    n_seq = int(max(1, min(4, w.B, REFERENCE_BUDGET_S / max(args.steps * per_seq, 1e-9))))
    seqs = list(range(n_seq))
    st = OracleStep(w, seqs)
    for _ in range(args.warmup):
        st.run()
    t0 = time.perf_counter()
    tokens = 0
    for _ in range(args.steps):
        tokens += st.run()
    el = time.perf_counter() - t0
    value = tokens / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "S": int(w.lens[0]), "H": w.H, "Q": w.Q, "d_c": w.d_c,
                   "d_r": w.d_r},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": st.cores, "kind": "oracle",
                         "sample": f"sequences {seqs} of the workload per step (newest token appended + decoded)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- CUDA arm --

def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest of every rank's x (the job's time is its slowest rank's);
    x itself when not distributed."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank_step: int, steps: int, max_total_ms: float) -> float:
    """Units all ranks processed per second: each of `world` replicas does
    `units_per_rank_step` units per step; the job takes the slowest rank's
    total time over `steps` steps."""
    return world * units_per_rank_step / (max_total_ms * 1e-3 / steps)


def run_cuda(args, w):
    import numpy as np
    import torch

    import head_latent_attention_27_b300 as mla
    import synth
    from synth.device import empty_pool, to_torch, upload

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    # ---- resident inputs: cache built by the append kernel from raw rows
    d = upload(w, dev)
    if args.lowp:   # low-precision cache rows (E4M3 latent, fp32 group scales, bf16 RoPE key)
        pool = torch.zeros((w.num_pages, 64, mla.FP8_ROW_BYTES), dtype=torch.uint8, device=dev)
    else:
        pool = empty_pool(w, dev, fill_nan=False)
    cache = mla.Cache(pool, d["page_table"], w.d_c, w.d_r)
    flags = mla.MLA_APPEND_RMSNORM | mla.MLA_APPEND_ROPE
    mla.mla_cache_append(cache, d["raw_c"], d["raw_k"], d["seq_ids"], d["positions"], eps=w.eps,
                         rope_base=w.rope_base, flags=flags)
    # the step's new rows: the last Q tokens of every sequence
    last = np.concatenate([w.row_offset[b] + np.arange(int(w.lens[b]) - w.Q, int(w.lens[b])) for b in range(w.B)])
    new_c = d["raw_c"][torch.from_numpy(last).to(dev)].contiguous()
    new_k = d["raw_k"][torch.from_numpy(last).to(dev)].contiguous()
    new_seq = d["seq_ids"][torch.from_numpy(last).to(dev)].contiguous()
    new_pos = d["positions"][torch.from_numpy(last).to(dev)].contiguous()
    del d["raw_c"], d["raw_k"]
    out = torch.empty((w.B, w.Q, w.H, w.d_c), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Q, w.H), dtype=torch.float32, device=dev)
    n_split = args.n_split
    ws = mla.alloc_workspace(w.B, w.Q, w.H, w.d_c, n_split, dev)
    scale = 1.0 / math.sqrt(w.d_h + w.d_r)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # The step's launches are captured once in CUDA graphs (append+plan,
    # attend, combine) so that host launch overhead does not starve the GPU;
    # the event pairs bracket the replays on the same stream.  The plan reads
    # only seq_lens, so it runs on a side stream beside the append (two
    # branches of the graph) and the attention waits for both.
    s_side = torch.cuda.Stream(dev)

    def pre():
        cur = torch.cuda.current_stream(dev)
        s_side.wait_stream(cur)
        with torch.cuda.stream(s_side):
            mla.mla_decode_plan(cache, d["seq_lens"], w.Q, w.H, ws, n_split=n_split)
        mla.mla_cache_append(cache, new_c, new_k, new_seq, new_pos, eps=w.eps, rope_base=w.rope_base, flags=flags)
        cur.wait_stream(s_side)

    def attend():
        mla.mla_decode_attend(cache, d["seq_lens"], d["q_nope"], d["q_rope"], out, ws, lse=lse, n_split=n_split,
                              softmax_scale=scale)

    def post():
        mla.mla_decode_combine(cache, out, ws, lse=lse, n_split=n_split)

    launches_per_step = 4  # append, plan, attend, combine

    for _ in range(args.warmup):    # eager warm-up (also initialises the library)
        pre(); attend(); post()
        flush.zero_()
    torch.cuda.synchronize(dev)
    status = mla.mla_decode_read_status(ws)
    if status != mla.MLA_OK:
        raise RuntimeError(f"kernel status {mla.mla_status_string(status)}")
    # one graph per step (the timed `value`), and the three phases as graphs
    # of their own, replayed with an event pair around the attention alone
    # (its roofline fraction)
    graphs = []
    for fn in (pre, attend, post):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append(g)
    g_pre, g_att, g_post = graphs
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        pre(); attend(); post()
    for _ in range(args.warmup):
        g_step.replay()
        flush.zero_()
        g_pre.replay(); g_att.replay(); g_post.replay()
        flush.zero_()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    ev_att = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    ev_pre = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    ev_post = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(dev) as clk:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            ev[i][0].record(stream)
            g_step.replay()
            ev[i][1].record(stream)
            flush.zero_()          # L2 flush between steps, outside the event pairs
        torch.cuda.synchronize(dev)
        t_wall1 = time.perf_counter()
        if dist is not None:
            dist.barrier()
        t_wall = t_wall1 - t_wall0
    # the attention kernel alone (same inputs, same plan), for its roofline
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        ev_pre[i][0].record(stream)
        g_pre.replay()
        ev_pre[i][1].record(stream)
        ev_att[i][0].record(stream)
        g_att.replay()
        ev_att[i][1].record(stream)
        ev_post[i][0].record(stream)
        g_post.replay()
        ev_post[i][1].record(stream)
        flush.zero_()
    torch.cuda.synchronize(dev)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    att_ms = [a.elapsed_time(b) for a, b in ev_att]
    pre_ms = [a.elapsed_time(b) for a, b in ev_pre]
    post_ms = [a.elapsed_time(b) for a, b in ev_post]
    tot_ms = max_over_ranks(sum(step_ms), dist, dev)
    status = mla.mla_decode_read_status(ws)
    if status != mla.MLA_OK:
        raise RuntimeError(f"kernel status {mla.mla_status_string(status)}")

    # ---- e2e through the public API with host buffers (pinned), per step:
    #      H2D of the step's queries and new raw rows, append + decode, D2H of
    #      out and lse.  Steps are software-pipelined the way a serving loop
    #      runs them: two buffer sets, the H2D of step i+1 and the D2H of step
    #      i-1 on their own streams overlap the compute of step i.  Every
    #      step's own copies are inside the timed region (first H2D to last
    #      D2H); the cache (302 MB) is larger than L2.
    # A step's inputs travel as ONE packed pinned buffer and its results as
    # another (one copy per direction: measured, four separate bf16 tensor
    # copies ran at 12-15 GB/s against 55 GB/s for one packed copy).
    def packed(tensors, device, pin):
        offs, tot = [], 0
        for t in tensors:
            offs.append(tot)
            tot += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = (torch.empty(tot, dtype=torch.uint8, pin_memory=True) if pin
               else torch.empty(tot, dtype=torch.uint8, device=device))
        views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
        return buf, views

    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_pipeline(in_src, out_src, compute):
        """Times args.steps pipelined steps: per step one packed H2D of the
        inputs (laid out like `in_src`, whose values they are), compute(i,
        device input views, device output views) on buffer set i, one packed
        D2H of the outputs (laid out like `out_src`).  Returns the timed
        milliseconds (max over ranks), the host output views of every set,
        the bytes per step each way and the link-only timings."""
        # The staging buffer is written by ONE host thread: written by 16
        # threads its lines stayed dirty in the cores' private caches and the
        # DMA reads that had to snoop them ran at 12-18 GB/s instead of 50-55.
        h_in, h_views = packed(in_src, None, True)
        host_threads = torch.get_num_threads()
        torch.set_num_threads(1)
        for hv, t in zip(h_views, in_src):
            hv.copy_(t.cpu())
        torch.set_num_threads(host_threads)
        n_sets = 2
        d_in, d_in_v, d_outbuf, d_out_v, h_outbuf, h_out_v = [], [], [], [], [], []
        for _ in range(n_sets):
            buf, views = packed(in_src, dev, False)
            d_in.append(buf); d_in_v.append(views)
            buf, views = packed(out_src, dev, False)
            d_outbuf.append(buf); d_out_v.append(views)
            buf, views = packed(out_src, None, True)
            h_outbuf.append(buf); h_out_v.append(views)
        h2d = sum(t.numel() * t.element_size() for t in in_src)
        d2h = sum(t.numel() * t.element_size() for t in out_src)
        with torch.cuda.stream(s_comp):
            for i in range(n_sets):      # eager warm-up of both buffer sets
                d_in[i].copy_(h_in, non_blocking=True)
                compute(i, d_in_v[i], d_out_v[i])
        torch.cuda.synchronize(dev)
        g_comp = []
        for i in range(n_sets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                compute(i, d_in_v[i], d_out_v[i])
            g_comp.append(g)
        torch.cuda.synchronize(dev)
        ev_in = [torch.cuda.Event() for _ in range(n_sets)]
        ev_comp = [torch.cuda.Event() for _ in range(n_sets)]
        ev_out = [torch.cuda.Event() for _ in range(n_sets)]

        def run_pipeline(n_steps, t0=None, t1=None):
            if t0 is not None:
                t0.record(s_in)
            for step in range(n_steps):
                i = step % n_sets
                with torch.cuda.stream(s_in):
                    if step >= n_sets:
                        s_in.wait_event(ev_comp[i])          # set i's inputs consumed by step - 2
                    d_in[i].copy_(h_in, non_blocking=True)
                    ev_in[i].record(s_in)
                with torch.cuda.stream(s_comp):
                    s_comp.wait_event(ev_in[i])
                    if step >= n_sets:
                        s_comp.wait_event(ev_out[i])         # set i's outputs read back by step - 2
                    g_comp[i].replay()
                    ev_comp[i].record(s_comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_comp[i])
                    h_outbuf[i].copy_(d_outbuf[i], non_blocking=True)
                    ev_out[i].record(s_out)
            if t1 is not None:
                s_out.wait_stream(s_in)
                s_out.wait_stream(s_comp)
                t1.record(s_out)

        run_pipeline(max(args.warmup, n_sets))
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        run_pipeline(args.steps, t0, t1)
        torch.cuda.synchronize(dev)
        tot = max_over_ranks(t0.elapsed_time(t1), dist, dev)

        # the host link alone: the same copies with no compute, each
        # direction alone and both together
        def copies_ms(h2d_on: bool, d2h_on: bool) -> float:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            a.record(s_in)
            s_out.wait_stream(s_in)
            for step in range(args.steps):
                i = step % n_sets
                if h2d_on:
                    with torch.cuda.stream(s_in):
                        d_in[i].copy_(h_in, non_blocking=True)
                if d2h_on:
                    with torch.cuda.stream(s_out):
                        h_outbuf[i].copy_(d_outbuf[i], non_blocking=True)
            s_in.wait_stream(s_out)
            b.record(s_in)
            torch.cuda.synchronize(dev)
            return a.elapsed_time(b) / args.steps

        copies_ms(True, True)   # warm
        link = {"h2d": copies_ms(True, False), "d2h": copies_ms(False, True), "both": copies_ms(True, True)}
        last = h_out_v[(args.steps - 1) % n_sets]
        return tot, last, h2d, d2h, link

    def compute(i, ins, outs, beside=None):
        # plan beside the append (it reads only seq_lens), then attend +
        # combine; beside(): more launches on a second side stream that the
        # attention also waits for
        qn, qr, c_new, k_new = ins
        o_, l_ = outs
        cur = torch.cuda.current_stream(dev)
        s_side.wait_stream(cur)
        with torch.cuda.stream(s_side):
            mla.mla_decode_plan(cache, d["seq_lens"], w.Q, w.H, ws, n_split=n_split)
        if beside is not None:
            s_side2.wait_stream(cur)
            with torch.cuda.stream(s_side2):
                beside()
        mla.mla_cache_append(cache, c_new, k_new, new_seq, new_pos, eps=w.eps, rope_base=w.rope_base, flags=flags)
        cur.wait_stream(s_side)
        if beside is not None:
            cur.wait_stream(s_side2)
        mla.mla_decode_attend(cache, d["seq_lens"], qn, qr, o_, ws, lse=l_, n_split=n_split, softmax_scale=scale)
        mla.mla_decode_combine(cache, o_, ws, lse=l_, n_split=n_split)

    e2e_tot, (h_out_last, h_lse_last), h2d, d2h, link = e2e_pipeline(
        [d["q_nope"], d["q_rope"], new_c, new_k], [out, lse], compute)
    # the last step's result came back and matches the device-resident run
    if not (torch.equal(h_out_last, out.cpu()) and torch.equal(h_lse_last, lse.cpu())):
        raise RuntimeError("e2e result differs from the device-resident step")

    # ---- the same step with the layer's own inputs and outputs: the
    #      per-head query q^C (d_h = 128) crosses the link instead of the
    #      absorbed q_nope (d_c = 512), and the per-head output o = W^UV u
    #      instead of the latent u; both absorption GEMMs run on the device
    #      inside the timed region (synthetic seeded weights W^UK, W^UV)
    bf = lambda shape, st, sc: to_torch(synth.normal(2024, st, int(np.prod(shape)), sc, 0, "bf16").reshape(shape),
                                        "bf16", device=dev)
    n_rows = w.B * w.Q
    w_uk, w_uv = bf((w.H, w.d_h, w.d_c), 1, 1 / math.sqrt(w.d_h)), bf((w.H, w.d_h, w.d_c), 2, 1 / math.sqrt(w.d_c))
    q_c = bf((n_rows, w.H, w.d_h), 3, 1.0)
    o_layer = torch.empty((n_rows, w.H, w.d_h), dtype=torch.bfloat16, device=dev)
    qn_s = [torch.empty_like(d["q_nope"]) for _ in range(2)]
    u_s = [torch.empty_like(out) for _ in range(2)]

    s_side2 = torch.cuda.Stream(dev)

    def compute_layer(i, ins, outs):
        # the query absorption depends only on q^C: it runs beside the plan
        # and the append, and the attention waits for all three
        qc_, qr, c_new, k_new = ins
        o_, l_ = outs
        compute(i, (qn_s[i], qr, c_new, k_new), (u_s[i], l_),
                beside=lambda: mla.mla_absorb_query(w_uk, qc_, qn_s[i].view(n_rows, w.H, w.d_c)))
        mla.mla_absorb_output(w_uv, u_s[i].view(n_rows, w.H, w.d_c), o_)

    lay_tot, (h_o_last, h_l_last), lay_h2d, lay_d2h, lay_link = e2e_pipeline(
        [q_c, d["q_rope"], new_c, new_k], [o_layer, lse], compute_layer)
    # device-resident run of the same layer step, for the bit-exact check
    lse_chk = torch.empty_like(lse)
    with torch.cuda.stream(s_comp):
        compute_layer(0, (q_c, d["q_rope"], new_c, new_k), (o_layer, lse_chk))
    torch.cuda.synchronize(dev)
    if not (torch.equal(h_o_last, o_layer.cpu()) and torch.equal(h_l_last, lse_chk.cpu())):
        raise RuntimeError("layer-io e2e result differs from the device-resident run")
    status = mla.mla_decode_read_status(ws)
    if status != mla.MLA_OK:
        raise RuntimeError(f"kernel status {mla.mla_status_string(status)}")

    if rank == 0:
        peaks, peak_kind = load_peaks()
        alg_bytes, flops, cache_bytes = algorithmic_counts(w, args.lowp)
        att_avg_s = statistics.mean(att_ms) * 1e-3
        step_s = tot_ms * 1e-3 / args.steps
        tokens_per_step = w.B * w.Q
        value = whole_job_rate(world, tokens_per_step, args.steps, tot_ms)
        hbm = peaks["hbm_gbs"]
        tc_peak = peaks["bf16_tflops"]
        t_mem = alg_bytes / (hbm * 1e9)
        t_tc = flops / (tc_peak * 1e12)
        bound = "hbm" if t_mem >= t_tc else "tensor"
        achieved_gbs = alg_bytes / att_avg_s / 1e9
        achieved_tf = flops / att_avg_s / 1e12
        if w.name.startswith("full_width"):
            traffic = kernel_traffic("decode_tc_lowp_full_width.md" if args.lowp else "decode_tc_full_width.md",
                                     "head_latent_attention_27_b300/csrc/decode_tc.cu")
        elif w.name.startswith("small_head") and not args.lowp:
            traffic = kernel_traffic("decode_sh_small_head.md", "head_latent_attention_27_b300/csrc/decode_sh.cu")
        else:
            traffic = None
        if bound == "hbm":
            roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
                    "frac": achieved_gbs / hbm, "traffic": traffic}
        else:
            roof = {"bound": "tensor", "achieved": achieved_tf, "peak": tc_peak, "unit": "TFLOP/s",
                    "frac": achieved_tf / tc_peak, "traffic": traffic}
        roof.update({"kernel": ("decode_sh_kernel" if w.Q * w.H <= 16 and not args.lowp else "decode_tc_kernel")
                               + " (mla_decode_attend)", "peak_source": f"{peak_kind} burst",
                     "kernel_ms": att_avg_s * 1e3, "alg_bytes": alg_bytes, "alg_flops": flops,
                     "roofline_ms": max(t_mem, t_tc) * 1e3, "frac_of_roofline": max(t_mem, t_tc) / att_avg_s,
                     "tensor_frac": achieved_tf / tc_peak})
        # oracle sample: whole sequences, at most ~300K cached tokens of fp64 history
        seqs, tok = [], 0
        for b in range(w.B):
            if seqs and tok + int(w.lens[b]) > 300_000:
                break
            seqs.append(b)
            tok += int(w.lens[b])
        cpu_v, cores, cpu_el, cpu_steps = oracle_throughput(w, seqs, budget_s=10.0)
        clocks = clk.summary(t_wall0, t_wall1)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16 (E4M3 cache)" if args.lowp else "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "S": int(w.lens[0]) if len(set(w.lens.tolist())) == 1 else
                       f"ragged, mean {float(np.mean(w.lens)):.0f}, max {int(np.max(w.lens))}", "H": w.H, "Q": w.Q,
                       "d_c": w.d_c, "d_r": w.d_r, "page_size": 64, "n_split": n_split,
                       "cache": ("low-precision rows: E4M3 latent + fp32 scale per 128 + bf16 RoPE key, 656 B/token"
                                 if args.lowp else "bf16 rows, 1152 B/token"), "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                       "l2": "flushed between steps (write > 2x L2 outside the per-step event pairs); "
                             f"cache {cache_bytes / 1e6:.0f} MB > L2"},
            "cache_read_gbs": cache_bytes / step_s / 1e9,
            "tflops": flops / step_s / 1e12,
            "step_roofline_frac": max(t_mem, t_tc) / step_s,
            "roofline": roof,
            "cpu_baseline": {"value": cpu_v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"sequences 0..{len(seqs) - 1} of {w.B}, newest token appended + decoded, "
                                       f"{cpu_steps} pass(es) in {cpu_el:.1f} s"},
            "e2e": {"value": whole_job_rate(world, tokens_per_step, args.steps, e2e_tot), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "pipelined": "H2D of step i+1 and D2H of step i-1 overlap step i (two buffer sets); "
                                 "one packed pinned copy per direction and step",
                    "copies_only_ms_per_step": link,
                    "link_gbs": {"h2d": h2d / link["h2d"] / 1e6, "d2h": d2h / link["d2h"] / 1e6}},
            "e2e_layer_io": {"value": whole_job_rate(world, tokens_per_step, args.steps, lay_tot), "unit": UNIT,
                             "h2d_bytes_per_step": lay_h2d, "d2h_bytes_per_step": lay_d2h,
                             "work": "absorb_query (W^UK, beside the append and plan) + the step + absorb_output "
                                     "(W^UV) per step; inputs "
                                     "q^C [B*Q, H, 128] + q_rope + new rows, outputs o [B*Q, H, 128] + lse",
                             "copies_only_ms_per_step": lay_link},
            "phases_ms": {"append_and_plan": statistics.median(pre_ms), "attend": statistics.median(att_ms),
                          "combine": statistics.median(post_ms),
                          "note": "each phase replayed as a graph of its own (no overlap between phases)"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "wall_s_timed_region": t_wall,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def run_profile_attend(w, n: int, lowp: bool = False) -> None:
    """The attention kernel alone, `n` launches on one plan, for profilers
    (`lowp`: over the low-precision cache rows)."""
    import torch

    import head_latent_attention_27_b300 as mla
    from synth.device import empty_pool, upload

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    d = upload(w, dev)
    if lowp:
        pool = torch.zeros((w.num_pages, 64, mla.FP8_ROW_BYTES), dtype=torch.uint8, device=dev)
    else:
        pool = empty_pool(w, dev, fill_nan=False)
    cache = mla.Cache(pool, d["page_table"], w.d_c, w.d_r)
    mla.mla_cache_append(cache, d["raw_c"], d["raw_k"], d["seq_ids"], d["positions"], eps=w.eps,
                         rope_base=w.rope_base, flags=mla.MLA_APPEND_RMSNORM | mla.MLA_APPEND_ROPE)
    out = torch.empty((w.B, w.Q, w.H, w.d_c), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Q, w.H), dtype=torch.float32, device=dev)
    ws = mla.alloc_workspace(w.B, w.Q, w.H, w.d_c, 0, dev)
    mla.mla_decode_plan(cache, d["seq_lens"], w.Q, w.H, ws)
    for _ in range(n):
        mla.mla_decode_attend(cache, d["seq_lens"], d["q_nope"], d["q_rope"], out, ws, lse=lse,
                              softmax_scale=1.0 / math.sqrt(w.d_h + w.d_r))
    torch.cuda.synchronize(dev)
    status = mla.mla_decode_read_status(ws)
    if status != mla.MLA_OK:
        raise RuntimeError(f"kernel status {mla.mla_status_string(status)}")


def run_absorb(args) -> None:
    """The two absorption GEMMs at the full-width decode's shape (n = B*Q = 64
    query rows, H = 128, d_h = 128, d_c = 512): q_nope = W^UK_h^T q^C_h and
    o = W^UV_h u_h, each captured in a CUDA graph and timed alone with CUDA
    events around the replay, L2 flushed before every launch (the 16.8 MB
    weights fit in L2).  Prints one JSON line."""
    import numpy as np
    import torch

    import head_latent_attention_27_b300 as mla
    import synth
    from synth.device import to_torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n, H, d_h, d_c = 64, 128, 128, 512
    bf = lambda shape, st, sc: to_torch(synth.normal(2024, st, int(np.prod(shape)), sc, 0, "bf16").reshape(shape),
                                        "bf16", device=dev)
    w_uk, w_uv = bf((H, d_h, d_c), 1, 1 / math.sqrt(d_h)), bf((H, d_h, d_c), 2, 1 / math.sqrt(d_c))
    q_c, u = bf((n, H, d_h), 3, 1.0), bf((n, H, d_c), 4, 1.0)
    q_nope = torch.empty((n, H, d_c), dtype=torch.bfloat16, device=dev)
    o = torch.empty((n, H, d_h), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    peaks, src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    res = {}
    for name, fn, x, y in (("absorb_query", mla.mla_absorb_query, (w_uk, q_c), q_nope),
                           ("absorb_output", mla.mla_absorb_output, (w_uv, u), o)):
        for _ in range(max(3, args.warmup)):
            fn(*x, y, status=status)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()      # replayed, so host-side set-up is not timed
        with torch.cuda.graph(g):
            fn(*x, y, status=status)
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            ts.append((a, b))
        torch.cuda.synchronize(dev)
        us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in ts)
        alg_bytes = sum(t.numel() * t.element_size() for t in (*x, y))
        flops = 2 * n * H * d_h * d_c
        res[name] = {"us": us, "alg_bytes": alg_bytes, "achieved_gbs": alg_bytes / us * 1e-3,
                     "frac_hbm": alg_bytes / us * 1e-3 / hbm, "tflops": flops / us * 1e-6}
    if int(status.item()) != 0:
        raise RuntimeError(f"absorb kernel status {int(status.item())}")
    line = {"metric": "absorption GEMMs (W^UK into the query, W^UV after the aggregation), GB/s vs HBM roofline",
            "config": {"workload": "full_width absorption", "n_rows": n, "H": H, "d_h": d_h, "d_c": d_c,
                       "dtype": "bf16", "l2": "flushed before every launch"},
            "steps": args.steps, "peak_hbm_gbs": hbm, "peak_source": src, **res}
    print(json.dumps(line), flush=True)


def run_prefill_bench(args) -> None:
    """The expanded (prefill) form at T = 4096 prompt tokens of one sequence,
    H = 128 (the full-width decode's per-sequence shape): the up-projection
    of the cached latents into per-head K^C and V, then the causal attention
    over [K^C || k^R].  Each phase is timed with CUDA events on the launching
    stream, the L2 flushed before every step.  Prints one JSON line."""
    import numpy as np
    import torch

    import head_latent_attention_27_b300 as mla
    import synth
    from synth.device import empty_pool, to_torch, upload

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = synth.prefill(T=args.prefill_tokens, H=128)
    T, H = int(w.lens[0]), w.H
    d = upload(w, dev)
    pool = empty_pool(w, dev, fill_nan=False)
    cache = mla.Cache(pool, d["page_table"], w.d_c, w.d_r)
    mla.mla_cache_append(cache, d["raw_c"], d["raw_k"], d["seq_ids"], d["positions"], eps=w.eps,
                         rope_base=w.rope_base, flags=mla.MLA_APPEND_RMSNORM | mla.MLA_APPEND_ROPE)
    inp = {k: to_torch(v, "bf16", device=dev) for k, v in synth.prefill_inputs(w).items()}
    out = torch.empty((T, H, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    ws = torch.empty(mla.mla_prefill_workspace_size(T, H), dtype=torch.uint8, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(128 + w.d_r)

    def project():
        mla.mla_prefill_project(cache, 0, T, inp["w_uk"], inp["w_uv"], ws)

    def attend():
        mla.mla_prefill_attend(cache, 0, T, inp["q_c"], inp["q_r"], out, ws, lse=lse, softmax_scale=scale)

    for _ in range(max(3, args.warmup)):
        project()
        attend()
    torch.cuda.synchronize(dev)
    if mla.mla_decode_read_status(ws) != mla.MLA_OK:
        raise RuntimeError("prefill kernel status not OK")
    steps = min(args.steps, 50)
    evs = []
    with ClockSampler(dev) as clk:
        t0 = time.perf_counter()
        for _ in range(steps):
            flush.zero_()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record()
            project()
            e[1].record()
            attend()
            e[2].record()
            evs.append(e)
        torch.cuda.synchronize(dev)
        t1 = time.perf_counter()
    if mla.mla_decode_read_status(ws) != mla.MLA_OK:
        raise RuntimeError("prefill kernel status not OK")
    proj_ms = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    attn_ms = statistics.median(e[1].elapsed_time(e[2]) for e in evs)
    peaks, src = load_peaks()
    tc = float(peaks["bf16_tflops"])
    f_proj = 2.0 * T * w.d_c * 2 * H * 128
    f_attn = 2.0 * H * (T * (T + 1) / 2) * (128 + w.d_r + 128)
    line = {
        "metric": "MLA expanded prefill TFLOP/s vs B300 bf16 roofline",
        "value": (f_proj + f_attn) / ((proj_ms + attn_ms) * 1e-3) / 1e12, "unit": "TFLOP/s",
        "tokens_per_s": T / ((proj_ms + attn_ms) * 1e-3), "steps": steps, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "T": T, "H": H, "d_h": 128, "d_c": w.d_c, "d_r": w.d_r, "causal": True,
                   "l2": "flushed before every step"},
        "project": {"kernel": "upproj_kernel", "ms": proj_ms, "flops": f_proj,
                    "tflops": f_proj / (proj_ms * 1e-3) / 1e12, "frac": f_proj / (proj_ms * 1e-3) / 1e12 / tc},
        "roofline": {"bound": "tensor", "kernel": "prefill_attn_kernel", "achieved": f_attn / (attn_ms * 1e-3) / 1e12,
                     "peak": tc, "unit": "TFLOP/s", "frac": f_attn / (attn_ms * 1e-3) / 1e12 / tc,
                     "kernel_ms": attn_ms, "alg_flops": f_attn, "peak_source": f"{src} burst",
                     "traffic": (kernel_traffic("prefill_attn_T4096_H128.md",
                                                "head_latent_attention_27_b300/csrc/prefill.cu")
                                 if T == 4096 and H == 128 else None)},
        "clocks": clk.summary(t0, t1),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--workload", default="full_width", choices=["full_width", "small_head", "ragged_paged",
                                                                    "long_split"])
    ap.add_argument("--n-split", type=int, default=None,
                    help="uniform split of every sequence (default: 64 for long_split, else the balanced plan)")
    ap.add_argument("--profile-attend", type=int, default=0, metavar="N",
                    help="run N attention launches on one plan and exit (no timing; for ncu)")
    ap.add_argument("--absorb", action="store_true",
                    help="time the two absorption GEMMs at the full-width shape instead (own JSON line)")
    ap.add_argument("--lowp", action="store_true",
                    help="decode over the low-precision cache rows (E4M3 latent) instead of bf16 rows")
    ap.add_argument("--prefill", action="store_true",
                    help="time the expanded (prefill) form instead: projection + causal attention (own JSON line)")
    ap.add_argument("--prefill-tokens", type=int, default=4096)
    args = ap.parse_args()
    if args.prefill:
        run_prefill_bench(args)
        return
    if args.absorb:
        args.steps = min(args.steps, 200)
        run_absorb(args)
        return
    if args.warmup < 3 and args.impl == "cuda":
        args.warmup = 3
    import synth
    w = getattr(synth, args.workload)()
    if args.n_split is None:
        args.n_split = 64 if args.workload == "long_split" else 0
    if args.profile_attend > 0:
        run_profile_attend(w, args.profile_attend, args.lowp)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_cuda(args, w)


if __name__ == "__main__":
    main()
