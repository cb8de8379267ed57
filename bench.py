"""Benchmark of the GVA decode hot path on B300: one step = append + absorb + decode attention.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 4] [--path auto|fma|mma]
    python bench.py --impl reference ...     # the fp64 CPU oracle on a bounded sample

Prints ONE JSON line (rank 0).  `value` is the cache bytes the step's decode attention must
read (algorithmic: sum_b T_b * (G*d_v + d_r) * elem bytes) divided by the device time of the
whole step, with every input resident in HBM.  The step is the library's one-call step,
gva_decode_step (automatic mode: the fused kernel, or the three kernels where the batch has
many segments per range); the same step as three calls is timed beside it.  `e2e` is the same
metric through the same C-ABI call when each step's inputs start in pinned host memory and its
output returns to the host.  `roofline` is for the step's split-T partial kernel.
Under torchrun every rank runs its own replica of the workload (sequences are independent;
no collective on the data path) and the line reports the total over ranks (weak scaling).
"""
import argparse
import dataclasses
import json
import math
import os
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from compact_kv_cache_gva_b300 import gva, synth  # noqa: E402
from compact_kv_cache_gva_b300.layer import GVADecodeLayer  # noqa: E402

METRIC = "GVA decode-attention cache-read GB/s (% of B300 HBM peak) and context tokens/s"
# DRAM bytes (read + write) of one launch of the step's split-T partial kernel (the fused one,
# or the plain one), from the ncu captures summarised in profiles/ (absent where no capture of
# the current kernel exists).  The ragged batch's figure is the capture of its first 32
# sequences (73,600 units) scaled to the full batch's 254,224 units.
TRAFFIC = {("long-context-bf16", "plain"): 570_688_256, ("long-context-bf16", "fused"): 571_011_072,
           ("long-context-bf16-dr32", "fused"): 604_663_040,
           ("layer-350m-bf16", "fused"): 71_835_904, ("dr24-bf16", "fused"): 295_033_600,
           ("ragged-paged-bf16", "plain"): 4_271_621_972,
           ("long-context-fp8", "plain"): 306_442_752, ("long-context-fp8", "fused"): 306_741_248}
L2_BYTES = 126 * 1024 * 1024
NOMINAL_HBM_GBS = 8000.0  # B300 HBM3e, nominal
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
NVML_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
                0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
                0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", type=int, default=4, choices=sorted(synth.WORKLOADS))
    p.add_argument("--path", default="auto", choices=["auto", "fma", "mma"])
    p.add_argument("--step-mode", default="auto", choices=["auto", "fused", "separate"],
                   help="form of the one-call step (gva_set_step_mode)")
    p.add_argument("--split-tokens", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-gqa", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--cpu-sample-seqs", type=int, default=0, help="sequences in the CPU sample (0 = auto)")
    p.add_argument("--graph", type=int, default=0,
                   help="launch the step's kernels directly (0: each is a programmatic dependent launch of the "
                        "kernel before it, so a step's partial kernel is scheduled while the previous combine "
                        "finishes) or replay the step as a captured CUDA graph (1: graph launches do not overlap)")
    p.add_argument("--nq", type=int, default=1,
                   help="query tokens per sequence per step (the last n_q positions: append n_q tokens, "
                        "absorb B*n_q query rows, gva_decode_attention_multi)")
    p.add_argument("--cache", default="default", choices=["default", "bf16", "fp8"],
                   help="cache dtype of the workload (default: its own; fp8 = E4M3 value cache with a "
                        "power-of-two scale per token and group, bf16 positional keys)")
    p.add_argument("--batch", type=int, default=0,
                   help="keep only the first N sequences of the workload (named <name>-b<N>), e.g. for a "
                        "profiler capture small enough to hold on the device twice")
    p.add_argument("--profile", action="store_true",
                   help="run only the step's split-T partial pass: --warmup launches, then --steps more, "
                        "and print one line (for a profiler's launch filter; no timing is reported)")
    p.add_argument("--workloads", default="2,3,5,4:fp8",
                   help="other configurations measured after the headline, in the same process "
                        "(comma-separated workload ids, each optionally :fp8 for the fp8 value cache; "
                        "empty for none)")
    p.add_argument("--workload-steps", type=int, default=200,
                   help="timed steps of each of those configurations (at least --steps)")
    p.add_argument("--dr", type=int, default=-1,
                   help="override the workload's positional width d_r (0 = no positional slice, the Shared-KV "
                        "cache layout); the workload is then named <name>-dr<d_r>")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- distributed

def dist_setup(n):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        rank = int(os.environ["RANK"])
        local = int(os.environ.get("LOCAL_RANK", rank))
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        return rank, ws
    return 0, 1


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    """Largest value of x over ranks (timing is the slowest rank's)."""
    if ws == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job(per_rank_units, ws, seconds):
    """Units processed by all ranks per second of the slowest rank (weak scaling)."""
    return per_rank_units * ws / seconds


# ----------------------------------------------------------------------------- clocks

class SmiClockSampler:
    """Fallback sampler: polls nvidia-smi (SM clock, max clock, active event-reason bits)."""

    def __init__(self, period_ms=20):
        import subprocess
        self.subprocess = subprocess
        self.period_ms = period_ms
        self.samples = []
        self.max_mhz = None
        self.proc = None
        try:
            self.dev = "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid).replace(
                "GPU-", "")
        except Exception:
            self.dev = str(torch.cuda.current_device())
        self.ok = True
        self.err = ""

    def __enter__(self):
        try:
            self.proc = self.subprocess.Popen(
                ["nvidia-smi", "-i", self.dev, "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=self.subprocess.PIPE, stderr=self.subprocess.DEVNULL, text=True)
        except Exception as e:
            self.ok, self.err = False, repr(e)
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            try:
                sm, mx = int(parts[0]), int(parts[1])
                reasons = int(parts[2], 16) if parts[2].startswith("0x") else int(parts[2])
            except Exception:
                continue
            self.max_mhz = mx
            self.samples.append((sm, reasons))

    def sample(self):
        pass  # the nvidia-smi process polls on its own

    summary = None  # set below


class _Nvml:
    """The few NVML reads the clock record needs, through the driver's libnvidia-ml by ctypes
    (read-only queries: SM clock, maximum SM clock, active clock-event reasons)."""
    NVML_CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        self._ok(self.lib.nvmlInit_v2(), "nvmlInit_v2")
        self.h = ctypes.c_void_p()
        uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            self._ok(self.lib.nvmlDeviceGetHandleByIndex_v2(torch.cuda.current_device(), ctypes.byref(self.h)),
                     "nvmlDeviceGetHandleByIndex_v2")
        try:
            self._reasons_fn = self.lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self._reasons_fn = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    @staticmethod
    def _ok(rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} returned {rc}")

    def _clock(self, fn):
        v = self.c.c_uint()
        self._ok(fn(self.h, self.NVML_CLOCK_SM, self.c.byref(v)), fn.__name__)
        return int(v.value)

    def max_sm(self):
        return self._clock(self.lib.nvmlDeviceGetMaxClockInfo)

    def sm(self):
        return self._clock(self.lib.nvmlDeviceGetClockInfo)

    def reasons(self):
        v = self.c.c_ulonglong()
        self._ok(self._reasons_fn(self.h, self.c.byref(v)), "clock-event reasons")
        return int(v.value)


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML while the timed region runs: a
    polling thread, plus readings that the timing loop takes while the device is busy."""

    def __new__(cls, period_s=0.01):
        try:
            nv = _Nvml()
        except Exception:
            return SmiClockSampler()
        self = super().__new__(cls)
        self.nv = nv
        return self

    def __init__(self, period_s=0.01):
        self.period = period_s
        self.samples = []
        self.max_mhz = None
        self.ok = False
        self.err = ""
        self._stop = threading.Event()
        try:
            self.max_mhz = self.nv.max_sm()
            self.ok = True
        except Exception as e:  # report that instead of guessing
            self.err = repr(e)

    def sample(self):
        """One reading now (also called from the timing loop while the device is busy, so that
        a timed region shorter than the polling period still has samples)."""
        if not self.ok:
            return
        try:
            self.samples.append((self.nv.sm(), self.nv.reasons()))
        except Exception:
            pass

    def _run(self):
        while not self._stop.is_set():
            self.sample()
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self.t.join()

    def summary(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "NVML unavailable: " + self.err}
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        mhz = sorted(s for s, _ in self.samples)
        bits = 0
        for _, r in self.samples:
            bits |= r
        names = [n for b, n in NVML_REASONS.items() if bits & b and n != "gpu_idle"]
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": self.max_mhz, "reasons": names,
                "samples": len(self.samples)}


SmiClockSampler.summary = ClockSampler.summary


# ----------------------------------------------------------------------------- workload

class Setup:
    """A resident workload: cache, block table, lengths, step inputs, layer buffers."""

    def __init__(self, w, seed, path, split_tokens, device="cuda", n_q=1, step_mode="auto"):
        self.w, self.n_q = w, n_q
        self.inp = synth.decode_inputs(w, seed=seed, device=device)
        self.lens_cpu = self.inp.seq_lens.cpu()
        # the step appends the current token(s) at T_b - n_q .. T_b - 1 and attends through them
        # (each query through its own position), so every step has the same work
        self.raw = synth.raw_inputs(w, self.lens_cpu, n_new=n_q, seed=seed + 1000, device=device, n_q=n_q)
        self.layer = GVADecodeLayer(w.H, w.G, w.d_v, w.d_n, w.d_r, w.dtype, w.B, w.max_seq_len, device=device,
                                    split_tokens=split_tokens,
                                    path={"auto": gva.GVA_PATH_AUTO, "fma": gva.GVA_PATH_FMA,
                                          "mma": gva.GVA_PATH_MMA}[path], n_q=n_q,
                                    step_mode={"auto": gva.GVA_STEP_AUTO, "fused": gva.GVA_STEP_FUSED,
                                               "separate": gva.GVA_STEP_SEPARATE}[step_mode])
        self.sum_T = int(self.lens_cpu.sum())
        self.bytes_per_token = w.bytes_per_token
        self.cache_bytes = self.sum_T * self.bytes_per_token
        # algorithmic bytes of the decode call: cache + queries + output + lengths + table rows used
        used_blocks = int(((self.lens_cpu + 63) // 64).sum())
        self.decode_bytes = (self.cache_bytes + n_q * (w.B * w.H * (w.d_v + w.d_r) * 4 + w.B * w.H * w.d_v * 4) +
                             w.B * 4 + used_blocks * 4)
        self.decode_flops = self.sum_T * w.H * (2 * (w.d_v + w.d_r) + 2 * w.d_v)
        # the fused partial pass reads the raw queries and the key maps instead of the absorbed
        # queries, and reads the new token (cache dtype; bf16 for the fp8 cache) and writes it
        self.step_bytes = (self.cache_bytes + w.B * w.H * (w.d_n + w.d_r) * 4 + w.H * w.d_v * w.d_n * 4 +
                           w.B * ((w.G * w.d_v + w.d_r) * w.elem_bytes + w.bytes_per_token) +
                           w.B * w.H * w.d_v * 4 + w.B * 4 +
                           used_blocks * 4)

        # the library's one-call step (gva_decode_step, or gva_decode_step_multi for n_q > 1)
        self.one_call = True
        self.fused = n_q == 1 and gva.gva_step_is_fused(self.layer.ctx, w.B, w.max_seq_len) == 1
        R = w.H // w.G
        cols = 16 if w.d_v == 64 else 8  # (query, head) column pairs of a pass
        nqp_max = 1
        while 2 * nqp_max <= 4 and 2 * nqp_max * R <= cols:
            nqp_max *= 2
        passes, q = 0, 0
        while q < n_q:  # the library's passes: the largest power of two that fits, then smaller
            p = 1
            while 2 * p <= min(nqp_max, n_q - q):
                p *= 2
            q += p
            passes += 1
        self.launches_per_step = 2 if self.fused else 2 + 2 * passes

    def prime_queries(self):
        """The layer's absorbed and rotated queries (what gva_decode_partial reads when it is
        timed alone) from this step's raw queries."""
        r = self.raw
        self.layer.absorb(r.q_c, r.q_r, r.pos_q, r.M)

    def step(self, stream=None):
        r, i = self.raw, self.inp
        return self.layer.fused_step(r.q_c, r.q_r, r.M, r.v_new, r.kr_new, i.block_table, i.seq_lens, i.v_pool,
                                     i.kr_pool, stream)

    def three_call_step(self, stream=None):
        r, i = self.raw, self.inp
        return self.layer.step(r.q_c, r.q_r, r.pos_q, r.M, r.v_new, r.kr_new, r.pos_new, i.block_table,
                               i.seq_lens, i.v_pool, i.kr_pool, stream)

    def timed_step(self, ev):
        """Same step with events between the three calls: (start, after absorb, after append, end)."""
        r, i, L = self.raw, self.inp, self.layer
        ev[0].record()
        L.absorb(r.q_c, r.q_r, r.pos_q, r.M)
        ev[1].record()
        L.append(r.v_new, r.kr_new, r.pos_new, i.block_table, i.v_pool, i.kr_pool)
        ev[2].record()
        L.attend(i.v_pool, i.kr_pool, i.block_table, i.seq_lens)
        ev[3].record()


def flusher():
    """Evicts the cache between timed steps: writes one buffer twice the size of L2, then
    reads another, so the step starts with a cold L2 that holds no dirty lines (their
    write-back would otherwise land inside the timed region)."""
    buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    rd = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    sink = torch.empty((), dtype=torch.float32, device="cuda")

    def flush():
        buf.fill_(1.0)
        torch.sum(rd, dim=0, out=sink)
    return flush


def head_start():
    """Keeps the device busy (a spin kernel of about 25 ms) while the host starts enqueueing a
    timed loop, so that the device never waits for the host inside the timed region: a flushed
    step is short, and a host thread slowed by the clock-sampling thread could otherwise fall
    behind it; and an unflushed loop would otherwise start with the device idle until the host
    has enqueued its first step."""
    torch.cuda._sleep(50_000_000)


def time_steps(run_step, K, flush, clocks=None):
    """Device seconds for K steps.  Inputs larger than L2: one event pair around the K
    back-to-back steps.  Otherwise L2 is flushed before every step, outside per-step events.
    With `clocks`, two clock readings are taken once every step is enqueued, while the device
    is still working through the queue (the host enqueues a step in a fraction of its device
    time), beside the sampler's polling thread; a reading inside the loop could stall the
    enqueueing host and leave the device idle inside the timed region."""
    tick = clocks.sample if clocks is not None else (lambda: None)
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        head_start()  # the first step's launch is queued before the device reaches e0
        e0.record()
        for _ in range(K):
            run_step()
        e1.record()
        tick()
        tick()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    head_start()
    for a, b in evs:
        flush()
        a.record()
        run_step()
        b.record()
    tick()
    tick()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / 1e3


def capture(fn):
    """fn's launches captured once into a CUDA graph (after a warm call on the capture stream)."""
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        fn()
        cap.synchronize()
        with torch.cuda.graph(graph, stream=cap):
            fn()
    torch.cuda.current_stream().wait_stream(cap)
    return graph


def workload(args):
    w = synth.WORKLOADS[args.workload]
    if args.cache != "default" and args.cache != w.dtype:
        w = synth.with_cache(w, args.cache)
    if args.dr >= 0 and args.dr != w.d_r:
        w = dataclasses.replace(w, d_r=args.dr, name=f"{w.name}-dr{args.dr}")
    if args.nq > 1:
        w = dataclasses.replace(w, name=f"{w.name}-nq{args.nq}")
    if args.batch and args.batch < w.B:
        w = dataclasses.replace(w, B=args.batch, name=f"{w.name}-b{args.batch}")
    return w


def run_profile(args):
    """The step's split-T partial pass alone, launched --warmup + --steps times, for a profiler."""
    torch.cuda.init()
    w = workload(args)
    S = Setup(w, seed=0, path=args.path, split_tokens=args.split_tokens, step_mode=args.step_mode, n_q=args.nq)
    S.prime_queries()
    # multi-query: the one-call step (append, absorb, then the multi-query partial pass and combine)
    partial = partial_calls(S)[0] if S.n_q == 1 else S.step
    for _ in range(args.warmup + args.steps):
        partial()
    torch.cuda.synchronize()
    if S.layer.device_error():
        raise RuntimeError("device reported an index error")
    units = int(((S.lens_cpu + 63) // 64).sum()) * w.G
    print(json.dumps({"profile": w.name, "kernel": "fused" if S.fused else "plain", "launches": args.warmup + args.steps,
                      "units_per_launch": units, "cache_bytes": S.cache_bytes,
                      "algorithmic_bytes_per_launch": S.step_bytes if S.fused else S.decode_bytes}), flush=True)


def run_ours(args, rank, ws):
    torch.cuda.init()
    w = workload(args)
    S = Setup(w, seed=rank, path=args.path, split_tokens=args.split_tokens, n_q=args.nq, step_mode=args.step_mode)
    need_flush = S.cache_bytes < 2 * L2_BYTES
    flush = flusher() if need_flush else None

    for _ in range(max(3, args.warmup)):
        if flush:
            flush()
        S.step()
    torch.cuda.synchronize()
    if S.layer.device_error():
        raise RuntimeError("device reported an index error during warm-up")
    run_step = S.step
    if args.graph:  # the step's C-ABI call(s), replayed as one graph
        run_step = capture(S.step).replay
        for _ in range(3):
            run_step()
        torch.cuda.synchronize()

    K = args.steps
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler() as clocks:
        step_s = time_steps(run_step, K, flush, clocks)
    barrier(ws)
    total_s = max_over_ranks(step_s, ws)

    # the same step as three calls (append on a side stream beside absorb, then decode), timed alike
    three_s = None
    if S.one_call:
        for _ in range(3):
            S.three_call_step()
        three_run = capture(S.three_call_step).replay if args.graph else S.three_call_step
        for _ in range(3):
            three_run()
        torch.cuda.synchronize()
        three_s = max_over_ranks(time_steps(three_run, K, flush), ws)

    # the decode call alone (split-T partial + combine), timed the same way
    dec_s = max_over_ranks(time_steps(lambda: S.layer.attend(S.inp.v_pool, S.inp.kr_pool, S.inp.block_table,
                                                             S.inp.seq_lens), K, flush), ws)
    # the dominant kernel, the split-T partial pass, alone: events around each gva_decode_partial
    # call (the combine runs after each, outside them)
    # (several queries per sequence: the multi-query call, all its passes, is the unit timed)
    part_s = (max_over_ranks(time_partial(S, min(K, 500), flush), ws) if S.n_q == 1 else dec_s / K)
    # per-call breakdown (events between calls; informative only, they stop launch overlap)
    nb = min(K, 100)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nb)]
    if flush:
        head_start()
    for k in range(nb):
        if flush:
            flush()
        S.timed_step(evs[k])
    torch.cuda.synchronize()
    br = {name: round(1e3 * sum(e[i].elapsed_time(e[i + 1]) for e in evs) / nb, 3)
          for i, name in enumerate(("absorb", "append", "decode"))}

    ms_per_step = total_s * 1e3 / K
    value = whole_job(S.cache_bytes * K, ws, total_s) / 1e9
    tokens_per_s = whole_job(S.sum_T * K, ws, total_s)
    pk, pk_kind = peaks()
    dec_us = dec_s * 1e6 / K
    part_us = part_s * 1e6
    part_bytes = S.step_bytes if S.fused else S.decode_bytes
    achieved = part_bytes / part_s / 1e9
    hbm_peak = pk["hbm_gbs"]
    step_desc = ("gva_decode_step, fused: the split-T partial kernel absorbs and rotates the query in its "
                 "prologue and appends the new token, then the combine" if S.fused else
                 "gva_decode_step as separate kernels: append + absorb + split-T partial + combine" if S.n_q == 1
                 else f"gva_decode_step_multi: append {S.n_q} tokens + absorb {S.n_q} query rows per sequence + "
                      "the causal multi-query decode")

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": dict(w.describe(), step=step_desc, step_mode=args.step_mode, decode_path=args.path, n_q=S.n_q,
                       cuda_graph=bool(args.graph),
                       split_plan=dict(zip(("split_tokens", "partial_warps"), S.layer.plan())),
                       l2="flushed before every step (252 MB write, then 252 MB read)" if need_flush else
                       f"inputs larger than L2 ({S.cache_bytes / 1e6:.0f} MB cache)",
                       parallelism=f"replicas x{ws}" if ws > 1 else "single GPU"),
        # against the B300's nominal ~8 TB/s HBM3e peak (the target's denominator); the
        # fraction of this machine's measured copy bandwidth is reported beside it
        "pct_of_hbm_peak": round(100 * value / ws / NOMINAL_HBM_GBS, 2),
        "hbm_peak_basis": f"nominal {NOMINAL_HBM_GBS:.0f} GB/s",
        "pct_of_measured_copy_bw": round(100 * value / ws / hbm_peak, 2),
        "context_tokens_per_s": round(tokens_per_s, 1),
        "decode_steps_per_s": round(K * ws / total_s, 2),
        "three_call_step_us": round(three_s * 1e6 / K, 3) if three_s else None,
        "breakdown_us": br,
        "roofline": {"kernel": ("fused split-T partial kernel of gva_decode_step (gva_decode_step_partial)" if S.fused
                                else "split-T partial pass of gva_decode_attention (gva_decode_partial)"
                                if S.n_q == 1 else
                                f"gva_decode_attention_multi, {S.n_q} queries per sequence (partial and combine "
                                "passes)"),
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_kind": f"{pk_kind} copy bandwidth (burst)",
                     "algorithmic_bytes_per_launch": part_bytes, "partial_us": round(part_us, 3),
                     "decode_call_us": round(dec_us, 3),
                     "decode_call_GBps": round(S.decode_bytes / (dec_s / K) / 1e9, 1),
                     "traffic": TRAFFIC.get((w.name, "fused" if S.fused else "plain")),
                     "traffic_ratio": (round(TRAFFIC[(w.name, "fused" if S.fused else "plain")] / part_bytes, 4)
                                       if (w.name, "fused" if S.fused else "plain") in TRAFFIC else None)},
        "gpu_launches": S.launches_per_step * K,
        "clocks": clocks.summary(),
    }
    if args.workloads and S.n_q == 1 and args.dr < 0:
        lines = []
        for x in args.workloads.split(","):
            wid, _, cache = x.partition(":")
            other = synth.WORKLOADS[int(wid)]
            other = synth.with_cache(other, cache) if cache and cache != other.dtype else other
            if other.name != w.name:
                lines.append(run_workload_line(other, args, rank, ws))
        out["workloads"] = lines
    out["e2e"] = run_e2e(S, args.e2e_steps, flush, graph=bool(args.graph), ws=ws)
    if not args.no_gqa and rank == 0 and w.dtype == "bf16":
        out["gqa_same_build"] = run_gqa(S, flush, min(K, 500))
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and S.n_q == 1:
        out["cpu_baseline"] = cpu_baseline(S, args)
    return out


def run_workload_line(w, args, rank, ws):
    """Another configuration measured in the same process as the headline, the same way: the
    one-call step, the decode call (partial + combine) and the split-T partial pass alone, each
    timed with CUDA events over K steps (L2 flushed before every step when the cache is smaller
    than twice L2), with the clocks sampled during the step's timed region."""
    S = Setup(w, seed=rank, path=args.path, split_tokens=args.split_tokens, step_mode=args.step_mode)
    flush = flusher() if S.cache_bytes < 2 * L2_BYTES else None
    K = max(args.steps, args.workload_steps)
    S.prime_queries()
    for _ in range(max(3, args.warmup)):
        if flush:
            flush()
        S.step()
    torch.cuda.synchronize()
    if S.layer.device_error():
        raise RuntimeError(f"{w.name}: device reported an index error during warm-up")
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler() as clocks:
        step_s = time_steps(S.step, K, flush, clocks)
    barrier(ws)
    step_s = max_over_ranks(step_s, ws)
    dec_s = max_over_ranks(time_steps(lambda: S.layer.attend(S.inp.v_pool, S.inp.kr_pool, S.inp.block_table,
                                                             S.inp.seq_lens), K, flush), ws)
    part_s = max_over_ranks(time_partial(S, K, flush), ws)
    pk, pk_kind = peaks()
    part_bytes = S.step_bytes if S.fused else S.decode_bytes
    achieved = part_bytes / part_s / 1e9
    traffic = TRAFFIC.get((w.name, "fused" if S.fused else "plain"))
    line = {
        "workload": w.name, "config": w.describe(), "steps": K,
        "step_form": "fused" if S.fused else "separate",
        "l2": "flushed before every step" if flush else "inputs larger than L2",
        "value": round(whole_job(S.cache_bytes * K, ws, step_s) / 1e9, 2), "unit": "GB/s",
        "step_us": round(step_s * 1e6 / K, 3),
        "decode_call_us": round(dec_s * 1e6 / K, 3),
        "partial_us": round(part_s * 1e6, 3),
        "context_tokens_per_s": round(whole_job(S.sum_T * K, ws, step_s), 1),
        "pct_of_hbm_peak": round(100 * S.cache_bytes / (step_s / K) / 1e9 / NOMINAL_HBM_GBS, 2),
        "bytes_per_token": w.bytes_per_token,
        "bf16_bytes_per_token": synth.with_cache(w, "bf16").bytes_per_token,
        "roofline": {"kernel": "fused split-T partial kernel (gva_decode_step_partial)" if S.fused else
                     "split-T partial pass (gva_decode_partial)", "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                     "peak_kind": f"{pk_kind} copy bandwidth (burst)", "algorithmic_bytes_per_launch": part_bytes,
                     "traffic": traffic,
                     "traffic_ratio": round(traffic / part_bytes, 4) if traffic else None},
        "clocks": clocks.summary(),
    }
    del S
    torch.cuda.empty_cache()
    return line


def partial_calls(S):
    """(partial, combine): the step's split-T partial pass (the fused kernel,
    gva_decode_step_partial, when the step is fused, else gva_decode_partial) and its combine."""
    L, i, r, w = S.layer, S.inp, S.raw, S.w

    def partial():
        if S.fused:
            gva.gva_decode_step_partial(L.ctx, r.q_c, r.q_r if w.d_r else None, r.M, r.v_new.reshape(w.B, w.G, w.d_v),
                                        r.kr_new.reshape(w.B, w.d_r) if w.d_r else None, i.v_pool,
                                        i.kr_pool if w.d_r else None, i.block_table, i.seq_lens, w.max_seq_len,
                                        L.workspace)
        else:
            gva.gva_decode_partial(L.ctx, L.q_abs, L.q_rot if w.d_r else None, i.v_pool,
                                   i.kr_pool if w.d_r else None, i.block_table, i.seq_lens, w.max_seq_len,
                                   L.workspace)

    def combine():
        gva.gva_decode_combine(L.ctx, S.w.B, S.w.max_seq_len, L.out, L.workspace)
    return partial, combine


def time_partial(S, K, flush):
    """Average device seconds of the step's split-T partial pass (events on the launching stream)."""
    partial, combine = partial_calls(S)
    for _ in range(3):
        partial()
        combine()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if flush:
        head_start()
    for a, b in evs:
        if flush:
            flush()
        a.record()
        partial()
        b.record()
        combine()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / 1e3 / K


def run_e2e(S, steps, flush, graph=True, ws=1):
    """Same step, with the step's inputs copied from pinned host memory and the output read back.

    The step's inputs (queries and new tokens; for the multi-query step also their positions)
    sit in one pinned host buffer, 256-byte aligned, and move with one copy; the output comes
    back with one copy.  With
    graph=True the copy in, the step's kernels and the copy out are one captured CUDA graph,
    replayed once per step, as a serving loop would run them."""
    r = S.raw
    # the one-call step takes no positions (the lengths imply them)
    names = ("q_c", "q_r", "v_new", "kr_new") if S.one_call else ("q_c", "q_r", "pos_q", "v_new", "kr_new", "pos_new")
    offs, total = {}, 0
    for k in names:
        t = getattr(r, k)
        offs[k] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device="cuda")

    def view(buf, k):
        t = getattr(r, k)
        n = t.numel() * t.element_size()
        return buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
    for k in names:
        view(host_buf, k).copy_(getattr(r, k).cpu())
    dev_in = {k: view(dev_buf, k) for k in names}
    host_out = torch.empty(S.layer.out.shape, dtype=torch.float32).pin_memory()
    h2d = sum(getattr(r, k).numel() * getattr(r, k).element_size() for k in names)
    d2h = host_out.numel() * 4

    def e2e_step():
        dev_buf.copy_(host_buf, non_blocking=True)
        if S.one_call:
            S.layer.fused_step(dev_in["q_c"], dev_in["q_r"], r.M, dev_in["v_new"], dev_in["kr_new"],
                               S.inp.block_table, S.inp.seq_lens, S.inp.v_pool, S.inp.kr_pool)
        else:
            S.layer.step(dev_in["q_c"], dev_in["q_r"], dev_in["pos_q"], r.M, dev_in["v_new"], dev_in["kr_new"],
                         dev_in["pos_new"], S.inp.block_table, S.inp.seq_lens, S.inp.v_pool, S.inp.kr_pool)
        host_out.copy_(S.layer.out, non_blocking=True)
    def timed(fn):
        """Device seconds of `steps` steps on this rank; the slowest rank's under torchrun."""
        run = capture(fn).replay if graph else fn
        barrier(ws)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        head_start()
        for k in range(steps + 3):
            if flush:
                flush()
            e = ev[k - 3] if k >= 3 else None
            if e:
                e[0].record()
            run()
            if e:
                e[1].record()
        torch.cuda.synchronize()
        return max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) / 1e3, ws)

    # every rank moves its own replica's inputs and output: whole-job bytes and GB/s
    h2d, d2h = h2d * ws, d2h * ws
    t = timed(e2e_step)
    copies = {"value": round(whole_job(S.cache_bytes * steps, ws, t) / 1e9, 2), "unit": "GB/s",
              "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(1e3 * t / steps, 5),
              "cuda_graph": bool(graph),
              "transfer": "one copy of the packed inputs in, one copy of the output out" +
                          (", in the step's graph" if graph else ", on the step's stream")}
    if not S.one_call:
        return copies
    # The one-call step reads its inputs from, and writes its output to, pinned host memory
    # directly (mapped under unified addressing): no copy before or after the kernels.
    host_in = {k: view(host_buf, k) for k in names}

    def zero_copy_step():
        S.layer.fused_step(host_in["q_c"], host_in["q_r"], r.M, host_in["v_new"], host_in["kr_new"],
                           S.inp.block_table, S.inp.seq_lens, S.inp.v_pool, S.inp.kr_pool, out=host_out)
    zero_copy_step()
    torch.cuda.synchronize()
    host_out.fill_(float("nan"))
    zero_copy_step()
    torch.cuda.synchronize()
    want = S.layer.fused_step(r.q_c, r.q_r, r.M, r.v_new, r.kr_new, S.inp.block_table, S.inp.seq_lens,
                              S.inp.v_pool, S.inp.kr_pool).cpu()
    if not torch.equal(host_out, want):
        raise RuntimeError("the step through pinned host buffers differs from the step through device buffers")
    t0 = timed(zero_copy_step)
    zero = {"value": round(whole_job(S.cache_bytes * steps, ws, t0) / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(1e3 * t0 / steps, 5), "cuda_graph": bool(graph),
            "transfer": "the kernels read the pinned host inputs and write the pinned host output across the "
                        "bus (mapped memory, no copy)"}
    return dict(zero, copies=copies)


def run_gqa(S, flush, steps):
    """The same-build GQA decode on a matching K+V cache (same B, T, G, head width), timed alike."""
    w = S.w
    wg = synth.custom(name=w.name + "-gqa", dtype=w.dtype, B=w.B, H=w.H, G=w.G, d_v=w.d_v, d_r=0,
                      T=w.T, T_range=w.T_range, shuffled=w.shuffled)
    inp = synth.decode_inputs(wg, seed=1, device="cuda", k_pool=True)
    ctx = gva.gva_create(w.H, w.G, w.d_v, w.d_v, 0, w.dtype)
    out = torch.empty((w.B, w.H, w.d_v), device="cuda")
    wsb = torch.empty(gva.gva_decode_workspace_size(ctx, w.B, w.max_seq_len), dtype=torch.uint8, device="cuda")
    gqa_bytes = int(inp.seq_lens.sum()) * 2 * w.G * w.d_v * w.elem_bytes

    def call():
        gva.gqa_decode_attention(ctx, inp.extra["q"], inp.extra["k_pool"], inp.v_pool, inp.block_table, inp.seq_lens,
                                 w.max_seq_len, out, wsb)
    for _ in range(5):
        call()
    need_flush = gqa_bytes < 2 * L2_BYTES
    t = time_steps(call, steps, flush if need_flush else None) / steps
    del inp
    return {"decode_us": round(t * 1e6, 3), "cache_bytes": gqa_bytes, "GBps": round(gqa_bytes / t / 1e9, 1)}


# ----------------------------------------------------------------------------- CPU oracle

def cpu_sample(S, nseq, max_tokens=None):
    """Host copy of the first nseq sequences (their blocks, identity table) + the step's raw inputs.
    With max_tokens, each sequence is cut to its first max_tokens positions (the step's query and
    appended token then sit at the last of them)."""
    w, inp = S.w, S.inp
    seqs = []
    raw = {k: getattr(S.raw, k).cpu().clone() for k in ("q_c", "q_r", "pos_q", "M", "v_new", "kr_new", "pos_new")}
    for b in range(nseq):
        T = int(S.lens_cpu[b]) if max_tokens is None else min(int(S.lens_cpu[b]), max_tokens)
        nblk = (T + 63) // 64
        ids = inp.block_table[b, :nblk].long()
        if w.dtype == "fp8":  # the blocks' codes, then their exponents
            codes, exps = gva.fp8_pool_views(inp.v_pool, w.G, w.d_v)
            vsel = torch.cat([codes.index_select(0, ids).reshape(-1),
                              exps.index_select(0, ids).view(torch.uint8).reshape(-1)])
        else:
            vsel = inp.v_pool.index_select(0, ids)
        seqs.append((b, T, synth.pool_bits(vsel), synth.pool_bits(inp.kr_pool.index_select(0, ids))))
        raw["pos_q"][b] = T - 1
        raw["pos_new"][b] = T - 1
    return seqs, raw


def oracle_step(w, seqs, raw):
    """One oracle step on the sample: absorb + append + decode of every head of each sequence.
    Returns (seconds, cache bytes read)."""
    import numpy as np
    import oracle
    t0 = time.perf_counter()
    nbytes = 0
    for b, T, vp, kp in seqs:
        vp = vp.copy()
        kp = kp.copy()
        table = np.arange(vp.shape[0], dtype=np.int32)[None]
        qa, qr = oracle.absorb(raw["q_c"][b:b + 1].double().numpy(), raw["q_r"][b:b + 1].double().numpy(),
                               raw["pos_q"][b:b + 1].numpy(), raw["M"].double().numpy())
        oracle.append(synth.pool_bits(raw["v_new"][b:b + 1]), synth.pool_bits(raw["kr_new"][b:b + 1]),
                      raw["pos_new"][b:b + 1].numpy(), table, vp, kp)
        oracle.decode(qa, qr, vp, kp, table, np.array([T], np.int32), G=w.G, d_n=w.d_n)
        nbytes += T * w.bytes_per_token
    return time.perf_counter() - t0, nbytes


def auto_sample_seqs(S):
    # about 1.5e9 multiply-adds of fp64 oracle work: seconds of CPU time on the host cores
    w = S.w
    per_token = w.H * (2 * w.d_v + w.d_r)
    budget = 1.5e9
    n, acc = 0, 0
    for b in range(w.B):
        acc += int(S.lens_cpu[b]) * per_token
        n += 1
        if acc >= budget:
            break
    return n


def cpu_baseline(S, args):
    import oracle
    nseq = args.cpu_sample_seqs or auto_sample_seqs(S)
    seqs, raw = cpu_sample(S, nseq)
    threads = oracle.get_threads()
    secs, nbytes = oracle_step(S.w, seqs, raw)
    toks = sum(T for _, T, _, _ in seqs)
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"one step (absorb+append+decode, all {S.w.H} heads) of the first {nseq} sequence(s) "
                      f"of the workload, {toks} context tokens, {secs:.2f} s wall",
            "context_tokens_per_s": round(toks / secs, 1)}


def run_reference(args, rank, ws):
    """The oracle as the reference arm: K timed steps of a bounded sample on the host cores."""
    import oracle
    w = workload(args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    S = Setup.__new__(Setup)
    S.w = w
    S.inp = synth.decode_inputs(w, seed=0, device=dev)
    S.lens_cpu = S.inp.seq_lens.cpu()
    S.raw = synth.raw_inputs(w, S.lens_cpu, n_new=1, seed=1000, device=dev)
    nseq = 1
    seqs, raw = cpu_sample(S, nseq)
    # bound the run to about 150 s: one step of the whole sequence sets the tokens per step
    full_s, _ = oracle_step(w, seqs, raw)
    budget = 150.0 / max(1, args.steps + args.warmup)
    T0 = int(S.lens_cpu[0])
    if full_s > budget:
        seqs, raw = cpu_sample(S, nseq, max_tokens=max(64, int(T0 * budget / full_s) // 64 * 64))
    for _ in range(args.warmup):
        oracle_step(w, seqs, raw)
    t, nbytes = 0.0, 0
    for _ in range(args.steps):
        dt, nb = oracle_step(w, seqs, raw)
        t += dt
        nbytes += nb
    value = nbytes / t / 1e9
    threads = oracle.get_threads()
    sample = (f"per step: absorb+append+decode of all {w.H} heads of sequence 0 of the workload, cut to its "
              f"first {seqs[0][1]} of {T0} context tokens (sized so the {args.steps}-step run takes about "
              f"150 s)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": w.describe(),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, ws = dist_setup(args.gpus)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, ws)), flush=True)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
    if args.profile:
        run_profile(args)
        return
    out = run_ours(args, rank, ws)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
