#!/usr/bin/env python
"""Benchmark of the q8-KV decode step on GB300.

One step = the whole hot path over one batch: quantise-append of the step's
new K/V token for every (layer, kv head), split-KV decode attention of every
query head over its paged int8 context, and the split merge: one
kvq8_decode_step call (two launches: the split kernel, which also appends the
step's new token, and the merge, whose launch overlaps the split's tail
through programmatic dependent launch; the three separate entry points --
append, split, merge -- called one by one are timed beside it as `unfused`).
The default workload is the 28-layer Qwen3-2B-shaped decode stack (16 query /
8 kv heads, hd 128, context 8192, batch 1), its layers folded into the batch
dimension of one call.

Prints one JSON line.  `value` is achieved algorithmic HBM throughput in GB/s
(bytes a step must move / device time per step) summed over ranks;
`us_per_step` and `ms_per_step` are the device time of one step.  Inputs are
resident in HBM; every timed loop rotates over several copies of the cache so
that every step streams from HBM (the working set is far above L2).

The dominant kernel's roofline comes from its own loop of at least 500
back-to-back launches (whatever --steps says), with CUDA events on the
launching stream around the loop; a second loop with events around every
launch gives the duration of a launch on its own (what ncu reports per
launch).  nvidia-smi samples the SM clock and throttle reasons over the
loaded window (those loops and the timed steps, which follow them).

With the default workload the line also carries `workloads`: the batched
decode (batch 64, ragged 512-32K), the 128K decode with outlier channels, the
single-head L=256 case, the bulk append, the INT4 group-64 decode and the
mixed-precision decode, each timed the same way (K steps, the dominant
kernel's loops, clocks).

`--impl reference` times the CPU oracle on the host cores instead.
`--gpus N` without a launcher around it starts N local ranks itself
(torch.distributed.run); multi-GPU runs are independent replicas: the path
needs no exchange between GPUs.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "q8-KV decode attention: μs/step and achieved HBM GB/s (% of GB300 peak)"
DEFAULT_WORKLOAD = "qwen3_2b_28layers_ctx8192"
# the other workloads reported in the default run's `workloads` record
SUB_WORKLOADS = ("batch64_ctx512to32768", "batch4_ctx131072_outliers", "single_head_l256",
                 "append_batch8_4096tokens", "int4g64_batch8_ctx32768",
                 "mixed_qwen3_2b_28layers_ctx8192")
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e nominal bandwidth (context beside the measured peak)
THROTTLE_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
ROOF_MIN_LAUNCHES = 500     # launches of the dominant kernel's own loops
ROOF_TARGET_S = 0.3         # device time of the back-to-back loop (at least)
CLOCK_INTERVAL_MS = 50
HOLD_CYCLES = 100_000       # spin kernel queued before a timed region: about 50 us at 2 GHz


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("kvq8", "reference"), default="kvq8")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--copies", type=int, default=0,
                    help="cache copies to rotate over (0 = enough to exceed 8x L2)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads' records in the default run")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0 = min(steps, 2000)")
    ap.add_argument("--no-f32", action="store_true",
                    help="skip the fp32-KV decode comparator leg")
    ap.add_argument("--plain-step", action="store_true",
                    help="time the decode step without KVQ8_STEP_CACHE_READY")
    ap.add_argument("--roof-launches", type=int, default=ROOF_MIN_LAUNCHES,
                    help="launches of each of the dominant kernel's loops (at least)")
    ap.add_argument("--roof-seconds", type=float, default=ROOF_TARGET_S,
                    help="device time of the back-to-back loop (at least)")
    return ap.parse_args(argv)


# ----------------------------------------------------------------- ranks ---
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def reduce_scalar(x: float, op: str, device) -> float:
    """max or sum of a per-rank scalar over all ranks (identity when alone)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate(per_rank_bytes: float, per_rank_seconds: float, device):
    """Whole-job throughput of independent replicas: all ranks' bytes / slowest rank's time."""
    total = reduce_scalar(per_rank_bytes, "sum", device)
    slowest = reduce_scalar(per_rank_seconds, "max", device)
    return total, slowest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def self_launch(n: int, argv) -> int:
    """`--gpus N` run without a launcher: start N local ranks of this script
    under torch.distributed.run (rendezvous on 127.0.0.1) and return their exit
    status; rank 0 prints the line."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.abspath(__file__), *argv]
    return subprocess.run(cmd, cwd=ROOT).returncode


# ---------------------------------------------------------------- clocks ---
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, each stamped with the
    host time of its arrival; stop() summarises the samples that fell inside
    the window opened by open() and closed by close()."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = CLOCK_INTERVAL_MS):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.thread = None
        self.error = None
        self.samples = []
        self.t0 = self.t1 = None
        self._first = threading.Event()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), line))
            self._first.set()

    def start(self, wait_s: float = 5.0):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError as e:
            self.error = f"nvidia-smi unavailable: {e}"
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        self._first.wait(wait_s)   # nvidia-smi is up before the loaded window opens
        return self

    def open(self):
        self.t0 = time.monotonic()

    def close(self):
        self.t1 = time.monotonic()

    def stop(self):
        if self.proc is None:
            return {"error": self.error or "not started"}
        time.sleep(2 * self.interval / 1e3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        t0 = self.t0 if self.t0 is not None else -math.inf
        t1 = (self.t1 if self.t1 is not None else math.inf) + 0.5 * self.interval / 1e3
        sm, smax, reasons = [], [], set()
        for ts, line in self.samples:
            if not t0 <= ts <= t1:
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(THROTTLE_REASONS, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        window_ms = None if self.t0 is None or self.t1 is None else round((self.t1 - self.t0) * 1e3, 1)
        if not sm:
            return {"error": "no samples in the loaded window", "window_ms": window_ms}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm), "window_ms": window_ms,
                "interval_ms": self.interval,
                "window": "the dominant kernel's loops and the timed steps right after them"}


# ------------------------------------------------------------------ peaks ---
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Sources that decide each timed kernel's code (the .cu and every header it
# includes); a DRAM-traffic record is used only while their hash matches.
_HEADERS = ("kvq8_device.cuh", "kvq8_internal.cuh", "kvq8_ptx.cuh", "../../include/kvq8.h")
KERNEL_SOURCES = {
    "decode_split_kernel": ("decode.cu",) + _HEADERS,
    "quantize_append_kernel": ("append.cu",) + _HEADERS,
    "kvq4_decode_attn": ("int4.cu", "decode.cu") + _HEADERS,
    "kvmix_decode_attn": ("int4.cu", "decode.cu") + _HEADERS,
}


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "int8_quantized_kv_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes (read + written) per launch of `kernel` on `workload`, from the
    committed ncu summary, if it was taken on the current source; else None."""
    p = os.path.join(ROOT, "profiles", "kernel_traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)["records"][kernel]
    except (OSError, ValueError, KeyError):
        return None
    if rec.get("source_hash") != kernel_source_hash(kernel):
        return None
    return rec.get("per_launch_bytes", {}).get(workload)


def finish_roofline(r: dict, us_per_step: float, clocks: dict, peak: float, peak_kind: str) -> dict:
    """Fill the derived fields of a roofline record: achieved GB/s and its
    fraction of the measured and the nominal peak, clock-normalised time, the
    traffic check -- and refuse the figure when the kernel's mean launch is
    longer than the whole step that contains it (an inconsistent measurement)."""
    us = r["us_per_launch"]
    r["peak"], r["peak_kind"], r["unit"] = peak, peak_kind, "GB/s"
    if r.get("part_of_step", True) and us > us_per_step * 1.0005:
        r["achieved"] = r["frac"] = None
        r["rejected"] = (f"mean launch {us:.2f} us exceeds the step {us_per_step:.2f} us that contains it: "
                         "not a valid roofline figure")
    else:
        achieved = r["algorithmic_bytes_per_launch"] / (us * 1e-6) / 1e9
        r["achieved"] = round(achieved, 2)
        r["frac"] = round(achieved / peak, 4)
        r["nominal_peak"] = NOMINAL_HBM_GBS
        r["frac_of_nominal"] = round(achieved / NOMINAL_HBM_GBS, 4)
    if isinstance(clocks, dict) and clocks.get("sm_mhz"):
        r["sm_mhz_median"] = clocks["sm_mhz"]
        r["us_x_sm_mhz"] = round(us * clocks["sm_mhz"], 1)   # SM cycles per launch at the median clock
    if r.get("traffic") and r.get("algorithmic_bytes_per_launch"):
        ratio = r["traffic"] / r["algorithmic_bytes_per_launch"]
        r["traffic_over_algorithmic"] = round(ratio, 4)
        if ratio > 1.05:
            r["traffic_check"] = "more than 5 % above the algorithmic bytes: re-reads"
        elif ratio < 0.95:
            r["traffic_check"] = ("more than 5 % below the algorithmic bytes: served from L2, or writes "
                                  "still in L2 at the kernel's end")
        else:
            r["traffic_check"] = "within 5 % of the algorithmic bytes"
    return r


# ------------------------------------------------------------- workloads ---
def step_bytes(cfg, lens):
    """Algorithmic bytes of one step: the decode pass plus the append of one
    token per (sequence, kv head)."""
    from int8_quantized_kv_gb300 import workloads as wl
    return (wl.algorithmic_decode_bytes(cfg, lens) +
            wl.algorithmic_append_bytes(cfg.batch * cfg.nkv, cfg.hd))


def split_kernel_bytes(cfg, lens):
    """Algorithmic bytes the split kernel moves: int8 K/V + two fp32 scales per
    (token, kv head), and the fp32 queries."""
    import numpy as np
    tok = int(np.asarray(lens, np.int64).sum())
    return tok * cfg.nkv * (2 * cfg.hd + 8) + cfg.batch * cfg.nqh * cfg.hd * 4


def f32_decode_bytes(cfg, lens):
    """Algorithmic bytes of the fp32-KV decode: fp32 K/V per (token, kv head),
    the fp32 queries and outputs."""
    import numpy as np
    tok = int(np.asarray(lens, np.int64).sum())
    return tok * cfg.nkv * 2 * cfg.hd * 4 + 2 * cfg.batch * cfg.nqh * cfg.hd * 4


def q8_cache_bytes(num_blocks: int, nkv: int, hd: int = 128) -> int:
    """Bytes of one int8 cache (both pools and both scale arrays)."""
    return num_blocks * nkv * 256 * (2 * hd + 8)


def q8_copies(cache_bytes: int, requested: int = 0):
    """(copies to rotate over, L2-resident?): enough copies that the working set
    exceeds 8x L2; a cache of a few hundred KB stays in L2 by construction."""
    l2_resident = cache_bytes * 8 < L2_BYTES // 16
    return requested or (1 if l2_resident else max(2, math.ceil(8 * L2_BYTES / cache_bytes))), l2_resident


def workload_config(cfg, lens, copies, world, sbytes):
    """The `config` of a q8 decode line (the same dict in both arms)."""
    import numpy as np
    c = {"workload": cfg.name, "layers_folded_into_batch": cfg.layers,
         "batch": cfg.batch // max(cfg.layers, 1), "nqh": cfg.nqh, "nkv": cfg.nkv, "hd": cfg.hd,
         "block_size": 256, "ctx": int(lens.max()) if cfg.ctx is not None else
         [int(lens.min()), int(lens.max())], "tokens": int(np.asarray(lens).sum()),
         "step": "append 1 token per (layer, kv head) + split-KV decode + merge",
         "block_table": "seeded shuffled physical blocks"}
    if copies == 1:
        c["l2"] = "one cache copy: L2-resident by construction, latency-bound"
    else:
        c["l2"] = f"rotates {copies} cache copies; working set >> 129 MB L2, no flush"
    c["parallelism"] = f"replicas{world}"
    c["bytes_per_step"] = sbytes
    c["arithmetic"] = "int8 x int8 -> int32 block dots, fp32 softmax and accumulation"
    return c


def q8_decode_config(cfg, world):
    """Everything the q8 decode `config` depends on, from the workload alone
    (no device work): lens, the table's pool size, the rotation."""
    from int8_quantized_kv_gb300 import workloads as wl
    lens = wl.ctx_lens(cfg)
    _, num_blocks = wl.block_table(cfg, lens)
    copies, l2_resident = q8_copies(q8_cache_bytes(num_blocks, cfg.nkv, cfg.hd))
    return lens, copies, l2_resident, workload_config(cfg, lens, copies, world, step_bytes(cfg, lens))


# ------------------------------------------------------------ CPU oracle ---
class OracleStep:
    """The oracle's share of one step for a sample of (sequence, kv head) units:
    quantise the new token's K/V rows and the G query heads, then the three-pass
    decode over the unit's int8 context (prepared beforehand: cache state)."""

    def __init__(self, cfg, lens, units, sm_scale):
        import numpy as np
        import oracle
        from int8_quantized_kv_gb300 import workloads as wl
        self.cfg, self.units, self.sm = cfg, units, sm_scale
        self.q = wl.queries(cfg)
        self.state = {}
        for b, h in units:
            L = int(lens[b])
            k, v = wl.unit_kv(cfg, b, h, L)
            kq, ks = oracle.kv_quantize_rows(k[:L - 1])
            vq, vs = oracle.kv_quantize_rows(v[:L - 1])
            self.state[(b, h)] = (np.concatenate([kq, np.zeros((1, cfg.hd), np.int8)]),
                                  np.concatenate([ks, np.zeros(1, np.float32)]),
                                  np.concatenate([vq, np.zeros((1, cfg.hd), np.int8)]),
                                  np.concatenate([vs, np.zeros(1, np.float32)]),
                                  k[L - 1:L].copy(), v[L - 1:L].copy())

    def run_unit(self, u):
        import oracle
        b, h = u
        kq, ks, vq, vs, kn, vn = self.state[u]
        nkq, nks = oracle.kv_quantize_rows(kn)
        nvq, nvs = oracle.kv_quantize_rows(vn)
        kq[-1], ks[-1], vq[-1], vs[-1] = nkq[0], nks[0], nvq[0], nvs[0]
        G = self.cfg.group
        qi, qsc = oracle.q_quantize_blocks(self.q[b, h * G:(h + 1) * G])
        return oracle.decode_quantized_unit(qi, qsc, kq, ks, vq, vs, self.sm)

    def run(self, threads):
        import oracle
        return oracle.run_parallel(self.run_unit, self.units, threads)


def sample_units(cfg, lens, target_seconds, threads, max_units=None):
    """Pick a seeded sample of units whose oracle step takes about target_seconds."""
    import numpy as np
    all_units = [(b, h) for b in range(cfg.batch) for h in range(cfg.nkv) if lens[b] > 1]
    rng = np.random.default_rng(12345)
    order = [all_units[i] for i in rng.permutation(len(all_units))]
    probe = order[:max(1, min(len(order), threads))]
    t0 = time.perf_counter()
    OracleStep(cfg, lens, probe, 1.0).run(threads)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(len(probe) * target_seconds / dt)
    n = max(len(probe), min(len(order), n))
    if max_units:
        n = min(n, max_units)
    return order[:n], all_units


def cpu_baseline(cfg, lens, target_seconds):
    import numpy as np
    threads = len(os.sched_getaffinity(0))
    sm = np.float32(1.0 / math.sqrt(cfg.hd))
    units, all_units = sample_units(cfg, lens, target_seconds / 2, threads)
    st = OracleStep(cfg, lens, units, sm)
    reps, t_total = 0, 0.0
    while reps < 1 or (t_total < target_seconds and reps < 5):
        t0 = time.perf_counter()
        st.run(threads)
        t_total += time.perf_counter() - t0
        reps += 1
    per_rep = t_total / reps
    total_tokens = sum(int(lens[b]) for b, _ in all_units)
    frac = sum(int(lens[b]) for b, _ in units) / total_tokens
    full_step_s = per_rep / frac
    value = step_bytes(cfg, lens) / full_step_s / 1e9
    # the same oracle on one core, over a smaller sample
    units1, _ = sample_units(cfg, lens, target_seconds / 4, 1)
    st1 = OracleStep(cfg, lens, units1, sm)
    t0 = time.perf_counter()
    st1.run(1)
    t1 = time.perf_counter() - t0
    frac1 = sum(int(lens[b]) for b, _ in units1) / total_tokens
    full1_s = t1 / frac1
    return {"value": round(value, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": (f"{len(units)} of {len(all_units)} (sequence, kv head) units of one step "
                       f"({frac:.1%} of its tokens), {reps} repetition(s), scaled to a full step "
                       f"of {full_step_s * 1e3:.1f} ms"),
            "ms_per_full_step": round(full_step_s * 1e3, 3),
            "single_core": {"value": round(step_bytes(cfg, lens) / full1_s / 1e9, 3), "unit": "GB/s",
                            "ms_per_full_step": round(full1_s * 1e3, 3),
                            "sample": f"{len(units1)} units ({frac1:.1%} of the step's tokens), once"}}


# ---------------------------------------------------------- GPU harness ---
class Gpu:
    """Per-rank device state shared by the workload runners."""

    def __init__(self, args, rank, world, local):
        import torch
        self.args, self.rank, self.world, self.local = args, rank, world, local
        self.dev = torch.device("cuda", local)
        torch.cuda.set_device(self.dev)
        dist_init(world, "nccl")
        from int8_quantized_kv_gb300 import kvq8
        kvq8.load()
        self.stream = torch.cuda.current_stream(self.dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.dev)

    def check_status(self, where: str):
        v = int(self.status.item())
        if v != 0:
            raise RuntimeError(f"device status {v:#x} {where}")

    def event(self):
        import torch
        return torch.cuda.Event(enable_timing=True)

    def hold(self):
        """Keeps the stream busy for about 50 us (a spin kernel queued before a
        timed region's first event) so that the host queues the region's first
        launches while the device still works: the region then times the
        device's execution of its steps, not the host's latency to submit the
        first one after an idle synchronise (the blocking-kernel technique of
        GPU benchmark harnesses)."""
        import torch
        torch.cuda._sleep(HOLD_CYCLES)

    def loop_s(self, fn, n: int, first: int = 0) -> float:
        """Device seconds per call of fn(i), i = first .. first+n-1, back to back
        (one pair of events around the whole loop)."""
        import torch
        e0, e1 = self.event(), self.event()
        torch.cuda.synchronize()
        self.hold()
        e0.record(self.stream)
        for i in range(first, first + n):
            fn(i)
        e1.record(self.stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / n

    def isolated_s(self, fn, n: int) -> float:
        """Mean device seconds of one call of fn(i) with events right around it,
        over n calls: the duration of a launch on its own."""
        import torch
        evs = [(self.event(), self.event()) for _ in range(n)]
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(evs):
            a.record(self.stream)
            fn(i)
            b.record(self.stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / 1e3 / n

    def measure(self, step, kernel_call, kernel_name, kernel_bytes, sbytes, launches_per_step,
                part_of_step=True):
        """The timing protocol of every workload.  After the warm-up steps: the
        clock sampler starts; the dominant kernel's call runs in its own loops
        (back to back for at least ROOF_TARGET_S and ROOF_MIN_LAUNCHES launches;
        then ROOF_MIN_LAUNCHES launches each between its own events); then
        exactly --steps steps run between one pair of events (barrier and
        synchronize on both sides).  Returns (per-rank step seconds, whole-job
        bytes, slowest rank's seconds, roofline record, clocks)."""
        import torch
        args = self.args
        for i in range(max(3, args.warmup)):
            step(i)
        torch.cuda.synchronize()
        self.check_status("during warm-up")
        est = self.loop_s(kernel_call, 3)
        n_roof = max(1, args.roof_launches)
        n_b2b = max(n_roof, int(math.ceil(args.roof_seconds / max(est, 1e-7))))
        sampler = ClockSampler(self.local).start()
        sampler.open()
        b2b = self.loop_s(kernel_call, n_b2b)
        iso = self.isolated_s(kernel_call, n_roof)
        t_start, t_end = self.event(), self.event()
        barrier()
        torch.cuda.synchronize()
        self.hold()
        t_start.record(self.stream)
        for i in range(args.steps):
            step(i)
        t_end.record(self.stream)
        torch.cuda.synchronize()
        sampler.close()
        barrier()
        clocks = sampler.stop()
        self.check_status("in the timed region")
        elapsed = t_start.elapsed_time(t_end) / 1e3
        total, slowest = aggregate(sbytes * args.steps, elapsed, self.dev)
        roof = {"bound": "hbm", "kernel": kernel_name, "algorithmic_bytes_per_launch": kernel_bytes,
                "us_per_launch": round(b2b * 1e6, 3), "launches": n_b2b,
                "us_per_launch_isolated": round(iso * 1e6, 3), "launches_isolated": n_roof,
                "timing": ("us_per_launch: mean of a loop of back-to-back launches rotating the cache "
                           "copies (CUDA events on the launching stream around the loop); "
                           "us_per_launch_isolated: mean over launches each between its own events"),
                "part_of_step": part_of_step}
        return elapsed / args.steps, total, slowest, roof, clocks, launches_per_step * args.steps


def finish_line(gpu, line, roof, clocks, us_per_step, traffic):
    peak, kind = hbm_peak()
    roof["traffic"] = traffic
    line["roofline"] = finish_roofline(roof, us_per_step, clocks, peak, kind)
    line["pct_of_hbm_peak"] = round(100 * (line["value"] / gpu.world) / peak, 2)
    line["clocks"] = clocks
    return line


def base_line(gpu, value, steps, slowest, dtype, config):
    per_step = slowest / steps
    return {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": gpu.world,
            "steps": steps, "warmup": gpu.args.warmup, "ms_per_step": round(per_step * 1e3, 5),
            "us_per_step": round(per_step * 1e6, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic", "config": config,
            "timed_region": ("the --steps steps between two CUDA events on the launching stream, "
                             "queued behind a ~50 us spin kernel so that the events time the device's "
                             "execution of the steps, not the host's latency to submit the first")}


# ------------------------------------------------------------- q8 decode ---
def bench_q8(gpu, cfg, full):
    """The q8 decode step (kvq8_decode_step) on a decode workload."""
    import numpy as np
    import torch
    from int8_quantized_kv_gb300 import kvq8
    from int8_quantized_kv_gb300 import workloads as wl
    args, dev, stream, status = gpu.args, gpu.dev, gpu.stream, gpu.status
    lens, copies, l2_resident, config = q8_decode_config(cfg, gpu.world)
    if args.copies:
        copies = args.copies
        config = workload_config(cfg, lens, copies, gpu.world, step_bytes(cfg, lens))
    table, num_blocks = wl.block_table(cfg, lens)
    max_blocks = table.shape[1]
    sm = 1.0 / math.sqrt(cfg.hd)

    # fill cache copy 0 with the first L-1 tokens of every sequence; the step
    # appends token L-1 (the same token every step, so steps are identical)
    c0 = kvq8.alloc_cache(num_blocks, cfg.nkv, dev)
    table_d = torch.from_numpy(table).to(dev)
    new_k = np.zeros((cfg.batch, 1, cfg.nkv, cfg.hd), np.float32)
    new_v = np.zeros_like(new_k)
    zero = torch.zeros(1, dtype=torch.int32, device=dev)
    # the fp32 comparator cache holds the same L tokens (the q8 cache has token
    # L-1 after the first step)
    cf = None if (args.no_f32 or not full) else kvq8.alloc_cachef32(num_blocks, cfg.nkv, dev)
    for b in range(cfg.batch):
        L = int(lens[b])
        k, v = wl.seq_kv(cfg, b, L)
        new_k[b, 0], new_v[b, 0] = k[L - 1], v[L - 1]
        if L > 1:
            kvq8.quantize_append(torch.from_numpy(k[None, :L - 1]).to(dev),
                                 torch.from_numpy(v[None, :L - 1]).to(dev), zero,
                                 table_d[b:b + 1], c0)
        if cf is not None and L > 0:
            kvq8.appendf32(torch.from_numpy(k[None]).to(dev), torch.from_numpy(v[None]).to(dev), zero,
                           table_d[b:b + 1], cf)
    caches = [c0] + [kvq8.KVCache(*[t.clone() for t in c0]) for _ in range(copies - 1)]
    q_d = torch.from_numpy(wl.queries(cfg)).to(dev)
    nk_d, nv_d = torch.from_numpy(new_k).to(dev), torch.from_numpy(new_v).to(dev)
    start_d = torch.from_numpy((lens - 1).clip(min=0).astype(np.int32)).to(dev)
    lens_d = torch.from_numpy(lens).to(dev)
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, max_blocks, dev)
    out = torch.empty_like(q_d)
    nk1, nv1 = nk_d[:, 0], nv_d[:, 0]   # the step's token, [batch][nkv][hd]

    # The steps of the timed loop differ only in their query and new token:
    # the kernel before each step's split (the previous step's merge) writes
    # only `out`, so every step may pass KVQ8_STEP_CACHE_READY
    ready = not args.plain_step

    def step(i):
        kvq8.decode_step(q_d, nk1, nv1, caches[i % copies], table_d, lens_d, out, ws, sm_scale=sm,
                         dev_status=status, stream=stream, cache_ready=ready)

    def split(i):
        kvq8.decode_split(q_d, caches[i % copies], table_d, lens_d, ws, sm_scale=sm, dev_status=status,
                          stream=stream)

    def unfused_step(i):
        c = caches[i % copies]
        kvq8.quantize_append(nk_d, nv_d, start_d, table_d, c, dev_status=status, stream=stream)
        kvq8.decode_split(q_d, c, table_d, lens_d, ws, sm_scale=sm, dev_status=status, stream=stream)
        kvq8.decode_combine(cfg.batch, cfg.nqh, cfg.nkv, max_blocks, lens_d, ws, out, stream=stream)

    sbytes = step_bytes(cfg, lens)
    split_bytes = split_kernel_bytes(cfg, lens)
    per_step_s, total, slowest, roof, clocks, launches = gpu.measure(
        step, split, "decode_split_kernel", split_bytes, sbytes, 2)
    line = base_line(gpu, total / slowest / 1e9, args.steps, slowest, "int8", config)
    line["gpu_launches"] = launches
    line["step_call"] = ("kvq8_decode_step_ex with KVQ8_STEP_CACHE_READY" if ready else
                         "kvq8_decode_step_ex without flags")
    finish_line(gpu, line, roof, clocks, line["us_per_step"],
                recorded_traffic("decode_split_kernel", cfg.name))
    if l2_resident:
        line["roofline"]["note"] = "L2-resident, latency-bound case: no roofline claim"
        line["roofline"]["achieved"] = line["roofline"]["frac"] = None
    if not full:
        return line

    # the same step as three launches (append, split, combine), for comparison
    n_unf = min(args.steps, 1000)
    for i in range(3):
        unfused_step(i)
    line["unfused"] = {"us_per_step": round(gpu.loop_s(unfused_step, n_unf) * 1e6, 2),
                       "launches_per_step": 3, "calls_per_step": 3, "steps": n_unf,
                       "path": "kvq8_quantize_append + kvq8_decode_split + kvq8_decode_combine"}

    # end to end: pinned host inputs in, result out, through the public calls
    e2e_steps = args.e2e_steps or min(args.steps, 2000)
    q_h = torch.from_numpy(wl.queries(cfg)).pin_memory()
    nk_h, nv_h = torch.from_numpy(new_k).pin_memory(), torch.from_numpy(new_v).pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    nk1_h, nv1_h = nk_h[:, 0], nv_h[:, 0]
    # a serving loop binds its buffers once (kvq8.DecodeStep) and makes one C
    # call per step; page-locked host buffers are read and written by the
    # kernels directly
    runners = [kvq8.DecodeStep(q_d, nk1, nv1, caches[j], table_d, lens_d, out, ws, sm_scale=sm,
                               dev_status=status, stream=stream, q_host=q_h, k_host=nk1_h, v_host=nv1_h,
                               out_host=out_h, cache_ready=ready) for j in range(copies)]

    def e2e_step(i):
        # host Q and the step's token in, the step, the result out; then the
        # host waits for it
        runners[i % copies].run_host()
        stream.synchronize()

    def e2e_checked_step(i):
        # the same through the per-call checked entry point
        kvq8.decode_step_host(q_h, nk1_h, nv1_h, out_h, q_d, nk1, nv1, caches[i % copies], table_d, lens_d,
                              out, ws, sm_scale=sm, stream=stream)
        stream.synchronize()

    def host_loop(fn, n):
        for i in range(3):
            fn(i)
        barrier()
        t0 = time.perf_counter()
        for i in range(n):
            fn(i)
        return time.perf_counter() - t0

    e2e_s = host_loop(e2e_step, e2e_steps)
    e2e_checked_s = host_loop(e2e_checked_step, e2e_steps)
    e_total, e_slowest = aggregate(sbytes * e2e_steps, e2e_s, dev)
    _, e_checked_slowest = aggregate(sbytes * e2e_steps, e2e_checked_s, dev)
    gpu.check_status("in the end-to-end steps")
    line["e2e"] = {"value": round(e_total / e_slowest / 1e9, 2), "unit": "GB/s",
                   "h2d_bytes_per_step": (q_h.numel() + nk_h.numel() + nv_h.numel()) * 4,
                   "d2h_bytes_per_step": out_h.numel() * 4,
                   "us_per_step": round(e_slowest / e2e_steps * 1e6, 2), "steps": e2e_steps,
                   "path": ("kvq8.DecodeStep.run_host: one C call on buffers bound once; "
                            + ("the kernels read Q and the new token from page-locked host memory and "
                               "write the result there" if runners[0].host_direct else
                               "copies through the device buffers")),
                   "checked_call_us_per_step": round(e_checked_slowest / e2e_steps * 1e6, 2)}
    if cf is not None:
        line["fp32_kv_comparator"] = f32_comparator(gpu, cfg, lens, cf, q_d, table_d, lens_d, ws, out,
                                                    roof["us_per_launch"] * 1e-6)
    if cfg.layers > 1 and cfg.batch == cfg.layers:
        line["per_layer_graph"] = per_layer_graph(gpu, cfg, sbytes, caches[0], q_d, nk1, nv1, table_d,
                                                  lens_d, out, sm, max_blocks)
    return line


def per_layer_graph(gpu, cfg, sbytes, cache, q_d, nk1, nv1, table_d, lens_d, out_folded, sm, max_blocks):
    """The same step as cfg.layers separate kvq8_decode_step calls, one per
    layer (batch 1 each, its own workspace), captured once in a CUDA graph and
    replayed: the launch form of an engine that runs one layer at a time.  One
    replay streams every layer's cache (the sum is far above L2), so replays
    read from HBM like the folded step.  Timed with KVQ8_STEP_CACHE_READY (each
    layer's call follows the previous layer's merge, which writes only its
    output) and without it."""
    import torch
    from int8_quantized_kv_gb300 import kvq8
    dev = q_d.device
    n_layers = cfg.batch
    outs = torch.empty_like(q_d)
    wss = [kvq8.alloc_workspace(1, cfg.nqh, cfg.nkv, max_blocks, dev) for _ in range(n_layers)]
    s = torch.cuda.Stream(dev)
    n = max(20, min(gpu.args.steps, 500))

    def timed(ready):
        def calls():
            for b in range(n_layers):
                kvq8.decode_step(q_d[b:b + 1], nk1[b:b + 1], nv1[b:b + 1], cache, table_d[b:b + 1],
                                 lens_d[b:b + 1], outs[b:b + 1], wss[b], sm_scale=sm, dev_status=gpu.status,
                                 stream=s, cache_ready=ready)

        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            calls()                       # once outside the graph
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            calls()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = gpu.event(), gpu.event()
        gpu.hold()
        e0.record()
        for _ in range(n):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        gpu.check_status("in the per-layer calls")
        return e0.elapsed_time(e1) / 1e3 / n

    t_plain = timed(False)
    t = timed(True)
    d = (outs.double() - out_folded.double()).abs()
    return {"us_per_step": round(t * 1e6, 2), "value": round(sbytes / t / 1e9, 2), "unit": "GB/s",
            "calls_per_step": n_layers, "launches_per_step": 2 * n_layers, "replays": n,
            "path": (f"{n_layers} kvq8_decode_step_ex calls (one layer each, KVQ8_STEP_CACHE_READY) in one "
                     "CUDA graph"),
            "plain_us_per_step": round(t_plain * 1e6, 2),
            "plain_path": "the same calls without flags",
            "max_abs_diff_vs_folded": float(d.max())}


def f32_comparator(gpu, cfg, lens, cf, q_d, table_d, lens_d, ws, out_q8, split_s):
    """The fp32-KV decode over the same context (the unquantised arm of the
    fp32-KV vs q8-KV comparison): its time and bandwidth beside the q8 split
    kernel's, and the per-dimension output delta between the two."""
    import torch
    from int8_quantized_kv_gb300 import kvq8
    sm = 1.0 / math.sqrt(cfg.hd)
    out = torch.empty_like(q_d)

    def run(i):
        kvq8.decode_attnf32(q_d, cf, table_d, lens_d, out, ws, sm_scale=sm, dev_status=gpu.status,
                            stream=gpu.stream)

    for i in range(3):
        run(i)
    t = gpu.loop_s(run, max(20, min(gpu.args.steps, 500)))
    gpu.check_status("in the fp32 decode")
    nbytes = f32_decode_bytes(cfg, lens)
    d = (out_q8.double() - out.double()).abs()
    return {"path": "kvf32_decode_attn (split + combine)", "us_per_decode": round(t * 1e6, 2),
            "GB_per_s": round(nbytes / t / 1e9, 2), "bytes_per_decode": nbytes,
            "kv_bytes_ratio_q8_over_f32": round(split_kernel_bytes(cfg, lens) / nbytes, 4),
            "time_ratio_q8_split_over_f32": round(split_s / t, 4),
            "cache_l2": "one fp32 cache copy; working set >> 129 MB L2 for this workload",
            "delta_q8_vs_f32": {"max_abs": float(d.max()), "mean_abs": float(d.mean())}}


# ------------------------------------------------------------ 4-bit cache ---
def int4_step_bytes(cfg, lens):
    """Algorithmic bytes of one 4-bit step: 64 code bytes + 4 fp32 per (token,
    kv head) for K and V, the fp32 query and output, and the one-token append
    (fp32 rows in, codes and parameters out)."""
    import numpy as np
    tok = int(np.asarray(lens, np.int64).sum())
    rows = cfg.batch * cfg.nkv
    return (tok * cfg.nkv * 2 * (cfg.hd // 2 + 16) + 2 * cfg.batch * cfg.nqh * cfg.hd * 4 +
            rows * 2 * (cfg.hd * 4 + cfg.hd // 2 + 16))


def bench_q4(gpu, cfg, full):
    """The 4-bit (asymmetric INT4 group-64) cache: a step appends one token per
    (sequence, kv head) and decodes with the fp32 query over the dequantised cache."""
    import numpy as np
    import torch
    from int8_quantized_kv_gb300 import kvq8
    from int8_quantized_kv_gb300 import workloads as wl
    args, dev, stream, status = gpu.args, gpu.dev, gpu.stream, gpu.status
    lens = wl.ctx_lens(cfg)
    table, num_blocks = wl.block_table(cfg, lens)
    max_blocks = table.shape[1]
    cache_bytes = num_blocks * 256 * cfg.nkv * 2 * (cfg.hd // 2 + 16)
    copies = args.copies or max(2, math.ceil(8 * L2_BYTES / cache_bytes))
    sm = 1.0 / math.sqrt(cfg.hd)
    c0 = kvq8.alloc_cache4(num_blocks, cfg.nkv, dev)
    table_d = torch.from_numpy(table).to(dev)
    new_k = np.zeros((cfg.batch, 1, cfg.nkv, cfg.hd), np.float32)
    new_v = np.zeros_like(new_k)
    zero = torch.zeros(1, dtype=torch.int32, device=dev)
    for b in range(cfg.batch):
        L = int(lens[b])
        k, v = wl.seq_kv(cfg, b, L)
        new_k[b, 0], new_v[b, 0] = k[L - 1], v[L - 1]
        if L > 1:
            kvq8.quantize_append4(torch.from_numpy(k[None, :L - 1]).to(dev),
                                  torch.from_numpy(v[None, :L - 1]).to(dev), zero,
                                  table_d[b:b + 1], c0)
    caches = [c0] + [kvq8.KV4Cache(*[t.clone() for t in c0]) for _ in range(copies - 1)]
    q_d = torch.from_numpy(wl.queries(cfg)).to(dev)
    # the step's token, [batch][nkv][hd] (kvq4_decode_step's layout)
    new_k, new_v = np.ascontiguousarray(new_k[:, 0]), np.ascontiguousarray(new_v[:, 0])
    nk_d, nv_d = torch.from_numpy(new_k).to(dev), torch.from_numpy(new_v).to(dev)
    lens_d = torch.from_numpy(lens).to(dev)
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, max_blocks, dev)
    out = torch.empty_like(q_d)

    def step(i, bufs=None):
        qq, kk, vv, oo = bufs or (q_d, nk_d, nv_d, out)
        # one call: the split kernel appends the token (n_new = 1) and decodes
        kvq8.decode_step4(qq, kk, vv, caches[i % copies], table_d, lens_d, oo, ws, sm_scale=sm,
                          dev_status=status, stream=stream)

    def decode(i):
        kvq8.decode_attn4(q_d, caches[i % copies], table_d, lens_d, out, ws, sm_scale=sm,
                          dev_status=status, stream=stream)

    sbytes = int4_step_bytes(cfg, lens)
    dec_bytes = sbytes - cfg.batch * cfg.nkv * 2 * (cfg.hd * 4 + cfg.hd // 2 + 16)
    per_step_s, total, slowest, roof, clocks, launches = gpu.measure(
        step, decode, "kvq4_decode_attn (int4 split + combine)", dec_bytes, sbytes, 2)
    config = {"workload": cfg.name, "batch": cfg.batch, "nqh": cfg.nqh, "nkv": cfg.nkv, "hd": cfg.hd,
              "block_size": 256, "ctx": int(lens.max()), "tokens": int(lens.sum()),
              "step": "kvq4_decode_step: the INT4 split-KV decode, which also appends the step's token "
                      "of every (sequence, kv head), + merge",
              "block_table": "seeded shuffled physical blocks",
              "l2": f"rotates {copies} cache copies; working set >> 129 MB L2, no flush",
              "parallelism": f"replicas{gpu.world}", "bytes_per_step": sbytes,
              "format": "asymmetric INT4 group-64 cache",
              "arithmetic": "fp32 query x dequantised codes, fp32 softmax and accumulation"}
    line = base_line(gpu, total / slowest / 1e9, args.steps, slowest, "int4", config)
    line["gpu_launches"] = launches
    finish_line(gpu, line, roof, clocks, line["us_per_step"], recorded_traffic("kvq4_decode_attn", cfg.name))
    if not full:
        return line

    e2e_steps = args.e2e_steps or min(args.steps, 2000)
    q_h = torch.from_numpy(wl.queries(cfg)).pin_memory()
    nk_h, nv_h = torch.from_numpy(new_k).pin_memory(), torch.from_numpy(new_v).pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    # the same public calls on the page-locked host buffers: the kernels read the
    # query and the new token there and write the result there (no copies)
    host_bufs = tuple(kvq8.HostMapped(t) for t in (q_h, nk_h, nv_h, out_h))

    def e2e_step(i):
        step(i, bufs=host_bufs)
        stream.synchronize()

    for i in range(3):
        e2e_step(i)
    barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    e2e_s = time.perf_counter() - t0
    e_total, e_slowest = aggregate(sbytes * e2e_steps, e2e_s, dev)
    line["e2e"] = {"value": round(e_total / e_slowest / 1e9, 2), "unit": "GB/s",
                   "h2d_bytes_per_step": (q_h.numel() + nk_h.numel() + nv_h.numel()) * 4,
                   "d2h_bytes_per_step": out_h.numel() * 4,
                   "us_per_step": round(e_slowest / e2e_steps * 1e6, 2), "steps": e2e_steps,
                   "path": ("kvq4_quantize_append + kvq4_decode_attn on kvq8.HostMapped page-locked "
                            "buffers: the kernels read the query and the new token and write the "
                            "result there, no copies")}
    return line


# ------------------------------------------------ mixed precision by age ---
def mixed_step_bytes(cfg, lens, n4):
    """Algorithmic bytes of one mixed decode: 160 B per (token, kv head) for the
    4-bit tokens, 264 B for the int8 tokens, the fp32 query and output."""
    import numpy as np
    lens = np.asarray(lens, np.int64)
    old = np.minimum(lens, 256 * np.asarray(n4, np.int64))
    t4, t8 = int(old.sum()), int((lens - old).sum())
    return (t4 * cfg.nkv * 2 * (cfg.hd // 2 + 16) + t8 * cfg.nkv * (2 * cfg.hd + 8) +
            2 * cfg.batch * cfg.nqh * cfg.hd * 4)


def bench_mixed(gpu, cfg, full):
    """Mixed precision by token age: every sequence's recent blocks in int8, the
    older ones requantised to 4-bit; a step is one decode over both
    (kvmix_decode_attn).  The requantisation of a block runs once per 256
    generated tokens and is not in the step."""
    import numpy as np
    import torch
    from int8_quantized_kv_gb300 import kvq8
    from int8_quantized_kv_gb300 import workloads as wl
    args, dev, stream, status = gpu.args, gpu.dev, gpu.stream, gpu.status
    lens = wl.ctx_lens(cfg)
    n4 = wl.mixed_old_blocks(lens)
    table, num_blocks = wl.block_table(cfg, lens)
    max_blocks = table.shape[1]
    table4 = np.random.default_rng(1000 * cfg.config_id + 77).permutation(num_blocks)[:table.size]
    table4 = table4.astype(np.int32).reshape(table.shape)
    cache_bytes = num_blocks * 256 * cfg.nkv * ((2 * cfg.hd + 8) + 2 * (cfg.hd // 2 + 16))
    copies = args.copies or max(2, math.ceil(8 * L2_BYTES / cache_bytes))
    sm = 1.0 / math.sqrt(cfg.hd)
    c8 = kvq8.alloc_cache(num_blocks, cfg.nkv, dev)
    c4 = kvq8.alloc_cache4(num_blocks, cfg.nkv, dev)
    table_d, table4_d = torch.from_numpy(table).to(dev), torch.from_numpy(table4).to(dev)
    zero = torch.zeros(1, dtype=torch.int32, device=dev)
    for b in range(cfg.batch):
        L = int(lens[b])
        k, v = wl.seq_kv(cfg, b, L)
        kvq8.quantize_append(torch.from_numpy(k[None]).to(dev), torch.from_numpy(v[None]).to(dev), zero,
                             table_d[b:b + 1], c8)
    n4_d = torch.from_numpy(n4).to(dev)
    kvq8.requantize_blocks(c8, table_d, c4, table4_d, torch.zeros_like(n4_d), n4_d, max(1, int(n4.max())),
                           dev_status=status)
    pairs = [(c8, c4)] + [(kvq8.KVCache(*[t.clone() for t in c8]), kvq8.KV4Cache(*[t.clone() for t in c4]))
                          for _ in range(copies - 1)]
    q_d = torch.from_numpy(wl.queries(cfg)).to(dev)
    lens_d = torch.from_numpy(lens).to(dev)
    ws = kvq8.alloc_mixed_workspace(cfg.batch, cfg.nqh, cfg.nkv, max_blocks, dev)
    out = torch.empty_like(q_d)

    def step(i, bufs=None):
        qq, oo = bufs or (q_d, out)
        a, b4 = pairs[i % copies]
        kvq8.decode_attn_mixed(qq, a, table_d, b4, table4_d, lens_d, n4_d, oo, ws, sm_scale=sm,
                               dev_status=status, stream=stream)

    sbytes = mixed_step_bytes(cfg, lens, n4)
    per_step_s, total, slowest, roof, clocks, launches = gpu.measure(
        step, step, "kvmix_decode_attn (both splits + combine)", sbytes, sbytes, 3, part_of_step=False)
    config = dict(workload_config(cfg, lens, copies, gpu.world, sbytes), old_blocks_4bit=int(n4.max()),
                  recent_blocks_int8=wl.MIXED_RECENT_BLOCKS,
                  format="old 256-token blocks INT4 group-64 (requantised from int8), recent blocks int8",
                  step="mixed decode (4-bit split + int8 split + combine); no append")
    config["arithmetic"] = ("int8 rows: int8 x int8 -> int32 block dots; 4-bit rows: fp32 query x "
                            "dequantised codes; fp32 softmax and accumulation")
    line = base_line(gpu, total / slowest / 1e9, args.steps, slowest, "int8+int4", config)
    line["gpu_launches"] = launches
    finish_line(gpu, line, roof, clocks, line["us_per_step"], recorded_traffic("kvmix_decode_attn", cfg.name))
    if not full:
        return line

    e2e_steps = args.e2e_steps or min(args.steps, 2000)
    q_h = torch.from_numpy(wl.queries(cfg)).pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    # the same public call on the page-locked host buffers (no copies)
    host_bufs = (kvq8.HostMapped(q_h), kvq8.HostMapped(out_h))

    def e2e_step(i):
        step(i, bufs=host_bufs)
        stream.synchronize()

    for i in range(3):
        e2e_step(i)
    barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    e2e_s = time.perf_counter() - t0
    e_total, e_slowest = aggregate(sbytes * e2e_steps, e2e_s, dev)
    line["e2e"] = {"value": round(e_total / e_slowest / 1e9, 2), "unit": "GB/s",
                   "h2d_bytes_per_step": q_h.numel() * 4, "d2h_bytes_per_step": out_h.numel() * 4,
                   "us_per_step": round(e_slowest / e2e_steps * 1e6, 2), "steps": e2e_steps,
                   "path": ("kvmix_decode_attn on kvq8.HostMapped page-locked buffers: the kernels read "
                            "the query and write the result there, no copies")}
    return line


# ------------------------------------------------------------- bulk append ---
def bench_append(gpu, cfg, full):
    """Quantise-append of n_new tokens per sequence (all kv heads) into the q8
    cache: 1288 algorithmic bytes per (token, kv head)."""
    import numpy as np
    import torch
    from int8_quantized_kv_gb300 import kvq8
    from int8_quantized_kv_gb300 import workloads as wl
    args, dev, stream, status = gpu.args, gpu.dev, gpu.stream, gpu.status
    n_new = int(wl.ctx_lens(cfg).max())
    lens = np.full(cfg.batch, n_new, np.int32)
    table, num_blocks = wl.block_table(cfg, lens)
    cache = kvq8.alloc_cache(num_blocks, cfg.nkv, dev)
    k = np.stack([wl.seq_kv(cfg, b, n_new)[0] for b in range(cfg.batch)])
    v = np.stack([wl.seq_kv(cfg, b, n_new)[1] for b in range(cfg.batch)])
    k_d, v_d = torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)
    start_d = torch.zeros(cfg.batch, dtype=torch.int32, device=dev)
    table_d = torch.from_numpy(table).to(dev)

    def step(i):
        kvq8.quantize_append(k_d, v_d, start_d, table_d, cache, dev_status=status, stream=stream)

    rows = cfg.batch * n_new * cfg.nkv
    sbytes = wl.algorithmic_append_bytes(rows, cfg.hd)
    per_step_s, total, slowest, roof, clocks, launches = gpu.measure(
        step, step, "quantize_append_kernel", sbytes, sbytes, 1, part_of_step=False)
    config = {"workload": cfg.name, "batch": cfg.batch, "n_new": n_new, "nkv": cfg.nkv,
              "hd": cfg.hd, "parallelism": f"replicas{gpu.world}", "bytes_per_step": sbytes,
              "l2": f"inputs {2 * k.nbytes / 2**20:.0f} MiB fp32 >> 129 MB L2, no flush",
              "step": "quantise-append of every new (token, kv head) row into the int8 cache"}
    line = base_line(gpu, total / slowest / 1e9, args.steps, slowest, "f32->int8", config)
    line["gpu_launches"] = launches
    finish_line(gpu, line, roof, clocks, line["us_per_step"],
                recorded_traffic("quantize_append_kernel", cfg.name))
    if not full:
        return line
    k_h, v_h = torch.from_numpy(k).pin_memory(), torch.from_numpy(v).pin_memory()
    e2e_steps = args.e2e_steps or min(args.steps, 50)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        # one C call: the host rows copied in and appended; then the host waits
        kvq8.quantize_append_host(k_h, v_h, k_d, v_d, start_d, table_d, cache, dev_status=status,
                                  stream=stream)
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    e_total, e_slowest = aggregate(sbytes * e2e_steps, e2e_s, dev)
    line["e2e"] = {"value": round(e_total / e_slowest / 1e9, 2), "unit": "GB/s",
                   "h2d_bytes_per_step": 2 * k.nbytes, "d2h_bytes_per_step": 0,
                   "us_per_step": round(e_slowest / e2e_steps * 1e6, 2), "steps": e2e_steps}
    return line


# ------------------------------------------------------------- dispatch ---
def runner_for(workload: str):
    if workload.startswith("int4"):
        return bench_q4
    if workload.startswith("append"):
        return bench_append
    if workload.startswith("mixed"):
        return bench_mixed
    return bench_q8


def sub_record(line: dict) -> dict:
    """The compact record of a workload in the default run's `workloads`."""
    r = line["roofline"]
    keep = ("kernel", "us_per_launch", "us_per_launch_isolated", "launches", "achieved", "frac",
            "frac_of_nominal", "us_x_sm_mhz", "traffic", "traffic_over_algorithmic", "algorithmic_bytes_per_launch",
            "note", "rejected")
    return {"us_per_step": line["us_per_step"], "GB_per_s": line["value"],
            "frac": round(line["pct_of_hbm_peak"] / 100, 4), "steps": line["steps"],
            "dtype": line["dtype"], "gpu_launches": line["gpu_launches"],
            "roofline": {k: r[k] for k in keep if k in r}, "clocks": line["clocks"],
            "config": line["config"]}


def run_gpu(args, rank, world, local):
    import torch
    from int8_quantized_kv_gb300 import workloads as wl
    gpu = Gpu(args, rank, world, local)
    cfg = wl.WORKLOADS[args.workload]
    line = runner_for(args.workload)(gpu, cfg, True)
    torch.cuda.empty_cache()
    if args.workload == DEFAULT_WORKLOAD and not args.no_workloads:
        line["workloads"] = {}
        for name in SUB_WORKLOADS:
            rec = runner_for(name)(gpu, wl.WORKLOADS[name], False)
            line["workloads"][name] = sub_record(rec)
            torch.cuda.empty_cache()
    if (rank == 0 and world == 1 and not args.no_cpu_baseline
            and runner_for(args.workload) is bench_q8):
        lens = wl.ctx_lens(cfg)
        line["cpu_baseline"] = cpu_baseline(cfg, lens, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------- reference arm ---
def run_reference(args, rank, world):
    """The CPU oracle as it stands, on the host cores, each step a bounded
    sample of the same workload (rank 0 only)."""
    if rank != 0:
        return
    import numpy as np
    from int8_quantized_kv_gb300 import workloads as wl
    if runner_for(args.workload) is not bench_q8:
        raise SystemExit("the reference arm times the q8 decode step; pick a decode workload")
    cfg = wl.WORKLOADS[args.workload]
    lens, copies, _, config = q8_decode_config(cfg, world)
    threads = len(os.sched_getaffinity(0))
    sm = np.float32(1.0 / math.sqrt(cfg.hd))
    budget = 120.0 / max(1, args.steps + args.warmup)
    units, all_units = sample_units(cfg, lens, budget, threads)
    st = OracleStep(cfg, lens, units, sm)
    for _ in range(args.warmup):
        st.run(threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        st.run(threads)
    dt = (time.perf_counter() - t0) / args.steps
    frac = sum(int(lens[b]) for b, _ in units) / sum(int(lens[b]) for b, _ in all_units)
    bytes_sample = step_bytes(cfg, lens) * frac
    value = bytes_sample / dt / 1e9
    sample = (f"{len(units)} of {len(all_units)} (sequence, kv head) units per step "
              f"({frac:.1%} of the step's tokens)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic", "config": config,
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    args = parse_args(argv)
    if args.steps < 1 or args.warmup < 0:
        raise SystemExit("--steps must be >= 1 and --warmup >= 0")
    if args.gpus < 1:
        raise SystemExit("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return self_launch(args.gpus, argv)
    rank, world, local = dist_env()
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but the launcher started {world} rank(s)")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, local)
    return 0


if __name__ == "__main__":
    sys.exit(main())
