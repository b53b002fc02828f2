#!/usr/bin/env python
"""Benchmark of the q8-KV decode step on GB300.

One step = the whole hot path over one batch: quantise-append of the step's
new K/V token for every (layer, kv head), split-KV decode attention of every
query head over its paged int8 context, and the split merge: one
kvq8_decode_step call (two launches: the split kernel, which also appends the
step's new token, and the merge, whose launch overlaps the split's tail
through programmatic dependent launch; the three separate entry points --
append, split, merge -- called one by one are timed beside it as `unfused`).
The default workload is the 28-layer
Qwen3-2B-shaped decode stack (16 query / 8 kv heads, hd 128, context 8192,
batch 1), its layers folded into the batch dimension of one call.

Prints one JSON line.  `value` is achieved algorithmic HBM throughput in GB/s
(bytes a step must move / device time per step) summed over ranks;
`us_per_step` and `ms_per_step` are the device time of one step.  Inputs are
resident in HBM; the timed region rotates over several copies of the cache so
that every step streams from HBM (the working set is far above L2).
`--impl reference` times the CPU oracle on the host cores instead.
Multi-GPU runs (torchrun) are independent replicas: the path needs no
exchange between GPUs.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "q8-KV decode attention: μs/step and achieved HBM GB/s (% of GB300 peak)"
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e nominal bandwidth (context beside the measured peak)
THROTTLE_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=("kvq8", "reference"), default="kvq8")
    ap.add_argument("--workload", default="qwen3_2b_28layers_ctx8192")
    ap.add_argument("--copies", type=int, default=0,
                    help="cache copies to rotate over (0 = enough to exceed 8x L2)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0 = min(steps, 2000)")
    ap.add_argument("--no-f32", action="store_true",
                    help="skip the fp32-KV decode comparator leg")
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


# ---------------------------------------------------------------- clocks ---
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.error = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError as e:
            self.error = f"nvidia-smi unavailable: {e}"

    def stop(self):
        if self.proc is None:
            return {"error": self.error or "not started"}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        for line in out.strip().splitlines():
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
        if not sm:
            return {"error": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


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


def cross_check_traffic(line):
    """The roofline's fraction of the nominal HBM bandwidth beside the measured
    one, and the traffic measured by ncu against the algorithmic bytes of the same launch:
    the ratio, and a flag when they differ by more than 5 %: above, bytes read
    more than once; below, bytes served from L2 or writes still in L2 (not yet
    written back) when the kernel ended."""
    r = line.get("roofline", {})
    if r.get("unit") == "GB/s" and r.get("achieved"):
        r["nominal_peak"] = NOMINAL_HBM_GBS
        r["frac_of_nominal"] = round(r["achieved"] / NOMINAL_HBM_GBS, 4)
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
    return line


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


def workload_config(cfg, lens, copies):
    import numpy as np
    c = {"workload": cfg.name, "layers_folded_into_batch": cfg.layers,
         "batch": cfg.batch // max(cfg.layers, 1), "nqh": cfg.nqh, "nkv": cfg.nkv, "hd": cfg.hd,
         "block_size": 256, "ctx": int(lens.max()) if cfg.ctx is not None else
         [int(lens.min()), int(lens.max())], "tokens": int(np.asarray(lens).sum()),
         "step": "append 1 token per (layer, kv head) + split-KV decode + merge",
         "block_table": "seeded shuffled physical blocks"}
    if copies:
        c["l2"] = f"rotates {copies} cache copies; working set >> 129 MB L2, no flush"
    return c


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


# ---------------------------------------------------------------- kvq8 arm ---
def run_kvq8(args, rank, world, local):
    import numpy as np
    import torch
    from int8_quantized_kv_gb300 import kvq8
    from int8_quantized_kv_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init(world, "nccl")
    kvq8.load()
    cfg = wl.WORKLOADS[args.workload]
    lens = wl.ctx_lens(cfg)
    table, num_blocks = wl.block_table(cfg, lens)
    max_blocks = table.shape[1]
    cache_bytes = 2 * kvq8.kv_pool_bytes(num_blocks, cfg.nkv) + 2 * kvq8.scale_pool_bytes(num_blocks, cfg.nkv)
    # a cache of a few hundred KB (the single-head case) stays in L2 by
    # construction: latency-bound, timed as it is, no roofline claim
    l2_resident = cache_bytes * 8 < L2_BYTES // 16
    copies = args.copies or (1 if l2_resident else max(2, math.ceil(8 * L2_BYTES / cache_bytes)))
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
    cf = None if args.no_f32 else kvq8.alloc_cachef32(num_blocks, cfg.nkv, dev)
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
    caches = [c0]
    for _ in range(copies - 1):
        caches.append(kvq8.KVCache(*[t.clone() for t in c0]))
    q_d = torch.from_numpy(wl.queries(cfg)).to(dev)
    nk_d, nv_d = torch.from_numpy(new_k).to(dev), torch.from_numpy(new_v).to(dev)
    start_d = torch.from_numpy((lens - 1).clip(min=0).astype(np.int32)).to(dev)
    lens_d = torch.from_numpy(lens).to(dev)
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, max_blocks, dev)
    out = torch.empty_like(q_d)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    nk1, nv1 = nk_d[:, 0], nv_d[:, 0]   # the step's token, [batch][nkv][hd]

    def step(i, ev=None):
        c = caches[i % copies]
        if ev is None:
            kvq8.decode_step(q_d, nk1, nv1, c, table_d, lens_d, out, ws, sm_scale=sm,
                             dev_status=status, stream=stream)
        else:
            # the step's work as three calls through their own entry points
            # (append, split, combine), with events around the split kernel
            # (the roofline's dominant kernel)
            kvq8.quantize_append(nk_d, nv_d, start_d, table_d, c, dev_status=status, stream=stream)
            ev[0].record(stream)
            kvq8.decode_split(q_d, c, table_d, lens_d, ws, sm_scale=sm, dev_status=status,
                              stream=stream)
            ev[1].record(stream)
            kvq8.decode_combine(cfg.batch, cfg.nqh, cfg.nkv, max_blocks, lens_d, ws, out,
                                stream=stream)

    def unfused_step(i):
        c = caches[i % copies]
        kvq8.quantize_append(nk_d, nv_d, start_d, table_d, c, dev_status=status, stream=stream)
        kvq8.decode_split(q_d, c, table_d, lens_d, ws, sm_scale=sm, dev_status=status, stream=stream)
        kvq8.decode_combine(cfg.batch, cfg.nqh, cfg.nkv, max_blocks, lens_d, ws, out, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item():#x} during warm-up")

    # device-timed region: K steps; every k_sample-th step runs as three calls
    # with events around the split kernel for its roofline (a recorded event
    # costs the stream about a microsecond, so not every step carries them)
    k_sample = 10
    split_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(0, args.steps, k_sample)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_start.record(stream)
    for i in range(args.steps):
        step(i, split_ev[i // k_sample] if i % k_sample == 0 else None)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    split_s = sum(a.elapsed_time(b) for a, b in split_ev) / 1e3 / len(split_ev)
    launches = 2 * args.steps + len(split_ev)   # sampled steps run three calls

    # the same step as three launches (append, split, combine), for comparison
    n_unf = min(args.steps, 1000)
    for i in range(3):
        unfused_step(i)
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    u0.record(stream)
    for i in range(n_unf):
        unfused_step(i)
    u1.record(stream)
    torch.cuda.synchronize()
    unfused_us = u0.elapsed_time(u1) * 1e3 / n_unf

    sbytes = step_bytes(cfg, lens)
    total_bytes, slowest = aggregate(sbytes * args.steps, elapsed, dev)
    per_step = slowest / args.steps
    value = total_bytes / slowest / 1e9

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
                               out_host=out_h) for j in range(copies)]

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
    h2d = (q_h.numel() + nk_h.numel() + nv_h.numel()) * 4
    d2h = out_h.numel() * 4

    if status.item() != 0:
        raise RuntimeError(f"device status {status.item():#x} in the timed region")
    comparator = None if cf is None else f32_comparator(args, cfg, lens, cf, q_d, table_d, lens_d, ws,
                                                        out, status, stream, split_s)

    peak, peak_kind = hbm_peak()
    split_bytes = split_kernel_bytes(cfg, lens)
    achieved = split_bytes / split_s / 1e9
    traffic = recorded_traffic("decode_split_kernel", cfg.name)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 5),
        "us_per_step": round(per_step * 1e6, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": dict(workload_config(cfg, lens, copies), parallelism=f"replicas{world}",
                       bytes_per_step=sbytes,
                       arithmetic="int8 x int8 -> int32 block dots, fp32 softmax and accumulation"),
        "pct_of_hbm_peak": round(100 * (value / world) / peak, 2),
        "roofline": {"bound": "hbm", "kernel": "decode_split_kernel",
                     "achieved": round(achieved, 2),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": peak_kind, "traffic": traffic,
                     "algorithmic_bytes_per_launch": split_bytes,
                     "us_per_launch": round(split_s * 1e6, 3)},
        "e2e": {"value": round(e_total / e_slowest / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": round(e_slowest / e2e_steps * 1e6, 2), "steps": e2e_steps,
                "path": ("kvq8.DecodeStep.run_host: one C call on buffers bound once; "
                         + ("the kernels read Q and the new token from page-locked host memory and "
                            "write the result there" if runners[0].host_direct else
                            "copies through the device buffers")),
                "checked_call_us_per_step": round(e_checked_slowest / e2e_steps * 1e6, 2)},
        "gpu_launches": launches,
        "unfused": {"us_per_step": round(unfused_us, 2), "launches_per_step": 3, "calls_per_step": 3,
                    "path": "kvq8_quantize_append + kvq8_decode_split + kvq8_decode_combine"},
        "clocks": clocks,
    }
    if comparator is not None:
        line["fp32_kv_comparator"] = comparator
    if l2_resident:
        line["config"]["l2"] = (f"one cache copy of {cache_bytes / 1024:.0f} KiB: L2-resident by "
                                "construction, latency-bound")
        line["roofline"]["note"] = "L2-resident, latency-bound case: no roofline claim"
    if cfg.layers > 1 and cfg.batch == cfg.layers:
        line["per_layer_graph"] = per_layer_graph(args, cfg, sbytes, caches[0], q_d, nk1, nv1, table_d,
                                                  lens_d, out, status, sm, max_blocks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, lens, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(cross_check_traffic(line)), flush=True)


def per_layer_graph(args, cfg, sbytes, cache, q_d, nk1, nv1, table_d, lens_d, out_folded, status, sm,
                    max_blocks):
    """The same step as cfg.layers separate kvq8_decode_step calls, one per
    layer (batch 1 each, its own workspace), captured once in a CUDA graph and
    replayed: the launch form of an engine that runs one layer at a time.  One
    replay streams every layer's cache (the sum is far above L2), so replays
    read from HBM like the folded step."""
    import torch
    from int8_quantized_kv_gb300 import kvq8
    dev = q_d.device
    n_layers = cfg.batch
    outs = torch.empty_like(q_d)
    wss = [kvq8.alloc_workspace(1, cfg.nqh, cfg.nkv, max_blocks, dev) for _ in range(n_layers)]
    s = torch.cuda.Stream(dev)

    def calls():
        for b in range(n_layers):
            kvq8.decode_step(q_d[b:b + 1], nk1[b:b + 1], nv1[b:b + 1], cache, table_d[b:b + 1],
                             lens_d[b:b + 1], outs[b:b + 1], wss[b], sm_scale=sm, dev_status=status,
                             stream=s)

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
    n = max(10, min(args.steps, 200))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item():#x} in the per-layer calls")
    t = e0.elapsed_time(e1) / 1e3 / n
    d = (outs.double() - out_folded.double()).abs()
    return {"us_per_step": round(t * 1e6, 2), "value": round(sbytes / t / 1e9, 2), "unit": "GB/s",
            "calls_per_step": n_layers, "launches_per_step": 2 * n_layers, "replays": n,
            "path": f"{n_layers} kvq8_decode_step calls (one layer each) in one CUDA graph",
            "max_abs_diff_vs_folded": float(d.max())}


def f32_comparator(args, cfg, lens, cf, q_d, table_d, lens_d, ws, out_q8, status, stream, split_s):
    """The fp32-KV decode over the same context (the unquantised arm of the
    fp32-KV vs q8-KV comparison): its time and bandwidth beside the q8 split
    kernel's, and the per-dimension output delta between the two."""
    import torch
    from int8_quantized_kv_gb300 import kvq8
    sm = 1.0 / math.sqrt(cfg.hd)
    out = torch.empty_like(q_d)
    n = min(args.steps, 500)

    def run():
        kvq8.decode_attnf32(q_d, cf, table_d, lens_d, out, ws, sm_scale=sm, dev_status=status,
                            stream=stream)

    for _ in range(3):
        run()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item():#x} in the fp32 decode")
    t = e0.elapsed_time(e1) / 1e3 / n
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


def run_kvq4(args, rank, world, local):
    """The 4-bit (asymmetric INT4 group-64) cache: a step appends one token per
    (sequence, kv head) and decodes with the fp32 query over the dequantised cache."""
    import numpy as np
    import torch
    from int8_quantized_kv_gb300 import kvq8
    from int8_quantized_kv_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init(world, "nccl")
    kvq8.load()
    cfg = wl.WORKLOADS[args.workload]
    lens = wl.ctx_lens(cfg)
    table, num_blocks = wl.block_table(cfg, lens)
    max_blocks = table.shape[1]
    cache_bytes = num_blocks * 256 * kvq8.cache4_bytes_per_token(cfg.nkv)
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
    nk_d, nv_d = torch.from_numpy(new_k).to(dev), torch.from_numpy(new_v).to(dev)
    start_d = torch.from_numpy((lens - 1).clip(min=0).astype(np.int32)).to(dev)
    lens_d = torch.from_numpy(lens).to(dev)
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, max_blocks, dev)
    out = torch.empty_like(q_d)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i, ev=None, bufs=None):
        qq, kk, vv, oo = bufs or (q_d, nk_d, nv_d, out)
        c = caches[i % copies]
        kvq8.quantize_append4(kk, vv, start_d, table_d, c, dev_status=status, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        kvq8.decode_attn4(qq, c, table_d, lens_d, oo, ws, sm_scale=sm, dev_status=status,
                          stream=stream)
        if ev is not None:
            ev[1].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item():#x} during warm-up")
    k_sample = 10
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(0, args.steps, k_sample)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_start.record(stream)
    for i in range(args.steps):
        step(i, evs[i // k_sample] if i % k_sample == 0 else None)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item():#x} in the timed region")
    elapsed = t_start.elapsed_time(t_end) / 1e3
    dec_s = sum(a.elapsed_time(b) for a, b in evs) / 1e3 / len(evs)
    sbytes = int4_step_bytes(cfg, lens)
    total_bytes, slowest = aggregate(sbytes * args.steps, elapsed, dev)
    per_step = slowest / args.steps
    value = total_bytes / slowest / 1e9

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
    peak, peak_kind = hbm_peak()
    dec_bytes = sbytes - cfg.batch * cfg.nkv * 2 * (cfg.hd * 4 + cfg.hd // 2 + 16)
    achieved = dec_bytes / dec_s / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 5),
        "us_per_step": round(per_step * 1e6, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4", "data": "synthetic",
        "config": dict(workload_config(cfg, lens, copies), parallelism=f"replicas{world}",
                       bytes_per_step=sbytes, format="asymmetric INT4 group-64 cache",
                       arithmetic="fp32 query x dequantised codes, fp32 softmax and accumulation"),
        "pct_of_hbm_peak": round(100 * (value / world) / peak, 2),
        "roofline": {"bound": "hbm", "kernel": "kvq4_decode_attn (int4 split + combine)",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": recorded_traffic("kvq4_decode_attn", cfg.name),
                     "algorithmic_bytes_per_launch": dec_bytes, "us_per_launch": round(dec_s * 1e6, 3)},
        "e2e": {"value": round(e_total / e_slowest / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": (q_h.numel() + nk_h.numel() + nv_h.numel()) * 4,
                "d2h_bytes_per_step": out_h.numel() * 4,
                "us_per_step": round(e_slowest / e2e_steps * 1e6, 2), "steps": e2e_steps,
                "path": "kvq4_quantize_append + kvq4_decode_attn on kvq8.HostMapped page-locked buffers: the kernels read the query and the new token and write the result there, no copies"},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(cross_check_traffic(line)), flush=True)


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


def run_mixed(args, rank, world, local):
    """Mixed precision by token age: every sequence's recent blocks in int8, the
    older ones requantised to 4-bit; a step is one decode over both
    (kvmix_decode_attn: 4-bit split, int8 split, one combine).  The
    requantisation of a block runs once per 256 generated tokens and is not in
    the step."""
    import numpy as np
    import torch
    from int8_quantized_kv_gb300 import kvq8
    from int8_quantized_kv_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init(world, "nccl")
    kvq8.load()
    cfg = wl.WORKLOADS[args.workload]
    lens = wl.ctx_lens(cfg)
    n4 = wl.mixed_old_blocks(lens)
    table, num_blocks = wl.block_table(cfg, lens)
    max_blocks = table.shape[1]
    table4 = np.random.default_rng(1000 * cfg.config_id + 77).permutation(num_blocks)[:table.size]
    table4 = table4.astype(np.int32).reshape(table.shape)
    cache_bytes = num_blocks * 256 * (kvq8.cache_bytes_per_token(cfg.nkv) + kvq8.cache4_bytes_per_token(cfg.nkv))
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
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kvq8.requantize_blocks(c8, table_d, c4, table4_d, torch.zeros_like(n4_d), n4_d, max(1, int(n4.max())),
                           dev_status=status)
    pairs = [(c8, c4)] + [(kvq8.KVCache(*[t.clone() for t in c8]), kvq8.KV4Cache(*[t.clone() for t in c4]))
                          for _ in range(copies - 1)]
    q_d = torch.from_numpy(wl.queries(cfg)).to(dev)
    lens_d = torch.from_numpy(lens).to(dev)
    ws = kvq8.alloc_mixed_workspace(cfg.batch, cfg.nqh, cfg.nkv, max_blocks, dev)
    out = torch.empty_like(q_d)
    stream = torch.cuda.current_stream(dev)

    def step(i, bufs=None):
        qq, oo = bufs or (q_d, out)
        a, b4 = pairs[i % copies]
        kvq8.decode_attn_mixed(qq, a, table_d, b4, table4_d, lens_d, n4_d, oo, ws, sm_scale=sm,
                               dev_status=status, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item():#x} during warm-up")
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_start.record(stream)
    for i in range(args.steps):
        step(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item():#x} in the timed region")
    elapsed = t_start.elapsed_time(t_end) / 1e3
    sbytes = mixed_step_bytes(cfg, lens, n4)
    total_bytes, slowest = aggregate(sbytes * args.steps, elapsed, dev)
    per_step = slowest / args.steps
    value = total_bytes / slowest / 1e9

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
    peak, peak_kind = hbm_peak()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 5),
        "us_per_step": round(per_step * 1e6, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8+int4", "data": "synthetic",
        "config": dict(workload_config(cfg, lens, copies), parallelism=f"replicas{world}",
                       bytes_per_step=sbytes, old_blocks_4bit=int(n4.max()),
                       recent_blocks_int8=wl.MIXED_RECENT_BLOCKS,
                       format="old 256-token blocks INT4 group-64 (requantised from int8), recent blocks int8",
                       step="mixed decode (4-bit split + int8 split + combine); no append"),
        "pct_of_hbm_peak": round(100 * (value / world) / peak, 2),
        "roofline": {"bound": "hbm", "kernel": "kvmix_decode_attn (both splits + combine)",
                     "achieved": round(value / world, 2), "peak": peak, "unit": "GB/s",
                     "frac": round((value / world) / peak, 4), "peak_kind": peak_kind,
                     "traffic": recorded_traffic("kvmix_decode_attn", cfg.name),
                     "algorithmic_bytes_per_launch": sbytes, "us_per_launch": round(per_step * 1e6, 3)},
        "e2e": {"value": round(e_total / e_slowest / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": q_h.numel() * 4, "d2h_bytes_per_step": out_h.numel() * 4,
                "us_per_step": round(e_slowest / e2e_steps * 1e6, 2), "steps": e2e_steps,
                "path": "kvmix_decode_attn on kvq8.HostMapped page-locked buffers: the kernels read the query and write the result there, no copies"},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(cross_check_traffic(line)), flush=True)


# ------------------------------------------------------------- bulk append ---
def run_append(args, rank, world, local):
    """Quantise-append of n_new tokens per sequence (all kv heads) into the q8
    cache: 1288 algorithmic bytes per (token, kv head)."""
    import numpy as np
    import torch
    from int8_quantized_kv_gb300 import kvq8
    from int8_quantized_kv_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init(world, "nccl")
    kvq8.load()
    cfg = wl.WORKLOADS[args.workload]
    n_new = int(wl.ctx_lens(cfg).max())
    lens = np.full(cfg.batch, n_new, np.int32)
    table, num_blocks = wl.block_table(cfg, lens)
    cache = kvq8.alloc_cache(num_blocks, cfg.nkv, dev)
    k = np.stack([wl.seq_kv(cfg, b, n_new)[0] for b in range(cfg.batch)])
    v = np.stack([wl.seq_kv(cfg, b, n_new)[1] for b in range(cfg.batch)])
    k_d, v_d = torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)
    start_d = torch.zeros(cfg.batch, dtype=torch.int32, device=dev)
    table_d = torch.from_numpy(table).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kvq8.quantize_append(k_d, v_d, start_d, table_d, cache, dev_status=status, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_start.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item():#x}")
    elapsed = t_start.elapsed_time(t_end) / 1e3
    rows = cfg.batch * n_new * cfg.nkv
    sbytes = wl.algorithmic_append_bytes(rows, cfg.hd)
    total_bytes, slowest = aggregate(sbytes * args.steps, elapsed, dev)
    per_step = slowest / args.steps
    value = total_bytes / slowest / 1e9
    peak, peak_kind = hbm_peak()
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
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 5),
        "us_per_step": round(per_step * 1e6, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32->int8", "data": "synthetic",
        "config": {"workload": cfg.name, "batch": cfg.batch, "n_new": n_new, "nkv": cfg.nkv,
                   "hd": cfg.hd, "parallelism": f"replicas{world}", "bytes_per_step": sbytes,
                   "l2": f"inputs {2 * k.nbytes / 2**20:.0f} MiB fp32 >> 129 MB L2, no flush"},
        "pct_of_hbm_peak": round(100 * (value / world) / peak, 2),
        "roofline": {"bound": "hbm", "kernel": "quantize_append_kernel", "achieved": round(value / world, 2),
                     "peak": peak, "unit": "GB/s", "frac": round(value / world / peak, 4),
                     "peak_kind": peak_kind, "traffic": recorded_traffic("quantize_append_kernel", cfg.name),
                     "algorithmic_bytes_per_launch": sbytes,
                     "us_per_launch": round(per_step * 1e6, 3)},
        "e2e": {"value": round(e_total / e_slowest / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": 2 * k.nbytes, "d2h_bytes_per_step": 0,
                "us_per_step": round(e_slowest / e2e_steps * 1e6, 2), "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(cross_check_traffic(line)), flush=True)


# ----------------------------------------------------------- reference arm ---
def run_reference(args, rank, world):
    """The CPU oracle as it stands, on the host cores, each step a bounded
    sample of the same workload (rank 0 only)."""
    if rank != 0:
        return
    import numpy as np
    from int8_quantized_kv_gb300 import workloads as wl
    if args.workload.startswith(("int4", "append", "mixed")):
        raise SystemExit("the reference arm times the q8 decode step; pick a decode workload")
    cfg = wl.WORKLOADS[args.workload]
    lens = wl.ctx_lens(cfg)
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
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": dict(workload_config(cfg, lens, 0), parallelism="host cores"),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.steps < 1 or args.warmup < 0:
        raise SystemExit("--steps must be >= 1")
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.workload.startswith("int4"):
        run_kvq4(args, rank, world, local)
    elif args.workload.startswith("append"):
        run_append(args, rank, world, local)
    elif args.workload.startswith("mixed"):
        run_mixed(args, rank, world, local)
    else:
        run_kvq8(args, rank, world, local)


if __name__ == "__main__":
    main()
