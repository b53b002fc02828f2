"""Helpers shared by the GPU parity tests: fill the paged cache through the
C ABI from a seeded workload, read it back in logical order, and run the
oracle on the same fp32 inputs.

The CUDA side only ever sees the workload arrays; the oracle only ever sees
the same workload arrays; the two meet in the comparisons below.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle
from int8_quantized_kv_gb300 import kvq8
from int8_quantized_kv_gb300 import workloads as wl

SM_SCALE = 1.0 / math.sqrt(128.0)
ABS_TOL = 1e-4
REL_TOL = 1e-3


def k_rows_logical(kp, phys, h, slots):
    """K codes of the given (physical block, slot)s in dim order: the cache stores
    the 16-byte chunk j of a slot's row at chunk position j ^ (slot & 7)."""
    slots = np.asarray(slots)
    rows = kp[phys, h, slots, :].reshape(len(slots), 8, 16)
    pos = np.arange(8)[None, :] ^ (slots & 7)[:, None]
    return np.take_along_axis(rows, pos[:, :, None], axis=1).reshape(len(slots), 128)


def v_rows_logical(vp, phys, h, slots):
    """V codes of the given (physical block, slot)s: quarters of 64 slots, dim-major."""
    slots = np.asarray(slots)
    return vp[phys, h, slots // 64, :, slots % 64]


# Largest errors seen per test (test id -> [max |d|, max |d| / max(1, |oracle|),
# max |d| / max |oracle|], d = gpu - oracle); conftest prints them at the end
# of the session.
ERRORS = {}


def _record(*vals):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    cur = ERRORS.setdefault(test, [0.0] * len(vals))
    for i, v in enumerate(vals):
        cur[i] = max(cur[i], v)


def v4_pos(t):
    """Position of token t (0..31) of a 32-token chunk in a byte column of the
    4-bit cache's V codes: word 2*t4 + k of the column holds the tokens
    16k + 2*t4 + {0, 8, 1, 9} in its bytes 0..3."""
    t = np.asarray(t)
    k, r = t >> 4, t & 15
    return 4 * (2 * ((r & 7) >> 1) + k) + 2 * (r & 1) + (r >> 3)


def v4_token_major(vc):
    """V codes of the 4-bit cache, uint8 [num_blocks][nkv][256][64] as stored
    (per 32-token chunk [64 byte columns][32 positions]), in token-major order
    [num_blocks][nkv][256 tokens][64 bytes]."""
    nb, nkv = vc.shape[:2]
    x = vc.reshape(nb, nkv, 8, 64, 32)[..., v4_pos(np.arange(32))]
    return np.ascontiguousarray(x.transpose(0, 1, 2, 4, 3).reshape(nb, nkv, 256, 64))


def assert_close(gpu, ref, what=""):
    """Output parity bar: "within 1e-4 max-abs and 1e-3 relative" of the
    oracle, read as two bars on d = gpu - oracle:
      - |d| <= 1e-4 for every element whose oracle value is at most 1 in
        magnitude, and |d| <= 1e-4 * |oracle| above (an fp32 output of 142
        has a spacing of 1.5e-5, so no fp32 computation holds an absolute 1e-4
        there; scaled, the bar stays ten times inside the relative one);
      - max |d| <= 1e-3 * max |oracle| (relative error in the max norm; an
        element-wise ratio is undefined where the output is near 0)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    if gpu.size == 0:
        return 0.0
    err = np.abs(gpu - ref)
    scaled = err / np.maximum(1.0, np.abs(ref))
    err_max, scaled_max = float(err.max()), float(scaled.max())
    ref_max = float(np.abs(ref).max())
    rel = err_max / ref_max if ref_max > 0 else (0.0 if err_max == 0 else math.inf)
    _record(err_max, scaled_max, rel)
    if scaled_max > ABS_TOL or rel > REL_TOL:
        i = np.unravel_index(np.argmax(scaled), err.shape)
        raise AssertionError(f"{what}: max |d|/max(1,|oracle|) = {scaled_max:.3e} (bar {ABS_TOL:g}), "
                             f"max |d|/max |oracle| = {rel:.3e} (bar {REL_TOL:g}); worst at {i}: "
                             f"gpu={gpu[i]!r} oracle={ref[i]!r}")
    return err_max


class Case:
    """A workload laid out on the device: cache filled, queries uploaded."""

    def __init__(self, cfg: wl.Workload, lens=None, device="cuda", spare_blocks=3,
                 append_chunk=None):
        self.cfg = cfg
        self.lens = wl.ctx_lens(cfg) if lens is None else np.asarray(lens, np.int32)
        self.table, self.num_blocks = wl.block_table(cfg, self.lens, spare_blocks=spare_blocks)
        self.max_blocks = self.table.shape[1]
        self.device = device
        self.cache = kvq8.alloc_cache(self.num_blocks, cfg.nkv, device)
        self.table_d = torch.from_numpy(self.table).to(device)
        self.lens_d = torch.from_numpy(self.lens).to(device)
        self.q = wl.queries(cfg)
        self.q_d = torch.from_numpy(self.q).to(device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        for b in range(cfg.batch):
            self.append_sequence(b, append_chunk)
        torch.cuda.synchronize()

    def append_sequence(self, b, chunk=None):
        L = int(self.lens[b])
        if L == 0:
            return
        k, v = wl.seq_kv(self.cfg, b, L)
        chunk = L if chunk is None else chunk
        row = self.table_d[b:b + 1]
        for s in range(0, L, chunk):
            e = min(L, s + chunk)
            kd = torch.from_numpy(k[s:e][None]).to(self.device)
            vd = torch.from_numpy(v[s:e][None]).to(self.device)
            start = torch.tensor([s], dtype=torch.int32, device=self.device)
            kvq8.quantize_append(kd, vd, start, row, self.cache, dev_status=self.status)

    def decode(self, sm_scale=SM_SCALE):
        out = torch.empty_like(self.q_d)
        ws = kvq8.alloc_workspace(self.cfg.batch, self.cfg.nqh, self.cfg.nkv, self.max_blocks,
                                  self.device)
        kvq8.decode_attn(self.q_d, self.cache, self.table_d, self.lens_d, out, ws,
                         sm_scale=sm_scale, dev_status=self.status)
        torch.cuda.synchronize()
        return out.cpu().numpy()

    def status_bits(self) -> int:
        return int(self.status.item())

    # -- reading the cache back in logical order ------------------------------
    def host_pools(self):
        c = self.cache
        return (c.k_pool.cpu().numpy(), c.v_pool.cpu().numpy(),
                c.k_scale.cpu().numpy(), c.v_scale.cpu().numpy())

    def gather_unit(self, pools, b, h):
        """(kq [L][128], ks [L], vq [L][128], vs [L]) of sequence b, kv head h."""
        kp, vp, ksp, vsp = pools
        L = int(self.lens[b])
        t = np.arange(L)
        phys = self.table[b, t // wl.BLOCK_TOKENS]
        slot = t % wl.BLOCK_TOKENS
        kq = k_rows_logical(kp, phys, h, slot)
        vq = v_rows_logical(vp, phys, h, slot)
        return kq, ksp[phys, h, slot], vq, vsp[phys, h, slot]

    # -- the oracle on the same inputs ------------------------------------------
    def oracle_unit(self, b, h, sm_scale=SM_SCALE):
        cfg = self.cfg
        G = cfg.group
        L = int(self.lens[b])
        k, v = wl.unit_kv(cfg, b, h, L)
        out, _ = oracle.decode_unit_q8(self.q[b, h * G:(h + 1) * G], k, v, sm_scale)
        return out


class StepCase(Case):
    """The cache holds the first L-1 tokens of every sequence; a decode step
    appends token L-1 (k_new, v_new) and attends over all L."""

    def __init__(self, cfg: wl.Workload, lens=None, device="cuda", spare_blocks=3):
        self._full = {}
        super().__init__(cfg, lens=lens, device=device, spare_blocks=spare_blocks)
        kn = np.zeros((cfg.batch, cfg.nkv, cfg.hd), np.float32)
        vn = np.zeros_like(kn)
        for b in range(cfg.batch):
            if b in self._full:
                kn[b], vn[b] = self._full[b][0][-1], self._full[b][1][-1]
        self.k_new, self.v_new = kn, vn
        self.k_new_d = torch.from_numpy(kn).to(device)
        self.v_new_d = torch.from_numpy(vn).to(device)

    def append_sequence(self, b, chunk=None):
        L = int(self.lens[b])
        if L == 0:
            return
        k, v = wl.seq_kv(self.cfg, b, L)
        self._full[b] = (k, v)
        if L > 1:
            kvq8.quantize_append(torch.from_numpy(k[None, :L - 1]).to(self.device),
                                 torch.from_numpy(v[None, :L - 1]).to(self.device),
                                 torch.zeros(1, dtype=torch.int32, device=self.device),
                                 self.table_d[b:b + 1], self.cache, dev_status=self.status)

    def step(self, workspace=None, sm_scale=SM_SCALE):
        out = torch.full_like(self.q_d, float("nan"))
        ws = workspace if workspace is not None else kvq8.alloc_workspace(
            self.cfg.batch, self.cfg.nqh, self.cfg.nkv, self.max_blocks, self.device)
        kvq8.decode_step(self.q_d, self.k_new_d, self.v_new_d, self.cache, self.table_d,
                         self.lens_d, out, ws, sm_scale=sm_scale, dev_status=self.status)
        torch.cuda.synchronize()
        return out.cpu().numpy()
