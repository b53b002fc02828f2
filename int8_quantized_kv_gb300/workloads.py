"""Seeded synthetic workloads for INT8-KV decode attention.

This module only draws numbers: it holds none of the quantisation or
attention arithmetic, and it imports neither the CUDA binding nor the oracle.
Both sides (the CUDA path and the CPU oracle) read the same arrays from here.

Every array is drawn on the host with numpy's PCG64, seeded through a
SeedSequence whose entropy is (1000 * config_id + stream, *indices); a
unit's K/V rows (one sequence x one kv head) come from their own stream, so
any unit can be regenerated alone (the oracle checks sampled units of the
full-size workloads that way).

Streams: 0 = K/V of a unit, 1 = queries of a sequence, 2 = block-table
permutation, 3 = per-sequence context lengths, 4 = outlier channel choice,
5 = tokens appended by a decode step, 6 = rows a whole batch appends in one
call.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

HEAD_DIM = 128
BLOCK_TOKENS = 256


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode workload.

    name:        short identifier
    config_id:   seed namespace
    batch:       sequences (decode layers of one model are folded into it)
    nqh, nkv:    query heads and kv heads per sequence (GQA group nqh/nkv)
    ctx:         context length of every sequence, or None when ragged
    ctx_range:   (lo, hi) inclusive uniform range of ragged context lengths
    outlier_channels: channels per kv head drawn heavy-tailed (0 = none)
    outlier_df, outlier_scale: Student-t degrees of freedom and multiplier
    layers:      how many decode layers `batch` folds (reporting only)
    """
    name: str
    config_id: int
    batch: int
    nqh: int
    nkv: int
    ctx: Optional[int] = None
    ctx_range: Optional[tuple] = None
    outlier_channels: int = 0
    outlier_df: float = 3.0
    outlier_scale: float = 10.0
    layers: int = 1
    hd: int = HEAD_DIM

    @property
    def group(self) -> int:
        return self.nqh // self.nkv


def _rng(cfg: Workload, stream: int, *idx: int) -> np.random.Generator:
    ss = np.random.SeedSequence([1000 * cfg.config_id + stream, *[int(i) for i in idx]])
    return np.random.Generator(np.random.PCG64(ss))


def ctx_lens(cfg: Workload) -> np.ndarray:
    """Per-sequence context lengths (int32 [batch])."""
    if cfg.ctx is not None:
        return np.full(cfg.batch, cfg.ctx, np.int32)
    lo, hi = cfg.ctx_range
    return _rng(cfg, 3).integers(lo, hi + 1, size=cfg.batch).astype(np.int32)


def blocks_needed(lens: np.ndarray) -> np.ndarray:
    return (np.asarray(lens, np.int64) + BLOCK_TOKENS - 1) // BLOCK_TOKENS


def block_table(cfg: Workload, lens: Optional[np.ndarray] = None, spare_blocks: int = 0):
    """Shuffled physical block ids: (table int32 [batch][max_blocks], num_blocks).

    Logical block j of sequence b maps to a physical block drawn from a seeded
    permutation of the pool, so neighbouring logical blocks are scattered.
    Entries past a sequence's last block are -1.
    """
    lens = ctx_lens(cfg) if lens is None else lens
    need = blocks_needed(lens)
    total = int(need.sum())
    num_blocks = total + spare_blocks
    perm = _rng(cfg, 2).permutation(num_blocks).astype(np.int32)
    max_blocks = max(int(need.max()) if len(need) else 1, 1)
    table = np.full((cfg.batch, max_blocks), -1, np.int32)
    k = 0
    for b in range(cfg.batch):
        n = int(need[b])
        table[b, :n] = perm[k:k + n]
        k += n
    return table, num_blocks


def _outlier_channels(cfg: Workload, h: int) -> np.ndarray:
    return np.sort(_rng(cfg, 4, h).choice(cfg.hd, cfg.outlier_channels, replace=False))


def _draw_rows(cfg: Workload, rng: np.random.Generator, n: int, h: int) -> np.ndarray:
    x = rng.standard_normal((n, cfg.hd), dtype=np.float32)
    if cfg.outlier_channels:
        ch = _outlier_channels(cfg, h)
        x[:, ch] = (rng.standard_t(cfg.outlier_df, size=(n, len(ch))) *
                    cfg.outlier_scale).astype(np.float32)
    return x


def unit_kv(cfg: Workload, b: int, h: int, L: Optional[int] = None):
    """fp32 K and V rows [L][hd] of sequence b, kv head h (its whole context)."""
    L = int(ctx_lens(cfg)[b]) if L is None else L
    rng = _rng(cfg, 0, b, h)
    k = _draw_rows(cfg, rng, L, h)
    v = _draw_rows(cfg, rng, L, h)
    return k, v


def _threads(threads: Optional[int]) -> int:
    return max(1, os.cpu_count() or 1) if threads is None else max(1, threads)


def seq_kv(cfg: Workload, b: int, L: Optional[int] = None, threads: Optional[int] = None):
    """fp32 K and V of sequence b laid out [L][nkv][hd] (token-major, as appended).

    Heads are drawn on several host threads; every head has its own stream,
    so the result does not depend on the thread count."""
    L = int(ctx_lens(cfg)[b]) if L is None else L
    k = np.empty((L, cfg.nkv, cfg.hd), np.float32)
    v = np.empty((L, cfg.nkv, cfg.hd), np.float32)

    def one(h):
        k[:, h], v[:, h] = unit_kv(cfg, b, h, L)

    n = min(_threads(threads), cfg.nkv)
    if n == 1:
        for h in range(cfg.nkv):
            one(h)
    else:
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(one, range(cfg.nkv)))
    return k, v


def batch_new_kv(cfg: Workload, n_new: int):
    """fp32 K and V [batch][n_new][nkv][hd] from one stream: the rows that every
    sequence of a batch appends in one call (cheap to draw for large batches)."""
    rng = _rng(cfg, 6, n_new)
    shape = (cfg.batch, n_new, cfg.nkv, cfg.hd)
    return (rng.standard_normal(shape, dtype=np.float32),
            rng.standard_normal(shape, dtype=np.float32))


def queries(cfg: Workload) -> np.ndarray:
    """fp32 queries [batch][nqh][hd]: one decode token per sequence."""
    q = np.empty((cfg.batch, cfg.nqh, cfg.hd), np.float32)
    for b in range(cfg.batch):
        q[b] = _rng(cfg, 1, b).standard_normal((cfg.nqh, cfg.hd), dtype=np.float32)
    return q


# ---------------------------------------------------------------------------
# The workloads the library is measured and checked on (sizes as specified).
# ---------------------------------------------------------------------------
SINGLE_HEAD_L256 = Workload("single_head_l256", 1, batch=1, nqh=1, nkv=1, ctx=256)
QWEN3_2B_28L_8K = Workload("qwen3_2b_28layers_ctx8192", 2, batch=28, nqh=16, nkv=8,
                           ctx=8192, layers=28)
BATCH64_RAGGED = Workload("batch64_ctx512to32768", 3, batch=64, nqh=32, nkv=8,
                          ctx_range=(512, 32768))
LONG128K_OUTLIERS = Workload("batch4_ctx131072_outliers", 4, batch=4, nqh=32, nkv=8,
                             ctx=131072, outlier_channels=4)
APPEND_8X4096 = Workload("append_batch8_4096tokens", 5, batch=8, nqh=32, nkv=8, ctx=4096)
INT4_G64_32K = Workload("int4g64_batch8_ctx32768", 6, batch=8, nqh=32, nkv=8, ctx=32768)
# Mixed precision by token age: the Qwen3-2B decode stack with the most recent
# MIXED_RECENT_BLOCKS blocks (2048 tokens) of every sequence in int8 and the
# older blocks requantised to 4-bit.
MIXED_QWEN3_8K = Workload("mixed_qwen3_2b_28layers_ctx8192", 7, batch=28, nqh=16, nkv=8,
                          ctx=8192, layers=28)
MIXED_RECENT_BLOCKS = 8


def mixed_old_blocks(lens, recent_blocks: int = MIXED_RECENT_BLOCKS) -> np.ndarray:
    """Per sequence, the leading 256-token blocks held in 4-bit (int32 [batch])."""
    nb = blocks_needed(lens)
    return np.maximum(nb - recent_blocks, 0).astype(np.int32)

def steered_unit(seed: int, L: int, G: int, shape: str, peak: float = 150.0,
                 hd: int = HEAD_DIM):
    """Queries and K/V rows of one (sequence, kv head) whose scores are steered.

    Every query head is a common unit direction c times 4 plus N(0, 0.3^2)
    noise; every K row is N(0, 1) noise plus a_t * c, so that a head's score
    of token t grows with a_t.  shape "ramp": a_t rises linearly from 0 to
    `peak` over the sequence (the running maximum of the softmax keeps
    rising, stage after stage); "spike": a_t = 0 except one token at 2L/3
    with a_t = `peak` (one late jump far above every earlier score).  V rows
    are N(0, 1).  Returns float32 q [G][hd], k [L][hd], v [L][hd].
    """
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([90_000, seed, L, G])))
    c = rng.standard_normal(hd)
    c /= np.linalg.norm(c)
    q = 4.0 * c[None, :] + 0.3 * rng.standard_normal((G, hd))
    if shape == "ramp":
        a = peak * np.arange(L) / max(L - 1, 1)
    elif shape == "spike":
        a = np.zeros(L)
        a[(2 * L) // 3] = peak
    else:
        raise ValueError(f"unknown shape {shape!r}")
    k = rng.standard_normal((L, hd)) + a[:, None] * c[None, :]
    v = rng.standard_normal((L, hd))
    return q.astype(np.float32), k.astype(np.float32), v.astype(np.float32)


WORKLOADS = {w.name: w for w in (SINGLE_HEAD_L256, QWEN3_2B_28L_8K, BATCH64_RAGGED,
                                 LONG128K_OUTLIERS, APPEND_8X4096, INT4_G64_32K,
                                 MIXED_QWEN3_8K)}


def scaled(cfg: Workload, *, name=None, batch=None, ctx=None, ctx_range=None,
           nqh=None, nkv=None) -> Workload:
    """A smaller workload with the same distributions (parity-test sizes)."""
    kw = {}
    if ctx is not None or ctx_range is not None:
        kw["ctx"] = ctx
        kw["ctx_range"] = ctx_range
    return dataclasses.replace(
        cfg, name=name or (cfg.name + "_small"),
        batch=cfg.batch if batch is None else batch,
        nqh=cfg.nqh if nqh is None else nqh,
        nkv=cfg.nkv if nkv is None else nkv, **kw)


def algorithmic_decode_bytes(cfg: Workload, lens: Optional[np.ndarray] = None) -> int:
    """Bytes one decode pass must move: int8 K+V and two fp32 scales per
    (token, kv head), plus the fp32 query and output."""
    lens = ctx_lens(cfg) if lens is None else lens
    tok = int(np.asarray(lens, np.int64).sum())
    per_tok_head = 2 * cfg.hd + 2 * 4
    return tok * cfg.nkv * per_tok_head + 2 * cfg.batch * cfg.nqh * cfg.hd * 4


def algorithmic_append_bytes(n_rows: int, hd: int = HEAD_DIM) -> int:
    """Bytes an append of n_rows (token, kv head) K rows and as many V rows moves:
    fp32 in, int8 plus one fp32 scale out, for K and V."""
    return n_rows * 2 * (hd * 4 + hd + 4)
