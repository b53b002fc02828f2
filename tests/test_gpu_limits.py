"""Decode at the size limits the library accepts, against the oracle.

* The largest batch: 65535 sequences (the grid's y limit, which the combine's
  grid uses for the batch; 65536 is rejected on the host), with context
  lengths 0..5, so most of the 65535 units are a single short stage and the
  persistent split kernel walks hundreds of units per CTA.  Decoded once as
  it stands, then as a decode step that appends one more token to every
  sequence.  Outputs are checked on a seeded sample of sequences (first and
  last included); empty sequences must give exactly 0.
* A long context: one sequence of 2^20 + 77 tokens (the 128K workloads are
  covered elsewhere), whose stages are spread over every CTA of the grid.

Bar: max |gpu - oracle| <= 1e-4 and <= 1e-3 * max |oracle| ([Day 9-2] §2
decode on the same quantised inputs, the oracle accumulating in fp64).
"""
import numpy as np
import pytest
import torch

import oracle
from int8_quantized_kv_gb300 import kvq8
from int8_quantized_kv_gb300 import workloads as wl
from kvq8_harness import SM_SCALE, Case, assert_close

pytestmark = pytest.mark.gpu
MAX_BATCH = 65535


def _sample(lens, n, seed):
    rng = np.random.default_rng(seed)
    idx = set(rng.choice(len(lens), size=n, replace=False).tolist()) | {0, len(lens) - 1}
    return sorted(idx)


def test_decode_at_the_largest_batch(gpu_lib):
    G, nkv = 2, 1
    cfg = wl.Workload("max_batch", 92, batch=MAX_BATCH, nqh=G * nkv, nkv=nkv, ctx_range=(0, 5))
    lens = wl.ctx_lens(cfg)
    assert (lens == 0).any() and (lens == 5).any()
    # one block per sequence; positions 0..5 are written below, 0..lens-1 read
    table, num_blocks = wl.block_table(cfg, np.full(MAX_BATCH, 6, np.int32))
    k, v = wl.batch_new_kv(cfg, 5)
    q = wl.queries(cfg)
    cache = kvq8.alloc_cache(num_blocks, nkv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    table_d = torch.from_numpy(table).cuda()
    start = torch.zeros(MAX_BATCH, dtype=torch.int32, device="cuda")
    kvq8.quantize_append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), start, table_d, cache,
                         dev_status=status)
    q_d = torch.from_numpy(q).cuda()
    ws = kvq8.alloc_workspace(MAX_BATCH, cfg.nqh, nkv, table.shape[1])

    # decode over lens tokens
    out = torch.full_like(q_d, float("nan"))
    kvq8.decode_attn(q_d, cache, table_d, torch.from_numpy(lens).cuda(), out, ws, sm_scale=SM_SCALE,
                     dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    out = out.cpu().numpy()
    assert np.all(out[lens == 0] == 0.0) and np.all(np.isfinite(out))
    for b in _sample(lens, 1500, 1):
        L = int(lens[b])
        if L == 0:
            continue
        ref, _ = oracle.decode_unit_q8(q[b], k[b, :L, 0], v[b, :L, 0], SM_SCALE)
        assert_close(out[b], ref, f"max batch: b={b} L={L}")

    # one decode step: every sequence appends one token at position lens and
    # attends over lens + 1 tokens
    kn, vn = wl.batch_new_kv(cfg, 1)
    lens1 = lens + 1
    out1 = torch.full_like(q_d, float("nan"))
    kvq8.decode_step(q_d, torch.from_numpy(kn[:, 0]).cuda(), torch.from_numpy(vn[:, 0]).cuda(), cache, table_d,
                     torch.from_numpy(lens1).cuda(), out1, ws, sm_scale=SM_SCALE, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    out1 = out1.cpu().numpy()
    assert np.all(np.isfinite(out1))
    for b in _sample(lens, 1500, 2):
        L = int(lens[b])
        kk = np.concatenate([k[b, :L, 0], kn[b, :, 0]])
        vv = np.concatenate([v[b, :L, 0], vn[b, :, 0]])
        ref, _ = oracle.decode_unit_q8(q[b], kk, vv, SM_SCALE)
        assert_close(out1[b], ref, f"max batch step: b={b} L={L + 1}")


def test_decode_one_context_of_a_million_tokens(gpu_lib):
    cfg = wl.Workload("long_context", 93, batch=1, nqh=4, nkv=1, ctx=(1 << 20) + 77)
    case = Case(cfg)
    out = case.decode()
    assert case.status_bits() == 0
    assert_close(out[0], case.oracle_unit(0, 0), "2^20 + 77 tokens")


@pytest.mark.parametrize("path", ["int4", "f32"])
def test_other_caches_at_the_largest_batch(gpu_lib, path):
    """The INT4 and fp32 caches' decode at 65535 sequences (their split grids
    hold the batch in z)."""
    G, nkv = 2, 1
    cfg = wl.Workload("max_batch", 92, batch=MAX_BATCH, nqh=G * nkv, nkv=nkv, ctx_range=(0, 5))
    lens = wl.ctx_lens(cfg)
    table, num_blocks = wl.block_table(cfg, np.full(MAX_BATCH, 6, np.int32))
    k, v = wl.batch_new_kv(cfg, 5)
    q = wl.queries(cfg)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    table_d = torch.from_numpy(table).cuda()
    start = torch.zeros(MAX_BATCH, dtype=torch.int32, device="cuda")
    kd, vd = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    q_d = torch.from_numpy(q).cuda()
    ws = kvq8.alloc_workspace(MAX_BATCH, cfg.nqh, nkv, table.shape[1])
    out = torch.full_like(q_d, float("nan"))
    lens_d = torch.from_numpy(lens).cuda()
    if path == "int4":
        cache = kvq8.alloc_cache4(num_blocks, nkv)
        kvq8.quantize_append4(kd, vd, start, table_d, cache, dev_status=status)
        kvq8.decode_attn4(q_d, cache, table_d, lens_d, out, ws, sm_scale=SM_SCALE, dev_status=status)
    else:
        cache = kvq8.alloc_cachef32(num_blocks, nkv)
        kvq8.appendf32(kd, vd, start, table_d, cache, dev_status=status)
        kvq8.decode_attnf32(q_d, cache, table_d, lens_d, out, ws, sm_scale=SM_SCALE, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    out = out.cpu().numpy()
    assert np.all(out[lens == 0] == 0.0) and np.all(np.isfinite(out))
    for b in _sample(lens, 1000, 3):
        L = int(lens[b])
        if L == 0:
            continue
        kk, vv = k[b, :L, 0], v[b, :L, 0]
        if path == "int4":
            kk = oracle.int4_dequantize_groups(*oracle.int4_quantize_groups(kk, 64), 64)
            vv = oracle.int4_dequantize_groups(*oracle.int4_quantize_groups(vv, 64), 64)
        ref = np.stack([oracle.attention_f64(q[b, g], kk, vv, SM_SCALE) for g in range(G)])
        assert_close(out[b], ref, f"{path} max batch: b={b} L={L}")
