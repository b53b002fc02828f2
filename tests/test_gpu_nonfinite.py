"""Non-finite inputs on the GPU path against the oracle.

The pages give their quantisation rules for finite values only.  The reading
taken (include/kvq8.h, "Non-finite inputs"): a unit of quantisation -- a K/V
row of the int8 cache, a 64-value group of the 4-bit cache, a 32-value block
of the query in the int8 decode -- holding a NaN or an infinity is quantised
as if all its values were zero, and KVQ8_DEV_NONFINITE is set in the status
word.  The oracle implements the same reading; payloads and scales must match
it bit for bit, outputs within the parity bar, and every output stays finite.
"""
import numpy as np
import pytest
import torch

import oracle
from int8_quantized_kv_gb300 import kvq8
from int8_quantized_kv_gb300 import workloads as wl
from kvq8_harness import SM_SCALE, Case, StepCase, assert_close, k_rows_logical, v4_token_major, v_rows_logical

pytestmark = pytest.mark.gpu
HD = 128


def _plant(x, seed, n_rows):
    """NaN, +inf and -inf planted in n_rows random rows of x [..., hd] (in place);
    returns the flat indices of the rows hit."""
    rng = np.random.default_rng(seed)
    flat = x.reshape(-1, x.shape[-1])
    rows = rng.choice(flat.shape[0], n_rows, replace=False)
    for j, r in enumerate(rows):
        flat[r, rng.integers(x.shape[-1])] = (np.nan, np.inf, -np.inf)[j % 3]
    return rows


@pytest.mark.parametrize("start,n_new", [(0, 1), (5, 1), (0, 64), (37, 200)])
def test_append_nonfinite_rows_bit_exact(gpu_lib, start, n_new):
    # whole 16-token runs and partial runs of the bulk kernel, and the
    # one-token kernel; rows hit in K and in V independently
    nkv, batch = 2, 2
    rng = np.random.default_rng(100 + start + n_new)
    k = rng.standard_normal((batch, n_new, nkv, HD)).astype(np.float32)
    v = rng.standard_normal((batch, n_new, nkv, HD)).astype(np.float32)
    nk = _plant(k, 1 + n_new, max(1, min(6, batch * n_new * nkv // 3)))
    _plant(v, 2 + n_new, max(1, min(6, batch * n_new * nkv // 3)))
    need = (start + n_new + 255) // 256
    num_blocks = batch * need + 1
    table = np.random.default_rng(7).permutation(num_blocks)[:batch * need].astype(np.int32).reshape(batch, need)
    cache = kvq8.alloc_cache(num_blocks, nkv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq8.quantize_append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                         torch.full((batch,), start, dtype=torch.int32, device="cuda"),
                         torch.from_numpy(table).cuda(), cache, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == kvq8.DEV_NONFINITE and len(nk) > 0
    kp, vp = cache.k_pool.cpu().numpy(), cache.v_pool.cpu().numpy()
    ksp, vsp = cache.k_scale.cpu().numpy(), cache.v_scale.cpu().numpy()
    pos = start + np.arange(n_new)
    replaced = 0
    for b in range(batch):
        phys, slot = table[b, pos // 256], pos % 256
        for h in range(nkv):
            kq, ks, nk_ = oracle.kv_quantize_rows(k[b, :, h], count_nonfinite=True)
            vq, vs, nv_ = oracle.kv_quantize_rows(v[b, :, h], count_nonfinite=True)
            replaced += nk_ + nv_
            assert np.array_equal(k_rows_logical(kp, phys, h, slot), kq)
            assert np.array_equal(v_rows_logical(vp, phys, h, slot), vq)
            assert np.array_equal(ksp[phys, h, slot].view(np.uint32), ks.view(np.uint32))
            assert np.array_equal(vsp[phys, h, slot].view(np.uint32), vs.view(np.uint32))
    assert replaced > 0


def test_finite_rows_leave_the_flag_clear(gpu_lib):
    # the largest finite values and subnormals are finite: no flag
    k = np.zeros((1, 3, 1, HD), np.float32)
    k[0, 0, 0, 0] = np.finfo(np.float32).max
    k[0, 1, 0, 5] = -np.finfo(np.float32).max
    k[0, 2, 0, :] = np.float32(1e-45)
    cache = kvq8.alloc_cache(1, 1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq8.quantize_append(torch.from_numpy(k).cuda(), torch.from_numpy(k).cuda(),
                         torch.zeros(1, dtype=torch.int32, device="cuda"),
                         torch.zeros((1, 1), dtype=torch.int32, device="cuda"), cache, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    kq, ks = oracle.kv_quantize_rows(k[0, :, 0])
    assert np.array_equal(cache.k_scale.cpu().numpy()[0, 0, :3].view(np.uint32), ks.view(np.uint32))
    assert np.array_equal(k_rows_logical(cache.k_pool.cpu().numpy(), np.zeros(3, int), 0, np.arange(3)), kq)


def test_decode_with_nonfinite_query_blocks(gpu_lib):
    # a NaN / inf in some query 32-blocks: those blocks count as zero blocks in
    # every CTA that quantises the unit's query; the output stays finite and
    # matches the oracle, and the status word carries only the non-finite bit
    cfg = wl.Workload("nonfinite_q", 910, batch=3, nqh=8, nkv=2, ctx_range=(100, 2500))
    case = Case(cfg)
    q = case.q.copy()
    q[0, 1, 3] = np.nan
    q[1, 4, 100] = np.inf
    q[2, 7, 64] = -np.inf
    q[2, 7, 65] = np.nan
    case.q = q
    case.q_d = torch.from_numpy(q).cuda()
    case.status.zero_()
    out = case.decode()
    assert case.status_bits() == kvq8.DEV_NONFINITE
    assert np.all(np.isfinite(out))
    G = cfg.group
    for b in range(cfg.batch):
        for h in range(cfg.nkv):
            assert_close(out[b, h * G:(h + 1) * G], case.oracle_unit(b, h), f"nonfinite q b={b} h={h}")


@pytest.mark.parametrize("val", [np.nan, np.inf, -np.inf])
def test_decode_step_appends_a_nonfinite_token_as_zeros(gpu_lib, val):
    # the decode step's own append of the new token follows the same reading:
    # the non-finite K (or V) row of the token is stored as the zero row, the
    # decode attends over it, the output is finite and equals the oracle's
    cfg = wl.Workload("nonfinite_step", 911, batch=3, nqh=4, nkv=2, ctx_range=(1, 900))
    case = StepCase(cfg)
    kn, vn = case.k_new.copy(), case.v_new.copy()
    kn[0, 1, 17] = val
    vn[2, 0, 90] = val
    case.k_new_d.copy_(torch.from_numpy(kn))
    case.v_new_d.copy_(torch.from_numpy(vn))
    case.status.zero_()
    out = case.step()
    assert case.status_bits() == kvq8.DEV_NONFINITE
    assert np.all(np.isfinite(out))
    pools = case.host_pools()
    G = cfg.group
    for b in range(cfg.batch):
        L = int(case.lens[b])
        for h in range(cfg.nkv):
            k, v = case._full[b]
            k_h, v_h = k[:, h].copy(), v[:, h].copy()
            k_h[L - 1], v_h[L - 1] = kn[b, h], vn[b, h]
            kq, ks = oracle.kv_quantize_rows(k_h)
            vq, vs = oracle.kv_quantize_rows(v_h)
            gk, gks, gv, gvs = case.gather_unit(pools, b, h)
            assert np.array_equal(gk, kq) and np.array_equal(gv, vq)
            assert np.array_equal(gks.view(np.uint32), ks.view(np.uint32))
            assert np.array_equal(gvs.view(np.uint32), vs.view(np.uint32))
            ref, _ = oracle.decode_unit_q8(case.q[b, h * G:(h + 1) * G], k_h, v_h, SM_SCALE)
            assert_close(out[b, h * G:(h + 1) * G], ref, f"nonfinite step b={b} h={h}")


def test_int4_append_nonfinite_groups_bit_exact(gpu_lib):
    nkv, n_new, start = 2, 70, 200
    rng = np.random.default_rng(912)
    k = rng.standard_normal((1, n_new, nkv, HD)).astype(np.float32)
    v = rng.standard_normal((1, n_new, nkv, HD)).astype(np.float32)
    _plant(k, 3, 9)
    _plant(v, 4, 9)
    k[0, 5, 1, 0] = np.nan
    k[0, 5, 1, 127] = np.inf      # both groups of one row
    need = (start + n_new + 255) // 256
    table = np.arange(need, dtype=np.int32)[None]
    cache = kvq8.alloc_cache4(need, nkv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq8.quantize_append4(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                          torch.tensor([start], dtype=torch.int32, device="cuda"),
                          torch.from_numpy(table).cuda(), cache, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == kvq8.DEV_NONFINITE
    kc, vc = cache.k_codes.cpu().numpy(), v4_token_major(cache.v_codes.cpu().numpy())
    kp, vp = cache.k_param.cpu().numpy(), cache.v_param.cpu().numpy()
    pos = start + np.arange(n_new)
    phys, slot = table[0, pos // 256], pos % 256
    replaced = 0
    for h in range(nkv):
        for x, codes, par in ((k[0, :, h], kc, kp), (v[0, :, h], vc, vp)):
            packed, sc, zr, n = oracle.int4_quantize_groups(x, 64, count_nonfinite=True)
            replaced += n
            assert np.array_equal(codes[phys, h, slot], packed)
            got = par[phys, h, slot]
            assert np.array_equal(got[:, [0, 2]].view(np.uint32), sc.view(np.uint32))
            assert np.array_equal(got[:, [1, 3]].view(np.uint32), zr.view(np.uint32))
    assert replaced >= 19


@pytest.mark.parametrize("val", [np.nan, np.inf, -np.inf])
def test_int4_decode_step_appends_a_nonfinite_token_as_zeros(gpu_lib, val):
    # kvq4_decode_step's own append follows the same reading: a 64-value group
    # of the new K (or V) row holding a NaN or an infinity is stored as the zero
    # group (scale 1, zero -0, codes 0), the status carries the non-finite bit,
    # and the output is finite and equals the oracle's over the stored cache
    cfg = wl.Workload("nonfinite_step4", 913, batch=3, nqh=8, nkv=2, ctx_range=(2, 900))
    lens = wl.ctx_lens(cfg)
    table, num_blocks = wl.block_table(cfg, lens, spare_blocks=1)
    table_d, lens_d = torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda()
    cache = kvq8.alloc_cache4(num_blocks, cfg.nkv)
    zero = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k_new = np.zeros((cfg.batch, cfg.nkv, HD), np.float32)
    v_new = np.zeros_like(k_new)
    full = []
    for b in range(cfg.batch):
        L = int(lens[b])
        k, v = wl.seq_kv(cfg, b, L)
        full.append((k.copy(), v.copy()))
        k_new[b], v_new[b] = k[L - 1], v[L - 1]
        kvq8.quantize_append4(torch.from_numpy(k[None, :L - 1]).cuda(), torch.from_numpy(v[None, :L - 1]).cuda(),
                              zero, table_d[b:b + 1], cache, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    k_new[0, 1, 17] = val                   # first group of a K row
    v_new[2, 0, 90] = val                   # second group of a V row
    q = wl.queries(cfg)
    out = torch.full((cfg.batch, cfg.nqh, HD), float("nan"), device="cuda")
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, table.shape[1])
    kvq8.decode_step4(torch.from_numpy(q).cuda(), torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda(),
                      cache, table_d, lens_d, out, ws, sm_scale=SM_SCALE, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == kvq8.DEV_NONFINITE
    o = out.cpu().numpy()
    assert np.all(np.isfinite(o))
    kc, vc = cache.k_codes.cpu().numpy(), v4_token_major(cache.v_codes.cpu().numpy())
    kp, vp = cache.k_param.cpu().numpy(), cache.v_param.cpu().numpy()
    G = cfg.group
    for b in range(cfg.batch):
        L = int(lens[b])
        phys, slot = table[b, (L - 1) // 256], (L - 1) % 256
        for h in range(cfg.nkv):
            k_h, v_h = full[b][0][:, h].copy(), full[b][1][:, h].copy()
            k_h[L - 1], v_h[L - 1] = k_new[b, h], v_new[b, h]
            for x, codes, par in ((k_h[L - 1], kc, kp), (v_h[L - 1], vc, vp)):
                packed, sc, zr = oracle.int4_quantize_groups(x[None], 64)
                assert np.array_equal(codes[phys, h, slot], packed[0])
                got = par[phys, h, slot]
                assert np.array_equal(got[[0, 2]].view(np.uint32), sc[0].view(np.uint32))
                assert np.array_equal(got[[1, 3]].view(np.uint32), zr[0].view(np.uint32))
            kd = oracle.int4_dequantize_groups(*oracle.int4_quantize_groups(k_h, 64), 64)
            vd = oracle.int4_dequantize_groups(*oracle.int4_quantize_groups(v_h, 64), 64)
            ref = np.stack([oracle.attention_f64(q[b, h * G + g], kd, vd, SM_SCALE) for g in range(G)])
            assert_close(o[b, h * G:(h + 1) * G], ref, f"int4 nonfinite step b={b} h={h}")
