"""The 4-bit (asymmetric INT4 group-64) cache path against the oracle.

Codes, scales and zeros must match the oracle's quantiser bit for bit; decode
outputs (fp32 query over dequantised K/V) must be within 1e-4 max-abs and
1e-3 relative (max norm) of fp64 attention over the oracle's dequantised K/V.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from int8_quantized_kv_gb300 import kvq8
from int8_quantized_kv_gb300 import workloads as wl
from kvq8_harness import SM_SCALE, assert_close, v4_token_major

pytestmark = pytest.mark.gpu
HD = 128
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


class Int4Case:
    def __init__(self, cfg, lens=None, spare_blocks=2):
        self.cfg = cfg
        self.lens = wl.ctx_lens(cfg) if lens is None else np.asarray(lens, np.int32)
        self.table, self.num_blocks = wl.block_table(cfg, self.lens, spare_blocks=spare_blocks)
        self.max_blocks = self.table.shape[1]
        self.cache = kvq8.alloc_cache4(self.num_blocks, cfg.nkv)
        self.table_d = torch.from_numpy(self.table).cuda()
        self.lens_d = torch.from_numpy(self.lens).cuda()
        self.q = wl.queries(cfg)
        self.q_d = torch.from_numpy(self.q).cuda()
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        zero = torch.zeros(1, dtype=torch.int32, device="cuda")
        for b in range(cfg.batch):
            L = int(self.lens[b])
            if L:
                k, v = wl.seq_kv(cfg, b, L)
                kvq8.quantize_append4(torch.from_numpy(k[None]).cuda(), torch.from_numpy(v[None]).cuda(),
                                      zero, self.table_d[b:b + 1], self.cache, dev_status=self.status)
        torch.cuda.synchronize()

    def decode(self):
        out = torch.full_like(self.q_d, float("nan"))
        ws = kvq8.alloc_workspace(self.cfg.batch, self.cfg.nqh, self.cfg.nkv, self.max_blocks)
        kvq8.decode_attn4(self.q_d, self.cache, self.table_d, self.lens_d, out, ws, sm_scale=SM_SCALE,
                          dev_status=self.status)
        torch.cuda.synchronize()
        return out.cpu().numpy()

    def oracle_unit(self, b, h):
        G = self.cfg.group
        L = int(self.lens[b])
        k, v = wl.unit_kv(self.cfg, b, h, L)
        kd = oracle.int4_dequantize_groups(*oracle.int4_quantize_groups(k, 64), 64)
        vd = oracle.int4_dequantize_groups(*oracle.int4_quantize_groups(v, 64), 64)
        return np.stack([oracle.attention_f64(self.q[b, h * G + g], kd, vd, SM_SCALE) for g in range(G)])


def _rows_with_fixtures(n, seed):
    rng = np.random.default_rng(seed)
    m = max(n, 5)
    x = (rng.standard_normal((m, HD)) * rng.uniform(0.01, 30, (m, 1))).astype(np.float32)
    g = json.load(open(os.path.join(GOLDEN, "int4_group64_hand_example.json")))
    row = np.full(HD, g["row_fill_group0"], np.float32)
    row[:len(g["row_head"])] = g["row_head"]
    row[64:] = g["row_group1_constant"]
    x[0] = row                                   # hand-worked example (one constant group)
    x[1] = 0.0                                   # all-zero row: both groups constant
    x[2, :64] = np.abs(x[2, :64]) + 1.0          # all-positive group: zero below 0
    x[3, 64:] = -np.abs(x[3, 64:]) - 1.0         # all-negative group: zero above 15
    x[4] = 7.0                                   # scale exactly 1 in both groups: ties
    x[4, :8] = [0.0, 15.0, 0.5, 1.5, 2.5, 3.5, 13.5, 14.5]      # codes on k + 1/2
    x[4, 64:70] = [-2.5, 12.5, 0.5, -1.5, 1.5, 10.5]          # zero = round(2.5)
    return x[:n] if n >= 5 else np.roll(x, -(5 - n), axis=0)[:n]


@pytest.mark.parametrize("start,n_new", [(0, 1), (5, 37), (250, 300)])
def test_int4_append_bit_exact(gpu_lib, start, n_new):
    nkv = 2
    k = np.stack([_rows_with_fixtures(n_new * nkv, 11 + n_new).reshape(n_new, nkv, HD)])
    v = np.stack([_rows_with_fixtures(n_new * nkv, 13 + n_new).reshape(n_new, nkv, HD)])
    need = (start + n_new + 255) // 256
    table = np.random.default_rng(3).permutation(need + 2)[:need].astype(np.int32)[None]
    cache = kvq8.alloc_cache4(need + 2, nkv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq8.quantize_append4(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                          torch.tensor([start], dtype=torch.int32, device="cuda"),
                          torch.from_numpy(table).cuda(), cache, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    kc, vc = cache.k_codes.cpu().numpy(), v4_token_major(cache.v_codes.cpu().numpy())
    kp, vp = cache.k_param.cpu().numpy(), cache.v_param.cpu().numpy()
    pos = start + np.arange(n_new)
    phys, slot = table[0, pos // 256], pos % 256
    for h in range(nkv):
        for x, codes, par in ((k[0, :, h], kc, kp), (v[0, :, h], vc, vp)):
            packed, sc, zr = oracle.int4_quantize_groups(x, 64)
            assert np.array_equal(codes[phys, h, slot], packed)
            got = par[phys, h, slot]
            assert np.array_equal(got[:, [0, 2]].view(np.uint32), sc.view(np.uint32))
            assert np.array_equal(got[:, [1, 3]].view(np.uint32), zr.view(np.uint32))


def test_int4_byte_count(gpu_lib):
    # 64 code bytes + 4 fp32 per (token, head) for K and V: 1280 B per token per layer at nkv = 8
    assert kvq8.cache4_bytes_per_token(8) == 1280
    c = kvq8.alloc_cache4(3, 8)
    assert sum(t.numel() * t.element_size() for t in c) == 3 * 256 * 1280


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_int4_decode_group_sizes(gpu_lib, G):
    cfg = wl.Workload(f"int4_g{G}", 500 + G, batch=3, nqh=2 * G, nkv=2, ctx_range=(1, 1400))
    case = Int4Case(cfg)
    out = case.decode()
    for b in range(cfg.batch):
        for h in range(cfg.nkv):
            assert_close(out[b, h * G:(h + 1) * G], case.oracle_unit(b, h), f"int4 G={G} b={b} h={h}")
    assert case.status.item() == 0


@pytest.mark.parametrize("L", [1, 31, 32, 33, 257, 3000])
def test_int4_decode_lengths(gpu_lib, L):
    cfg = wl.Workload("int4_len", 510, batch=1, nqh=4, nkv=1, ctx=L)
    case = Int4Case(cfg)
    assert_close(case.decode()[0], case.oracle_unit(0, 0), f"int4 L={L}")


def test_int4_decode_empty_and_bad_block(gpu_lib):
    cfg = wl.Workload("int4_edge", 520, batch=3, nqh=4, nkv=2, ctx_range=(300, 900))
    case = Int4Case(cfg, lens=np.array([0, 700, 600], np.int32))
    out = case.decode()
    assert not out[0].any()
    case.table_d[2, 1] = case.num_blocks + 3          # block 1 of sequence 2 out of range
    out = case.decode()
    assert case.status.item() & kvq8.DEV_BAD_BLOCK_ID
    G = cfg.group
    for h in range(cfg.nkv):
        assert_close(out[1, h * G:(h + 1) * G], case.oracle_unit(1, h))
        k, v = wl.unit_kv(cfg, 2, h, 600)
        keep = np.r_[0:256, 512:600]
        kd = oracle.int4_dequantize_groups(*oracle.int4_quantize_groups(k[keep], 64), 64)
        vd = oracle.int4_dequantize_groups(*oracle.int4_quantize_groups(v[keep], 64), 64)
        ref = np.stack([oracle.attention_f64(case.q[2, h * G + g], kd, vd, SM_SCALE) for g in range(G)])
        assert_close(out[2, h * G:(h + 1) * G], ref)


def test_int4_workload_scaled(gpu_lib):
    cfg = wl.scaled(wl.INT4_G64_32K, batch=2, ctx=2500)
    case = Int4Case(cfg)
    out = case.decode()
    G = cfg.group
    for b in range(cfg.batch):
        for h in range(cfg.nkv):
            assert_close(out[b, h * G:(h + 1) * G], case.oracle_unit(b, h), f"b={b} h={h}")


@pytest.mark.slow
def test_int4_workload_full_size_sampled(gpu_lib):
    cfg = wl.INT4_G64_32K
    case = Int4Case(cfg, spare_blocks=0)
    out = case.decode()
    assert case.status.item() == 0 and np.all(np.isfinite(out))
    rng = np.random.default_rng(6)
    G = cfg.group
    for b, h in {(int(rng.integers(cfg.batch)), int(rng.integers(cfg.nkv))) for _ in range(4)}:
        assert_close(out[b, h * G:(h + 1) * G], case.oracle_unit(b, h), f"full int4 b={b} h={h}")


def test_int4_decode_on_host_mapped_buffers(gpu_lib):
    """The same call with the query read from, and the result written to,
    page-locked host memory (kvq8.HostMapped) gives the device call's output
    bit for bit."""
    cfg = wl.Workload("int4_host", 690, batch=3, nqh=8, nkv=2, ctx_range=(100, 1500))
    case = Int4Case(cfg)
    dev_out = case.decode()
    q_h = torch.from_numpy(case.q).pin_memory()
    out_h = torch.full(tuple(q_h.shape), float("nan")).pin_memory()
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, case.max_blocks)
    kvq8.decode_attn4(kvq8.HostMapped(q_h), case.cache, case.table_d, case.lens_d, kvq8.HostMapped(out_h), ws,
                      sm_scale=SM_SCALE, dev_status=case.status)
    torch.cuda.synchronize()
    assert case.status.item() == 0
    assert np.array_equal(out_h.numpy(), dev_out)
    with pytest.raises(ValueError):
        kvq8.HostMapped(torch.zeros(4))          # pageable: not addressable by the device


def test_int4_back_to_back_calls_share_the_workspace(gpu_lib):
    # three calls on one stream and one workspace with no synchronisation in
    # between, the second with another query: each split may start before the
    # merge of the call before it has read the workspace, and must wait for it
    # (programmatic dependent launch); every output equals its own decode
    cfg = wl.Workload("int4_b2b", 530, batch=3, nqh=8, nkv=2, ctx_range=(700, 3000))
    case = Int4Case(cfg)
    q1 = case.q
    q2 = np.random.default_rng(531).standard_normal(q1.shape).astype(np.float32) * 2.0
    q1_d, q2_d = case.q_d, torch.from_numpy(q2).cuda()
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, case.max_blocks)
    outs = [torch.full_like(q1_d, float("nan")) for _ in range(3)]
    for q_d, out in zip((q1_d, q2_d, q1_d), outs):
        kvq8.decode_attn4(q_d, case.cache, case.table_d, case.lens_d, out, ws, sm_scale=SM_SCALE,
                          dev_status=case.status)
    torch.cuda.synchronize()
    assert case.status.item() == 0
    o1, o2, o3 = (o.cpu().numpy() for o in outs)
    assert np.array_equal(o1, o3)
    G = cfg.group
    for q, o in ((q1, o1), (q2, o2)):
        case.q = q
        for b in range(cfg.batch):
            for h in range(cfg.nkv):
                assert_close(o[b, h * G:(h + 1) * G], case.oracle_unit(b, h), f"int4 back to back b={b} h={h}")
    case.q = q1


def test_int4_merge_without_directory_ragged(gpu_lib):
    # 64 units: at most 8 splits per unit, so the merge reads each unit's
    # records at u * nsplit + j without the record directory and takes their
    # count from the unit's length; lengths from empty to several blocks,
    # several too short to give every split a chunk
    lens = np.array([0, 1, 31, 33, 200, 1000, 3000, 5000], np.int32)
    cfg = wl.Workload("int4_fixed_merge", 540, batch=8, nqh=32, nkv=8, ctx=int(lens.max()))
    case = Int4Case(cfg, lens=lens)
    out = case.decode()
    assert case.status.item() == 0
    assert not out[0].any()
    G = cfg.group
    for b in range(1, cfg.batch):
        for h in range(cfg.nkv):
            assert_close(out[b, h * G:(h + 1) * G], case.oracle_unit(b, h), f"int4 fixed merge b={b} h={h}")


@pytest.mark.parametrize("G", [1, 4, 8])
def test_int4_decode_step_appends_the_token(gpu_lib, G):
    # kvq4_decode_step on a cache holding L - 1 tokens: the new token lands at
    # position L - 1 bit for bit as the oracle quantises it, the output equals
    # the oracle's decode over the L tokens, and both equal a separate append
    # followed by a decode, bit for bit; an empty sequence appends nothing
    cfg = wl.Workload(f"int4_step_g{G}", 550 + G, batch=5, nqh=2 * G, nkv=2, ctx_range=(2, 1500))
    lens = wl.ctx_lens(cfg)
    lens[0], lens[1], lens[2] = 0, 1, 257          # empty, only the new token, a block's first slot
    table, num_blocks = wl.block_table(cfg, lens, spare_blocks=2)
    table_d = torch.from_numpy(table).cuda()
    lens_d = torch.from_numpy(lens).cuda()
    zero = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    caches = [kvq8.alloc_cache4(num_blocks, cfg.nkv) for _ in range(2)]
    k_new = np.zeros((cfg.batch, cfg.nkv, HD), np.float32)
    v_new = np.zeros_like(k_new)
    for b in range(cfg.batch):
        L = int(lens[b])
        if L == 0:
            continue
        k, v = wl.seq_kv(cfg, b, L)
        k_new[b], v_new[b] = k[L - 1], v[L - 1]
        if L > 1:
            for c in caches:
                kvq8.quantize_append4(torch.from_numpy(k[None, :L - 1]).cuda(),
                                      torch.from_numpy(v[None, :L - 1]).cuda(), zero, table_d[b:b + 1], c,
                                      dev_status=status)
    q = wl.queries(cfg)
    q_d, kn_d, vn_d = torch.from_numpy(q).cuda(), torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda()
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, table.shape[1])
    out_step = torch.full_like(q_d, float("nan"))
    kvq8.decode_step4(q_d, kn_d, vn_d, caches[0], table_d, lens_d, out_step, ws, sm_scale=SM_SCALE,
                      dev_status=status)
    # the same as a separate append of the token and a decode
    start = torch.from_numpy((lens - 1).clip(min=0).astype(np.int32)).cuda()
    has = torch.from_numpy((lens > 0).astype(np.int32)).cuda()
    for b in range(cfg.batch):
        if lens[b] > 0:
            kvq8.quantize_append4(kn_d[b:b + 1, None], vn_d[b:b + 1, None], start[b:b + 1], table_d[b:b + 1],
                                  caches[1], dev_status=status)
    out_two = torch.full_like(q_d, float("nan"))
    kvq8.decode_attn4(q_d, caches[1], table_d, lens_d, out_two, ws, sm_scale=SM_SCALE, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0 and has.numel() == cfg.batch
    o_step, o_two = out_step.cpu().numpy(), out_two.cpu().numpy()
    assert np.array_equal(o_step, o_two)
    assert not o_step[0].any()
    kc, vc = caches[0].k_codes.cpu().numpy(), v4_token_major(caches[0].v_codes.cpu().numpy())
    kp, vp = caches[0].k_param.cpu().numpy(), caches[0].v_param.cpu().numpy()
    case = Int4Case.__new__(Int4Case)
    case.cfg, case.lens, case.q = cfg, lens, q
    for b in range(1, cfg.batch):
        L = int(lens[b])
        phys, slot = table[b, (L - 1) // 256], (L - 1) % 256
        for h in range(cfg.nkv):
            for x, codes, par in ((k_new[b, h], kc, kp), (v_new[b, h], vc, vp)):
                packed, sc, zr = oracle.int4_quantize_groups(x[None], 64)
                assert np.array_equal(codes[phys, h, slot], packed[0])
                got = par[phys, h, slot]
                assert np.array_equal(got[[0, 2]].view(np.uint32), sc[0].view(np.uint32))
                assert np.array_equal(got[[1, 3]].view(np.uint32), zr[0].view(np.uint32))
            assert_close(o_step[b, h * G:(h + 1) * G], case.oracle_unit(b, h), f"int4 step G={G} b={b} h={h}")
