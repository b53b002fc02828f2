"""The fp32 K/V cache (the comparator of the int8 cache) against the oracle.

Append is a copy: the cache must hold the input rows bit for bit.  Decode
outputs must be within 1e-4 max-abs and 1e-3 relative (max norm) of fp64
attention over the same fp32 K/V.  The comparison of [Day 9-3] §1 (one attention over fp32 K/V, the same
attention over the int8 cache, compare per dimension) run on the GPU must
give the oracle's per-dimension deltas.
"""
import numpy as np
import pytest
import torch

import oracle
from int8_quantized_kv_gb300 import kvq8
from int8_quantized_kv_gb300 import workloads as wl
from kvq8_harness import ABS_TOL, REL_TOL, SM_SCALE, Case, assert_close

pytestmark = pytest.mark.gpu
HD = 128


class F32Case:
    def __init__(self, cfg, lens=None, spare_blocks=2, append_chunk=None):
        self.cfg = cfg
        self.lens = wl.ctx_lens(cfg) if lens is None else np.asarray(lens, np.int32)
        self.table, self.num_blocks = wl.block_table(cfg, self.lens, spare_blocks=spare_blocks)
        self.max_blocks = self.table.shape[1]
        self.cache = kvq8.alloc_cachef32(self.num_blocks, cfg.nkv)
        self.table_d = torch.from_numpy(self.table).cuda()
        self.lens_d = torch.from_numpy(self.lens).cuda()
        self.q = wl.queries(cfg)
        self.q_d = torch.from_numpy(self.q).cuda()
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        for b in range(cfg.batch):
            L = int(self.lens[b])
            if not L:
                continue
            k, v = wl.seq_kv(cfg, b, L)
            step = L if append_chunk is None else append_chunk
            for s in range(0, L, step):
                e = min(L, s + step)
                kvq8.appendf32(torch.from_numpy(k[None, s:e]).cuda(), torch.from_numpy(v[None, s:e]).cuda(),
                               torch.tensor([s], dtype=torch.int32, device="cuda"), self.table_d[b:b + 1],
                               self.cache, dev_status=self.status)
        torch.cuda.synchronize()

    def decode(self):
        out = torch.full_like(self.q_d, float("nan"))
        ws = kvq8.alloc_workspace(self.cfg.batch, self.cfg.nqh, self.cfg.nkv, self.max_blocks)
        kvq8.decode_attnf32(self.q_d, self.cache, self.table_d, self.lens_d, out, ws, sm_scale=SM_SCALE,
                            dev_status=self.status)
        torch.cuda.synchronize()
        return out.cpu().numpy()

    def oracle_unit(self, b, h):
        G = self.cfg.group
        k, v = wl.unit_kv(self.cfg, b, h, int(self.lens[b]))
        return np.stack([oracle.attention_f64(self.q[b, h * G + g], k, v, SM_SCALE) for g in range(G)])


@pytest.mark.parametrize("start,n_new", [(0, 1), (7, 100), (250, 600)])
def test_f32_append_copies_rows(gpu_lib, start, n_new):
    nkv = 3
    rng = np.random.default_rng(40 + n_new)
    k = rng.standard_normal((2, n_new, nkv, HD), dtype=np.float32)
    v = rng.standard_normal((2, n_new, nkv, HD), dtype=np.float32)
    need = (start + n_new + 255) // 256
    table = rng.permutation(2 * need + 1)[:2 * need].astype(np.int32).reshape(2, need)
    cache = kvq8.alloc_cachef32(2 * need + 1, nkv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq8.appendf32(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                   torch.tensor([start, start], dtype=torch.int32, device="cuda"),
                   torch.from_numpy(table).cuda(), cache, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    kc, vc = cache.k_cache.cpu().numpy(), cache.v_cache.cpu().numpy()
    pos = start + np.arange(n_new)
    for b in range(2):
        phys, slot = table[b, pos // 256], pos % 256
        for h in range(nkv):
            assert np.array_equal(kc[phys, h, slot].view(np.uint32), k[b, :, h].view(np.uint32))
            assert np.array_equal(vc[phys, h, slot].view(np.uint32), v[b, :, h].view(np.uint32))


def test_f32_append_flags_bad_position_and_block(gpu_lib):
    cache = kvq8.alloc_cachef32(2, 1)
    cache.k_cache.zero_()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = torch.ones((1, 4, 1, HD), dtype=torch.float32, device="cuda")
    table = torch.tensor([[0, 5]], dtype=torch.int32, device="cuda")    # block 5 does not exist
    kvq8.appendf32(k, k, torch.tensor([510], dtype=torch.int32, device="cuda"), table, cache,
                   dev_status=status)
    torch.cuda.synchronize()
    assert status.item() & kvq8.DEV_BAD_BLOCK_ID
    assert status.item() & kvq8.DEV_BAD_POSITION      # positions 512, 513 are past the table
    assert not cache.k_cache.any().item()


def test_f32_byte_count(gpu_lib):
    # 128 fp32 for K and V per (token, head): 8192 B per token per layer at nkv = 8
    assert kvq8.cachef32_bytes_per_token(8) == 8192
    assert kvq8.cachef32_bytes_per_token(8) * 2112 == kvq8.cache_bytes_per_token(8) * 8192


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_f32_decode_group_sizes(gpu_lib, G):
    cfg = wl.Workload(f"f32_g{G}", 600 + G, batch=3, nqh=2 * G, nkv=2, ctx_range=(1, 1400))
    case = F32Case(cfg)
    out = case.decode()
    for b in range(cfg.batch):
        for h in range(cfg.nkv):
            assert_close(out[b, h * G:(h + 1) * G], case.oracle_unit(b, h), f"f32 G={G} b={b} h={h}")
    assert case.status.item() == 0


@pytest.mark.parametrize("L", [1, 7, 8, 9, 63, 64, 65, 257, 3000])
def test_f32_decode_lengths(gpu_lib, L):
    cfg = wl.Workload("f32_len", 610, batch=1, nqh=4, nkv=1, ctx=L)
    case = F32Case(cfg, append_chunk=100)
    assert_close(case.decode()[0], case.oracle_unit(0, 0), f"f32 L={L}")


def test_f32_decode_empty_and_bad_block(gpu_lib):
    cfg = wl.Workload("f32_edge", 620, batch=3, nqh=4, nkv=2, ctx_range=(300, 900))
    case = F32Case(cfg, lens=np.array([0, 700, 600], np.int32))
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
        ref = np.stack([oracle.attention_f64(case.q[2, h * G + g], k[keep], v[keep], SM_SCALE)
                        for g in range(G)])
        assert_close(out[2, h * G:(h + 1) * G], ref)


def test_f32_workload_scaled_outliers(gpu_lib):
    cfg = wl.scaled(wl.LONG128K_OUTLIERS, batch=2, ctx=5000)
    case = F32Case(cfg)
    out = case.decode()
    G = cfg.group
    for b in range(cfg.batch):
        for h in range(cfg.nkv):
            assert_close(out[b, h * G:(h + 1) * G], case.oracle_unit(b, h), f"b={b} h={h}")


@pytest.mark.parametrize("cfg", [wl.SINGLE_HEAD_L256, wl.scaled(wl.QWEN3_2B_28L_8K, batch=2, ctx=1500)],
                         ids=lambda c: c.name)
def test_fp32_vs_q8_comparison_matches_oracle(gpu_lib, cfg):
    # [Day 9-3] §1: the same attention over fp32 K/V and over the int8 cache;
    # the GPU's per-dimension delta must be the oracle's, within both sides' bars
    f32 = F32Case(cfg).decode()
    q8 = Case(cfg).decode()
    G = cfg.group
    for b in range(cfg.batch):
        for h in range(cfg.nkv):
            k, v = wl.unit_kv(cfg, b, h, int(wl.ctx_lens(cfg)[b]))
            ref32 = np.stack([oracle.attention_f64(wl.queries(cfg)[b, h * G + g], k, v, SM_SCALE)
                              for g in range(G)])
            ref8, _ = oracle.decode_unit_q8(wl.queries(cfg)[b, h * G:(h + 1) * G], k, v, SM_SCALE)
            d_gpu = q8[b, h * G:(h + 1) * G] - f32[b, h * G:(h + 1) * G]
            d_orc = ref8 - ref32
            bound = 2 * ABS_TOL + REL_TOL * (np.abs(ref8) + np.abs(ref32))
            assert np.all(np.abs(d_gpu - d_orc) <= bound), f"b={b} h={h}"
            assert abs(np.abs(d_gpu).mean() - np.abs(d_orc).mean()) <= 2 * ABS_TOL
