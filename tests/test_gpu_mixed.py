"""Mixed precision by token age (UltraQuant §3.3): the old 256-token blocks of a
sequence requantised from int8 to INT4 group-64, the recent ones kept int8,
one decode over both.

Requantised codes, scales and zeros must match the oracle's (INT4 rule applied
to the int8 rows' fp32 values) bit for bit; decode outputs must be within
1e-4 max-abs and 1e-3 relative (max norm) of the oracle's mixed decode; with no old blocks the result
is the int8 decode's, with only old blocks the 4-bit decode's, bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from int8_quantized_kv_gb300 import kvq8
from int8_quantized_kv_gb300 import workloads as wl
from kvq8_harness import SM_SCALE, Case, assert_close, k_rows_logical, v4_token_major, v_rows_logical

pytestmark = pytest.mark.gpu
BS = 256


class MixedCase(Case):
    """An int8 cache holding every token, plus a 4-bit pool into which the
    first n4[b] logical blocks of each sequence are requantised."""

    def __init__(self, cfg, n4, lens=None, seed=0):
        super().__init__(cfg, lens=lens)
        # requantisation converts whole 256-token tiles: the slots past a
        # sequence's end hold whatever the pool held (never read as tokens);
        # zeros there keep the status word free of flags raised by leftovers
        self._zero_unused_slots()
        B, mb = self.table.shape
        rng = np.random.default_rng(900 + seed)
        self.num_blocks4 = B * mb + 3
        self.table4 = rng.permutation(self.num_blocks4)[:B * mb].astype(np.int32).reshape(B, mb)
        self.table4_d = torch.from_numpy(self.table4).cuda()
        self.cache4 = kvq8.alloc_cache4(self.num_blocks4, cfg.nkv)
        self.n4 = np.minimum(np.asarray(n4, np.int32), mb).astype(np.int32)
        self.n4_d = torch.from_numpy(self.n4).cuda()
        zero = torch.zeros(B, dtype=torch.int32, device="cuda")
        kvq8.requantize_blocks(self.cache, self.table_d, self.cache4, self.table4_d, zero, self.n4_d,
                               max(1, int(self.n4.max())), dev_status=self.status)
        torch.cuda.synchronize()

    def _zero_unused_slots(self):
        torch.cuda.synchronize()
        B, mb = self.table.shape
        for b in range(B):
            L = int(self.lens[b])
            j = L // 256                      # the sequence's last, partly filled block
            if L % 256 and j < mb and self.table[b, j] >= 0:
                phys = int(self.table[b, j])
                self.cache.k_scale[phys, :, L % 256:] = 0.0
                self.cache.v_scale[phys, :, L % 256:] = 0.0
        torch.cuda.synchronize()

    def decode_mixed(self):
        out = torch.full_like(self.q_d, float("nan"))
        ws = kvq8.alloc_mixed_workspace(self.cfg.batch, self.cfg.nqh, self.cfg.nkv, self.max_blocks)
        kvq8.decode_attn_mixed(self.q_d, self.cache, self.table_d, self.cache4, self.table4_d, self.lens_d,
                               self.n4_d, out, ws, sm_scale=SM_SCALE, dev_status=self.status)
        torch.cuda.synchronize()
        return out.cpu().numpy()

    def oracle_mixed(self, b, h):
        G = self.cfg.group
        L = int(self.lens[b])
        k, v = wl.unit_kv(self.cfg, b, h, L)
        return oracle.decode_mixed_unit(self.q[b, h * G:(h + 1) * G], k, v, min(L, BS * int(self.n4[b])), SM_SCALE)


def test_requantised_tiles_bit_exact(gpu_lib):
    cfg = wl.Workload("mix_req", 700, batch=2, nqh=4, nkv=2, ctx_range=(600, 1100))
    case = MixedCase(cfg, n4=[2, 3])
    assert case.status_bits() == 0
    pools = case.host_pools()
    kc, vc = case.cache4.k_codes.cpu().numpy(), v4_token_major(case.cache4.v_codes.cpu().numpy())
    kp, vp = case.cache4.k_param.cpu().numpy(), case.cache4.v_param.cpu().numpy()
    for b in range(cfg.batch):
        for h in range(cfg.nkv):
            for j in range(int(case.n4[b])):
                slots = np.arange(BS)
                p8, p4 = case.table[b, j], case.table4[b, j]
                L = int(case.lens[b])
                ok = slots[(j * BS + slots) < L]        # slots that hold tokens
                kq = k_rows_logical(pools[0], p8, h, ok)
                vq = v_rows_logical(pools[1], p8, h, ok)
                for rows, sc, codes, par in ((kq, pools[2][p8, h, ok], kc, kp), (vq, pools[3][p8, h, ok], vc, vp)):
                    packed, s4, z4 = oracle.requantize_q8_to_q4(rows, sc)
                    assert np.array_equal(codes[p4, h, ok], packed), (b, h, j)
                    got = par[p4, h, ok]
                    assert np.array_equal(got[:, [0, 2]].view(np.uint32), s4.view(np.uint32))
                    assert np.array_equal(got[:, [1, 3]].view(np.uint32), z4.view(np.uint32))


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_mixed_decode_group_sizes(gpu_lib, G):
    cfg = wl.Workload(f"mix_g{G}", 710 + G, batch=4, nqh=2 * G, nkv=2, ctx_range=(1, 2000))
    lens = wl.ctx_lens(cfg)
    n4 = [(int(L) // BS) // 2 + (i % 2) for i, L in enumerate(lens)]
    case = MixedCase(cfg, n4=n4, seed=G)
    out = case.decode_mixed()
    for b in range(cfg.batch):
        for h in range(cfg.nkv):
            assert_close(out[b, h * G:(h + 1) * G], case.oracle_mixed(b, h), f"mixed G={G} b={b} h={h}")
    assert case.status_bits() == 0


@pytest.mark.parametrize("L,n4", [(256, 1), (257, 1), (600, 2), (600, 3), (1500, 5), (3000, 4)])
def test_mixed_decode_boundaries(gpu_lib, L, n4):
    cfg = wl.Workload("mix_len", 720, batch=1, nqh=4, nkv=1, ctx=L)
    case = MixedCase(cfg, n4=[n4])
    assert_close(case.decode_mixed()[0], case.oracle_mixed(0, 0), f"mixed L={L} n4={n4}")


def test_mixed_without_old_blocks_is_the_int8_decode(gpu_lib):
    cfg = wl.Workload("mix_zero", 730, batch=3, nqh=8, nkv=2, ctx_range=(100, 3000))
    case = MixedCase(cfg, n4=[0, 0, 0])
    assert np.array_equal(case.decode_mixed(), case.decode())


def test_mixed_with_only_old_blocks_is_the_4bit_decode(gpu_lib):
    cfg = wl.Workload("mix_all", 731, batch=3, nqh=8, nkv=2, ctx_range=(100, 3000))
    lens = wl.ctx_lens(cfg)
    case = MixedCase(cfg, n4=[(int(L) + BS - 1) // BS for L in lens])
    mixed = case.decode_mixed()
    out = torch.full_like(case.q_d, float("nan"))
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, case.max_blocks)
    kvq8.decode_attn4(case.q_d, case.cache4, case.table4_d, case.lens_d, out, ws, sm_scale=SM_SCALE)
    torch.cuda.synchronize()
    assert np.array_equal(mixed, out.cpu().numpy())


def test_mixed_empty_sequence_and_bad_blocks(gpu_lib):
    cfg = wl.Workload("mix_edge", 740, batch=3, nqh=4, nkv=2, ctx_range=(700, 1200))
    case = MixedCase(cfg, n4=[1, 1, 2], lens=np.array([0, 900, 1000], np.int32))
    out = case.decode_mixed()
    assert not out[0].any()
    for h in range(cfg.nkv):
        assert_close(out[1, 2 * h:2 * h + 2], case.oracle_mixed(1, h))
    # an out-of-range 4-bit tile id in sequence 2 is flagged and its block skipped
    case.table4_d[2, 1] = case.num_blocks4 + 5
    case.decode_mixed()
    assert case.status_bits() & kvq8.DEV_BAD_BLOCK_ID
    # a requantisation range past the table is flagged
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq8.requantize_blocks(case.cache, case.table_d, case.cache4, case.table4_d,
                           torch.zeros(3, dtype=torch.int32, device="cuda"),
                           torch.full((3,), case.max_blocks + 2, dtype=torch.int32, device="cuda"),
                           case.max_blocks + 2, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & kvq8.DEV_BAD_POSITION


def test_mixed_qwen_shape_sampled(gpu_lib):
    cfg = wl.scaled(wl.QWEN3_2B_28L_8K, batch=4, ctx=8192)
    case = MixedCase(cfg, n4=[24, 16, 31, 0])
    out = case.decode_mixed()
    assert case.status_bits() == 0 and np.all(np.isfinite(out))
    G = cfg.group
    rng = np.random.default_rng(7)
    for b, h in {(int(rng.integers(cfg.batch)), int(rng.integers(cfg.nkv))) for _ in range(5)}:
        assert_close(out[b, h * G:(h + 1) * G], case.oracle_mixed(b, h), f"qwen mixed b={b} h={h}")


def test_mixed_back_to_back_calls_share_the_workspace(gpu_lib):
    # three calls on one stream and one workspace with no synchronisation in
    # between, the second with another query: the 4-bit split of a call may
    # start before the merge of the call before it has read the workspace, and
    # must wait for it; every output equals its own decode
    cfg = wl.Workload("mix_b2b", 760, batch=3, nqh=8, nkv=2, ctx_range=(900, 2600))
    case = MixedCase(cfg, n4=[2, 3, 1], seed=7)
    q1 = case.q
    q2 = np.random.default_rng(761).standard_normal(q1.shape).astype(np.float32) * 2.0
    q1_d, q2_d = case.q_d, torch.from_numpy(q2).cuda()
    ws = kvq8.alloc_mixed_workspace(cfg.batch, cfg.nqh, cfg.nkv, case.max_blocks)
    outs = [torch.full_like(q1_d, float("nan")) for _ in range(3)]
    for q_d, out in zip((q1_d, q2_d, q1_d), outs):
        kvq8.decode_attn_mixed(q_d, case.cache, case.table_d, case.cache4, case.table4_d, case.lens_d,
                               case.n4_d, out, ws, sm_scale=SM_SCALE, dev_status=case.status)
    torch.cuda.synchronize()
    assert case.status_bits() == 0
    o1, o2, o3 = (o.cpu().numpy() for o in outs)
    assert np.array_equal(o1, o3)
    G = cfg.group
    for q, o in ((q1, o1), (q2, o2)):
        case.q = q
        for b in range(cfg.batch):
            for h in range(cfg.nkv):
                assert_close(o[b, h * G:(h + 1) * G], case.oracle_mixed(b, h), f"mixed back to back b={b} h={h}")
    case.q = q1
