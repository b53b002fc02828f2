"""CUDA path vs CPU oracle, through the C ABI, on seeded workloads.

Quantised payloads and scales must match bit for bit; attention outputs must
be within 1e-4 max-abs and 1e-3 relative (max norm) of the oracle's fp64
result on the same
quantised inputs.  Sizes span several tiles and ragged tails; the full-size
workloads are checked on sampled (sequence, kv head) units.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from int8_quantized_kv_gb300 import kvq8
from int8_quantized_kv_gb300 import workloads as wl
from kvq8_harness import Case, SM_SCALE, assert_close, k_rows_logical, v_rows_logical

pytestmark = pytest.mark.gpu
HD = 128


def _unit_cfg(G, nkv=2, batch=1, ctx=None, ctx_range=None, cid=100, outliers=0):
    return wl.Workload(f"test_g{G}", cid, batch=batch, nqh=G * nkv, nkv=nkv, ctx=ctx,
                       ctx_range=ctx_range, outlier_channels=outliers)


# ------------------------------------------------------------ quantisation ---
def test_quantize_q_bit_exact(gpu_lib):
    rng = np.random.default_rng(0)
    rows = [rng.standard_normal(HD).astype(np.float32) * s for s in (1.0, 1e-3, 50.0)]
    z = np.zeros(HD, np.float32)
    z[32:64] = 4e-7
    z[64] = np.float32(1e-6)
    z[96] = np.nextafter(np.float32(1e-6), np.float32(0))
    rows.append(z)
    t = np.zeros(HD, np.float32)
    t[:8] = [127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5]
    t[32:38] = [63.5, 1.25, 1.75, -1.25, 0.25, -63.5]
    rows.append(t)
    rows += list(rng.standard_normal((2000, HD)).astype(np.float32))
    x = np.stack(rows)
    xd = torch.from_numpy(x).cuda()
    codes = torch.empty(x.shape, dtype=torch.int8, device="cuda")
    scales = torch.empty((len(x), 4), dtype=torch.float32, device="cuda")
    kvq8.quantize_q(xd, codes, scales)
    torch.cuda.synchronize()
    qi, qsc = oracle.q_quantize_blocks(x)
    assert np.array_equal(codes.cpu().numpy(), qi)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), qsc.view(np.uint32))


def _kv_rows_special():
    rng = np.random.default_rng(1)
    rows = []
    a = np.zeros(HD, np.float32)
    a[:13] = [127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5, -1.5, 126.5, -126.5, 0.25, -0.75]
    rows.append(a)
    b = np.zeros(HD, np.float32)
    b[:9] = [254.0, 5.0, 7.0, -5.0, 1.0, 3.0, -3.0, 253.0, -9.0]
    rows.append(b)
    rows.append(np.zeros(HD, np.float32))                    # all-zero row: scale 0
    d = np.zeros(HD, np.float32)
    d[:4] = [1e-40, -5e-41, 2e-41, -1e-40]                   # subnormal scale
    rows.append(d)
    rows.append(rng.standard_normal(HD).astype(np.float32) * np.float32(1e30))
    rows.append(rng.standard_normal(HD).astype(np.float32) * np.float32(1e-30))
    return np.stack(rows)


@pytest.mark.parametrize("start,n_new", [(0, 1), (0, 256), (37, 300), (255, 2), (0, 1000), (480, 33)])
def test_quantize_append_bit_exact(gpu_lib, start, n_new):
    nkv = 3
    rng = np.random.default_rng(start * 7919 + n_new)
    k = rng.standard_normal((2, n_new, nkv, HD)).astype(np.float32)
    v = (rng.standard_normal((2, n_new, nkv, HD)) * 3.0).astype(np.float32)
    sp = _kv_rows_special()
    m = min(len(sp), n_new)
    k[0, :m, 0] = sp[:m]
    v[1, :m, nkv - 1] = sp[::-1][:m]
    need = (start + n_new + 255) // 256
    max_blocks = need + 1
    num_blocks = 2 * max_blocks + 2
    perm = np.random.default_rng(5).permutation(num_blocks).astype(np.int32)
    table = perm[:2 * max_blocks].reshape(2, max_blocks)
    cache = kvq8.alloc_cache(num_blocks, nkv)
    for t in cache:
        t.fill_(0x55 if t.dtype == torch.int8 else 7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq8.quantize_append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                         torch.tensor([start, start], dtype=torch.int32, device="cuda"),
                         torch.from_numpy(table).cuda(), cache, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    kp, vp = cache.k_pool.cpu().numpy(), cache.v_pool.cpu().numpy()
    ksp, vsp = cache.k_scale.cpu().numpy(), cache.v_scale.cpu().numpy()
    pos = start + np.arange(n_new)
    for b in range(2):
        phys, slot = table[b, pos // 256], pos % 256
        for h in range(nkv):
            kq, ks = oracle.kv_quantize_rows(k[b, :, h])
            vq, vs = oracle.kv_quantize_rows(v[b, :, h])
            assert np.array_equal(k_rows_logical(kp, phys, h, slot), kq)
            assert np.array_equal(v_rows_logical(vp, phys, h, slot), vq)
            assert np.array_equal(ksp[phys, h, slot].view(np.uint32), ks.view(np.uint32))
            assert np.array_equal(vsp[phys, h, slot].view(np.uint32), vs.view(np.uint32))
    # slots outside the appended range are untouched
    written = np.zeros((num_blocks, nkv, 256), bool)
    for b in range(2):
        written[table[b, pos // 256], :, pos % 256] = True
    assert np.all(ksp[~written] == 7.0)
    assert np.all(kp.transpose(0, 1, 2, 3)[~written] == 0x55)


def _near_half_rows(n_rows, seed):
    """Rows whose quotients v / scale sit within a few ulps of half-integers:
    row max m (so scale = m/127 in fp32), then values fl((k + 0.5) * scale)
    moved by -3..3 ulps.  Multiplying by the rounded reciprocal instead of
    dividing rounds some of these to the other integer."""
    rng = np.random.default_rng(seed)
    rows = np.empty((n_rows, HD), np.float32)
    for i in range(n_rows):
        m = np.float32(rng.uniform(0.3, 700.0))
        sc = m / np.float32(127.0)
        k = rng.integers(-126, 126, HD).astype(np.float32)
        v = ((k + np.float32(0.5)) * sc).astype(np.float32)
        for j, steps in enumerate(rng.integers(-3, 4, HD)):
            for _ in range(abs(int(steps))):
                v[j] = np.nextafter(v[j], np.float32(np.inf if steps > 0 else -np.inf))
        v[rng.integers(HD)] = m if rng.random() < 0.5 else -m
        rows[i] = v
    return rows


def _multiply_rounds_differently(rows):
    """How many values of the rows a plain v * (1/scale) would code differently
    from round_half_even(fl(v / scale))."""
    m = np.abs(rows).max(axis=1, keepdims=True)
    sc = (m / np.float32(127.0)).astype(np.float32)
    inv = (np.float32(1.0) / sc).astype(np.float32)
    return int(np.sum(np.rint(rows * inv) != np.rint(rows / sc)))


@pytest.mark.parametrize("n_new", [1, 64, 200])
def test_quantize_append_quotients_near_half_integers(gpu_lib, n_new):
    """K/V codes stay bit-exact where the quotient is within ulps of a rounding
    boundary: the kernels multiply by the reciprocal only where that provably
    rounds like the division, and divide elsewhere."""
    batch, nkv = (48, 2) if n_new == 1 else (2, 2)
    rows = _near_half_rows(batch * n_new * nkv * 2, seed=n_new)
    assert _multiply_rounds_differently(rows) > 0
    k = rows[: batch * n_new * nkv].reshape(batch, n_new, nkv, HD)
    v = rows[batch * n_new * nkv:].reshape(batch, n_new, nkv, HD)
    max_blocks = (n_new + 255) // 256
    table = np.arange(batch * max_blocks, dtype=np.int32).reshape(batch, max_blocks)
    cache = kvq8.alloc_cache(batch * max_blocks, nkv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq8.quantize_append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                         torch.zeros(batch, dtype=torch.int32, device="cuda"),
                         torch.from_numpy(table).cuda(), cache, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    kp, vp = cache.k_pool.cpu().numpy(), cache.v_pool.cpu().numpy()
    pos = np.arange(n_new)
    for b in range(batch):
        phys, slot = table[b, pos // 256], pos % 256
        for h in range(nkv):
            kq, _ = oracle.kv_quantize_rows(k[b, :, h])
            vq, _ = oracle.kv_quantize_rows(v[b, :, h])
            assert np.array_equal(k_rows_logical(kp, phys, h, slot), kq), (b, h)
            assert np.array_equal(v_rows_logical(vp, phys, h, slot), vq), (b, h)


def test_byte_count_of_allocated_cache(gpu_lib):
    # 2112 bytes per token per layer for 8 kv heads of 128 ([Day 9-1] §2)
    nb = 5
    cache = kvq8.alloc_cache(nb, 8)
    total = sum(t.numel() * t.element_size() for t in cache)
    assert total == nb * 256 * 2112 == nb * 256 * kvq8.cache_bytes_per_token(8)


# ------------------------------------------------------------------ decode ---
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_decode_group_sizes(gpu_lib, G):
    cfg = _unit_cfg(G, nkv=2, batch=3, ctx_range=(1, 1300), cid=110 + G)
    case = Case(cfg)
    out = case.decode()
    for b in range(cfg.batch):
        for h in range(cfg.nkv):
            ref = case.oracle_unit(b, h)
            assert_close(out[b, h * G:(h + 1) * G], ref, f"G={G} b={b} h={h}")
    assert case.status_bits() == 0


@pytest.mark.parametrize("L", [1, 2, 31, 32, 33, 255, 256, 257, 511, 513, 4097])
def test_decode_lengths(gpu_lib, L):
    cfg = _unit_cfg(4, nkv=1, batch=1, ctx=L, cid=120)
    case = Case(cfg)
    out = case.decode()
    assert_close(out[0], case.oracle_unit(0, 0), f"L={L}")


def test_decode_multi_block_splits(gpu_lib):
    # enough units x blocks that a split spans several cache blocks
    cfg = _unit_cfg(1, nkv=8, batch=8, ctx_range=(6000, 10000), cid=125)
    case = Case(cfg)
    out = case.decode()
    for b in range(cfg.batch):
        for h in range(cfg.nkv):
            assert_close(out[b, h:h + 1], case.oracle_unit(b, h), f"b={b} h={h}")


def test_decode_zero_length_sequences(gpu_lib):
    cfg = _unit_cfg(2, nkv=2, batch=4, ctx_range=(1, 700), cid=130)
    lens = np.array([0, 300, 0, 650], np.int32)
    case = Case(cfg, lens=lens)
    out = case.decode()
    assert not out[0].any() and not out[2].any()
    for b in (1, 3):
        for h in range(2):
            assert_close(out[b, h * 2:(h + 1) * 2], case.oracle_unit(b, h))


def test_decode_two_ctas_per_sm_ragged(gpu_lib):
    # G = 2 over 32 units and a 47-block table: the split runs two CTAs per SM
    # (6-stage rings); ragged lengths, an empty and a one-token sequence
    cfg = _unit_cfg(2, nkv=8, batch=4, ctx_range=(1, 12000), cid=135)
    lens = np.array([0, 11900, 1, 7777], np.int32)
    case = Case(cfg, lens=lens)
    out = case.decode()
    assert not out[0].any()
    for b in (1, 2, 3):
        for h in range(cfg.nkv):
            assert_close(out[b, h * 2:(h + 1) * 2], case.oracle_unit(b, h), f"b={b} h={h}")
    assert case.status_bits() == 0


def test_single_head_l256_and_fp32_kv_delta(gpu_lib):
    cfg = wl.SINGLE_HEAD_L256
    case = Case(cfg)
    out = case.decode()
    ref = case.oracle_unit(0, 0)
    assert_close(out[0], ref, "single head L=256")
    # The page's experiment: the fp32-KV output vs the q8 output.
    k, v = wl.unit_kv(cfg, 0, 0)
    f32 = oracle.attention_f64(case.q[0, 0], k, v, SM_SCALE)
    d = np.abs(out[0, 0] - f32)
    assert d.max() < 0.05 and d.mean() > 1e-5


def test_decode_sm_scale_argument(gpu_lib):
    cfg = _unit_cfg(2, nkv=1, batch=1, ctx=700, cid=140)
    case = Case(cfg)
    out = case.decode(sm_scale=0.3)
    assert_close(out[0], case.oracle_unit(0, 0, sm_scale=np.float32(0.3)))


def test_decode_on_side_stream_matches(gpu_lib):
    cfg = _unit_cfg(4, nkv=2, batch=2, ctx=900, cid=150)
    case = Case(cfg)
    ref = case.decode()
    s = torch.cuda.Stream()
    out = torch.empty_like(case.q_d)
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, case.max_blocks)
    with torch.cuda.stream(s):
        kvq8.decode_attn(case.q_d, case.cache, case.table_d, case.lens_d, out, ws)
    s.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref)


def test_split_and_combine_equal_decode_attn(gpu_lib):
    cfg = _unit_cfg(8, nkv=2, batch=2, ctx_range=(100, 3000), cid=160)
    case = Case(cfg)
    ref = case.decode()
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, case.max_blocks)
    out = torch.empty_like(case.q_d)
    kvq8.decode_split(case.q_d, case.cache, case.table_d, case.lens_d, ws)
    kvq8.decode_combine(cfg.batch, cfg.nqh, cfg.nkv, case.max_blocks, case.lens_d, ws, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref)


def test_cache_filled_in_small_appends_matches_one_append(gpu_lib):
    cfg = _unit_cfg(2, nkv=2, batch=2, ctx_range=(300, 900), cid=170)
    a = Case(cfg)
    b = Case(cfg, append_chunk=77)
    pa, pb = a.host_pools(), b.host_pools()   # unwritten slots are uninitialised: compare tokens
    for bb in range(cfg.batch):
        for h in range(cfg.nkv):
            for x, y in zip(a.gather_unit(pa, bb, h), b.gather_unit(pb, bb, h)):
                assert np.array_equal(x, y)
    assert np.array_equal(a.decode(), b.decode())


# ------------------------------------------------------- device-side faults ---
def test_bad_block_id_is_flagged_and_skipped(gpu_lib):
    cfg = _unit_cfg(2, nkv=1, batch=1, ctx=1000, cid=180)
    case = Case(cfg)
    good = case.table[0, 1]
    case.table_d[0, 1] = case.num_blocks + 5          # logical block 1 now out of range
    out = case.decode()
    assert case.status_bits() & kvq8.DEV_BAD_BLOCK_ID
    # the kernel skips the 256 tokens of that block: same as the oracle without them
    k, v = wl.unit_kv(cfg, 0, 0)
    keep = np.r_[0:256, 512:1000]
    ref, _ = oracle.decode_unit_q8(case.q[0], k[keep], v[keep], SM_SCALE)
    assert_close(out[0], ref)
    case.table_d[0, 1] = int(good)


def test_bad_ctx_len_is_flagged_and_clamped(gpu_lib):
    cfg = _unit_cfg(1, nkv=1, batch=1, ctx=512, cid=190)
    case = Case(cfg, spare_blocks=0)
    case.lens_d[0] = case.max_blocks * 256 + 10
    out = case.decode()
    assert case.status_bits() & kvq8.DEV_BAD_CTX_LEN
    assert_close(out[0], case.oracle_unit(0, 0))


def test_bounded_wait_gives_up_and_the_context_stays_usable(gpu_lib):
    # the decode kernels' wait routine on a barrier phase that nothing completes:
    # it must give up after its bound, flag the timeout and return
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    kvq8.selftest_bounded_wait(2_000_000, status, waited)
    torch.cuda.synchronize()
    assert status.item() == kvq8.DEV_TIMEOUT
    assert 2_000_000 <= waited.item() < 1_000_000_000
    # the context still works: a decode right after it matches the oracle
    cfg = _unit_cfg(2, nkv=2, batch=1, ctx=700, cid=195)
    case = Case(cfg)
    out = case.decode()
    assert case.status_bits() == 0
    for h in range(cfg.nkv):
        assert_close(out[0, 2 * h:2 * h + 2], case.oracle_unit(0, h))


def test_append_bad_position_is_flagged(gpu_lib):
    nkv = 1
    cache = kvq8.alloc_cache(2, nkv)
    cache.k_scale.fill_(3.0)
    table = torch.tensor([[0, 1]], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = torch.randn(1, 4, nkv, HD, device="cuda")
    kvq8.quantize_append(k, k, torch.tensor([510], dtype=torch.int32, device="cuda"), table, cache,
                         dev_status=status)
    torch.cuda.synchronize()
    assert status.item() & kvq8.DEV_BAD_POSITION
    ks = cache.k_scale.cpu().numpy()
    # positions 510, 511 land in block 1 slots 254, 255; 512, 513 are past the table
    assert ks[1, 0, 254] != 3.0 and ks[1, 0, 255] != 3.0 and ks[1, 0, 253] == 3.0
    assert np.all(ks[0] == 3.0)


def test_host_errors_on_device(gpu_lib):
    cfg = _unit_cfg(2, nkv=1, batch=1, ctx=300, cid=200)
    case = Case(cfg)
    out = torch.empty_like(case.q_d)
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq8.Kvq8Error) as e:
        kvq8.decode_attn(case.q_d, case.cache, case.table_d, case.lens_d, out, small)
    assert e.value.status == kvq8.ERR_WORKSPACE


# --------------------------------------------------- the specified workloads ---
SMALL = [
    wl.scaled(wl.QWEN3_2B_28L_8K, batch=4, ctx=1500),
    wl.scaled(wl.BATCH64_RAGGED, batch=6, ctx_range=(512, 2600)),
    wl.scaled(wl.LONG128K_OUTLIERS, batch=2, ctx=3000),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_specified_workloads_scaled_all_outputs(gpu_lib, cfg):
    case = Case(cfg)
    out = case.decode()
    G = cfg.group
    for b in range(cfg.batch):
        for h in range(cfg.nkv):
            assert_close(out[b, h * G:(h + 1) * G], case.oracle_unit(b, h), f"{cfg.name} b={b} h={h}")


FULL = [wl.QWEN3_2B_28L_8K, wl.BATCH64_RAGGED, wl.LONG128K_OUTLIERS]


@pytest.mark.slow
@pytest.mark.parametrize("cfg", FULL, ids=lambda c: c.name)
def test_specified_workloads_full_size_sampled(gpu_lib, cfg):
    case = Case(cfg, spare_blocks=0)
    out = case.decode()
    assert case.status_bits() == 0
    assert np.all(np.isfinite(out))
    rng = np.random.default_rng(cfg.config_id)
    G = cfg.group
    units = {(int(rng.integers(cfg.batch)), int(rng.integers(cfg.nkv))) for _ in range(6)}
    units.add((cfg.batch - 1, cfg.nkv - 1))
    for b, h in sorted(units):
        assert_close(out[b, h * G:(h + 1) * G], case.oracle_unit(b, h), f"{cfg.name} b={b} h={h}")
    # every appended token of a sampled unit is bit-exact too
    pools = case.host_pools()
    b, h = sorted(units)[0]
    kq, ks, vq, vs = case.gather_unit(pools, b, h)
    k, v = wl.unit_kv(cfg, b, h)
    okq, oks = oracle.kv_quantize_rows(k)
    ovq, ovs = oracle.kv_quantize_rows(v)
    assert np.array_equal(kq, okq) and np.array_equal(vq, ovq)
    assert np.array_equal(ks, oks) and np.array_equal(vs, ovs)


# ------------------------------------------------------ fused decode step ---
from kvq8_harness import StepCase  # noqa: E402


def _check_step(case, out):
    cfg = case.cfg
    G = cfg.group
    pools = case.host_pools()
    for b in range(cfg.batch):
        L = int(case.lens[b])
        if L == 0:
            assert not out[b].any()
            continue
        for h in range(cfg.nkv):
            assert_close(out[b, h * G:(h + 1) * G], case.oracle_unit(b, h), f"step b={b} h={h} L={L}")
            kq, ks, vq, vs = case.gather_unit(pools, b, h)       # the appended token is bit-exact
            okq, oks = oracle.kv_quantize_rows(case.k_new[b, h][None])
            ovq, ovs = oracle.kv_quantize_rows(case.v_new[b, h][None])
            assert np.array_equal(kq[L - 1], okq[0]) and np.array_equal(vq[L - 1], ovq[0])
            assert ks[L - 1] == oks[0] and vs[L - 1] == ovs[0]


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_decode_step_group_sizes(gpu_lib, G):
    cfg = _unit_cfg(G, nkv=2, batch=4, ctx_range=(1, 1500), cid=400 + G)
    lens = wl.ctx_lens(cfg).copy()
    lens[0] = 1                                    # the new token is the whole context
    case = StepCase(cfg, lens=lens)
    out = case.step()
    _check_step(case, out)
    assert case.status_bits() == 0


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 255, 256, 257, 4097])
def test_decode_step_token_positions(gpu_lib, L):
    cfg = _unit_cfg(2, nkv=1, batch=1, ctx=L, cid=410)
    case = StepCase(cfg)
    _check_step(case, case.step())


def test_decode_step_empty_sequences_and_ragged_batch(gpu_lib):
    cfg = _unit_cfg(4, nkv=2, batch=5, ctx_range=(1, 900), cid=420)
    lens = np.array([0, 700, 0, 1, 333], np.int32)
    case = StepCase(cfg, lens=lens)
    _check_step(case, case.step())


def test_decode_step_two_ctas_per_sm(gpu_lib):
    # the decode step on the two-CTAs-per-SM grid (G = 2, 32 units, 47 blocks)
    cfg = _unit_cfg(2, nkv=8, batch=4, ctx_range=(1, 12000), cid=425)
    lens = np.array([11900, 1, 0, 5000], np.int32)
    case = StepCase(cfg, lens=lens)
    _check_step(case, case.step())
    assert case.status_bits() == 0


def test_decode_step_unit_over_many_ctas(gpu_lib):
    # one long unit spread over most CTAs: the last CTA to finish merges them all
    cfg = _unit_cfg(8, nkv=1, batch=1, ctx=30001, cid=430)
    case = StepCase(cfg)
    _check_step(case, case.step())


def test_decode_step_twice_on_one_workspace(gpu_lib):
    cfg = wl.scaled(wl.QWEN3_2B_28L_8K, batch=6, ctx=2500)
    case = StepCase(cfg)
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, case.max_blocks)
    first = case.step(ws)
    second = case.step(ws)          # appending the same token again: identical results
    assert np.array_equal(first, second)
    _check_step(case, second)


def _chain(call, q0, n, sync_between):
    """n calls, each taking the previous call's output as its query."""
    outs, x = [], q0
    for _ in range(n):
        o = torch.full_like(q0, float("nan"))
        call(x, o)
        if sync_between:
            torch.cuda.synchronize()
        outs.append(o)
        x = o
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in outs]


def test_output_fed_back_as_query_without_sync(gpu_lib):
    """The combine lets the next kernel launch early, and the decode and the
    step launch as programmatic dependents: a call that reads, as its query,
    the output the call just before it is still writing must see that output
    complete (the same results as with a full synchronisation in between)."""
    cfg = wl.scaled(wl.BATCH64_RAGGED, batch=6, ctx_range=(300, 5000))
    case = StepCase(cfg)
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, case.max_blocks)

    def attn(x, o):
        kvq8.decode_attn(x, case.cache, case.table_d, case.lens_d, o, ws, dev_status=case.status)

    def step(x, o):
        kvq8.decode_step(x, case.k_new_d, case.v_new_d, case.cache, case.table_d, case.lens_d, o, ws,
                         dev_status=case.status)

    def step_ready(x, o):
        # the cache, table and lengths are final before each call's preceding
        # kernel begins (only the query comes from it): the flagged step still
        # waits for its query
        kvq8.decode_step(x, case.k_new_d, case.v_new_d, case.cache, case.table_d, case.lens_d, o, ws,
                         dev_status=case.status, cache_ready=True)

    step(case.q_d, torch.empty_like(case.q_d))   # the appended token is in place from here on
    for call in (attn, step, step_ready):
        fast = _chain(call, case.q_d, 6, sync_between=False)
        slow = _chain(call, case.q_d, 6, sync_between=True)
        for a, b in zip(fast, slow):
            assert np.isfinite(a).all()
            assert np.array_equal(a, b)
    assert case.status_bits() == 0


def test_decode_step_cache_ready_flag_gives_identical_results(gpu_lib):
    # KVQ8_STEP_CACHE_READY only lets the split kernel start copying earlier
    cfg = wl.scaled(wl.BATCH64_RAGGED, batch=7, ctx_range=(1, 6000))
    a, b = StepCase(cfg), StepCase(cfg)
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, a.max_blocks)
    plain = a.step(ws)
    out = torch.full_like(b.q_d, float("nan"))
    kvq8.decode_step(b.q_d, b.k_new_d, b.v_new_d, b.cache, b.table_d, b.lens_d, out, ws,
                     dev_status=b.status, cache_ready=True)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), plain)
    pa, pb = a.host_pools(), b.host_pools()
    for bb in range(cfg.batch):
        for h in range(cfg.nkv):
            for x, y in zip(a.gather_unit(pa, bb, h), b.gather_unit(pb, bb, h)):
                assert np.array_equal(x, y)
    _check_step(b, out.cpu().numpy())
    assert b.status_bits() == 0


@pytest.mark.parametrize("cache_ready", [False, True])
def test_per_layer_step_calls_in_a_graph(gpu_lib, cache_ready):
    """A decode that runs one layer per call: 28 kvq8_decode_step calls at batch
    1 (one per layer of the Qwen3-2B stack, each with its own workspace, all in
    one pool), captured in a CUDA graph and replayed twice; every layer's output
    against the oracle, and the flagged chain against the plain one bit for bit."""
    cfg = wl.scaled(wl.QWEN3_2B_28L_8K, ctx=1500)
    case = StepCase(cfg)
    layers = cfg.batch
    wss = [kvq8.alloc_workspace(1, cfg.nqh, cfg.nkv, case.max_blocks) for _ in range(layers)]
    outs = torch.full_like(case.q_d, float("nan"))
    s = torch.cuda.Stream()

    def calls():
        for l in range(layers):
            kvq8.decode_step(case.q_d[l:l + 1], case.k_new_d[l:l + 1], case.v_new_d[l:l + 1], case.cache,
                             case.table_d[l:l + 1], case.lens_d[l:l + 1], outs[l:l + 1], wss[l],
                             dev_status=case.status, stream=s, cache_ready=cache_ready)

    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        calls()
    s.synchronize()
    first = outs.cpu().numpy()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls()
    outs.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    got = outs.cpu().numpy()
    assert np.array_equal(got, first)
    assert case.status_bits() == 0
    _check_step(case, got)


def test_decode_step_equals_append_then_decode(gpu_lib):
    cfg = wl.scaled(wl.BATCH64_RAGGED, batch=5, ctx_range=(512, 3000))
    a = StepCase(cfg)
    fused = a.step()
    b = StepCase(cfg)
    start = torch.from_numpy((b.lens - 1).astype(np.int32)).cuda()
    kvq8.quantize_append(b.k_new_d[:, None], b.v_new_d[:, None], start, b.table_d, b.cache)
    two_call = b.decode()
    assert_close(fused, two_call, "fused step vs append + decode_attn")
    pa, pb = a.host_pools(), b.host_pools()
    for bb in range(cfg.batch):
        for h in range(cfg.nkv):
            for x, y in zip(a.gather_unit(pa, bb, h), b.gather_unit(pb, bb, h)):
                assert np.array_equal(x, y)


@pytest.mark.parametrize("pinned", [True, False])
def test_decode_step_host_buffers_equal_device_call(gpu_lib, pinned):
    """kvq8_decode_step_host (host q and new rows in, host result out) gives the
    device call's results bit for bit, pools included, and the oracle's: with
    page-locked buffers (read and written by the kernels themselves) and with
    pageable ones (copied through the device buffers)."""
    cfg = wl.scaled(wl.QWEN3_2B_28L_8K, batch=3, ctx=1300)
    a = StepCase(cfg)
    dev_out = a.step()
    b = StepCase(cfg)
    host = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    q_h = host(torch.from_numpy(wl.queries(cfg)))
    k_h = host(torch.from_numpy(b.k_new))
    v_h = host(torch.from_numpy(b.v_new))
    out_h = host(torch.full(tuple(q_h.shape), float("nan")))
    assert q_h.is_pinned() == pinned and out_h.is_pinned() == pinned
    q_d, k_d, v_d = torch.zeros_like(b.q_d), torch.zeros_like(b.k_new_d), torch.zeros_like(b.v_new_d)
    out_d = torch.empty_like(b.q_d)
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, b.max_blocks)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()          # the cache was filled on the default stream
    kvq8.decode_step_host(q_h, k_h, v_h, out_h, q_d, k_d, v_d, b.cache, b.table_d, b.lens_d, out_d, ws,
                          sm_scale=SM_SCALE, dev_status=b.status, stream=stream)
    stream.synchronize()
    assert b.status.item() == 0
    assert np.array_equal(out_h.numpy(), dev_out)
    pa, pb = a.host_pools(), b.host_pools()
    for bb in range(cfg.batch):
        for h in range(cfg.nkv):
            for x, y in zip(a.gather_unit(pa, bb, h), b.gather_unit(pb, bb, h)):
                assert np.array_equal(x, y)
    _check_step(b, out_h.numpy())


def test_decode_attn_on_host_mapped_buffers(gpu_lib):
    """decode_attn reading the query from and writing the result to page-locked
    host memory (kvq8.HostMapped) equals the device call bit for bit."""
    cfg = _unit_cfg(4, nkv=2, batch=3, ctx_range=(100, 3000), cid=470)
    case = Case(cfg)
    dev_out = case.decode()
    q_h = torch.from_numpy(case.q).pin_memory()
    out_h = torch.full(tuple(q_h.shape), float("nan")).pin_memory()
    ws = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, case.max_blocks)
    kvq8.decode_attn(kvq8.HostMapped(q_h), case.cache, case.table_d, case.lens_d, kvq8.HostMapped(out_h), ws,
                     sm_scale=SM_SCALE, dev_status=case.status)
    torch.cuda.synchronize()
    assert case.status_bits() == 0
    assert np.array_equal(out_h.numpy(), dev_out)


def test_host_device_pointer(gpu_lib):
    """kvq8_host_device_pointer: a device address for page-locked host memory
    (16-byte aligned there), NULL for pageable, device or misaligned memory."""
    lib = kvq8.load()
    pinned = torch.zeros(64).pin_memory()
    addr = lib.kvq8_host_device_pointer(pinned.data_ptr())
    assert addr is not None and addr % 16 == 0
    assert lib.kvq8_host_device_pointer(pinned.data_ptr() + 4) is None
    assert lib.kvq8_host_device_pointer(torch.zeros(64).data_ptr()) is None
    assert lib.kvq8_host_device_pointer(torch.zeros(64, device="cuda").data_ptr()) is None
    assert lib.kvq8_host_device_pointer(None) is None


@pytest.mark.parametrize("pinned", [True, False])
def test_bound_decode_step_equals_the_calls(gpu_lib, pinned):
    """kvq8.DecodeStep (arguments checked and converted once): run() gives
    kvq8_decode_step's results and run_host() those of the host-buffer call,
    bit for bit, over several steps with the inputs refilled in between."""
    cfg = wl.scaled(wl.QWEN3_2B_28L_8K, batch=3, ctx=1300)
    a = StepCase(cfg)
    b = StepCase(cfg)
    host = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    q_h = host(torch.from_numpy(wl.queries(cfg)))
    k_h = host(torch.from_numpy(b.k_new))
    v_h = host(torch.from_numpy(b.v_new))
    out_h = host(torch.full(tuple(q_h.shape), float("nan")))
    q_d, k_d, v_d = torch.zeros_like(b.q_d), torch.zeros_like(b.k_new_d), torch.zeros_like(b.v_new_d)
    out_d = torch.empty_like(b.q_d)
    ws_a = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, a.max_blocks)
    ws_b = kvq8.alloc_workspace(cfg.batch, cfg.nqh, cfg.nkv, b.max_blocks)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    dev_step = kvq8.DecodeStep(a.q_d, a.k_new_d, a.v_new_d, a.cache, a.table_d, a.lens_d, out_d, ws_a,
                               sm_scale=SM_SCALE, dev_status=a.status, stream=stream)
    host_step = kvq8.DecodeStep(q_d, k_d, v_d, b.cache, b.table_d, b.lens_d, torch.empty_like(out_d), ws_b,
                                sm_scale=SM_SCALE, dev_status=b.status, stream=stream,
                                q_host=q_h, k_host=k_h, v_host=v_h, out_host=out_h)
    assert host_step.host_direct == pinned
    rng = np.random.default_rng(7)
    for it in range(3):
        qn = rng.standard_normal(tuple(q_h.shape)).astype(np.float32)
        q_h.copy_(torch.from_numpy(qn))
        a.q_d.copy_(torch.from_numpy(qn))
        torch.cuda.synchronize()
        dev_step.run()
        host_step.run_host()
        stream.synchronize()
        assert np.array_equal(out_h.numpy(), out_d.cpu().numpy()), f"step {it}"
        ref = out_d.cpu().numpy().copy()
        kvq8.decode_step(a.q_d, a.k_new_d, a.v_new_d, a.cache, a.table_d, a.lens_d, out_d, ws_a,
                         sm_scale=SM_SCALE, dev_status=a.status, stream=stream)
        stream.synchronize()
        assert np.array_equal(ref, out_d.cpu().numpy())
    assert a.status.item() == 0 and b.status.item() == 0
    pa, pb = a.host_pools(), b.host_pools()
    for bb in range(cfg.batch):
        for h in range(cfg.nkv):
            for x, y in zip(a.gather_unit(pa, bb, h), b.gather_unit(pb, bb, h)):
                assert np.array_equal(x, y)


def test_quantize_append_host_buffers_equal_device_call(gpu_lib):
    nkv, n_new, batch = 2, 300, 2
    rng = np.random.default_rng(77)
    k = rng.standard_normal((batch, n_new, nkv, HD)).astype(np.float32)
    v = (rng.standard_normal((batch, n_new, nkv, HD)) * 2).astype(np.float32)
    table = np.arange(2 * batch, dtype=np.int32).reshape(batch, 2)
    start = torch.tensor([5, 100], dtype=torch.int32, device="cuda")
    td = torch.from_numpy(table).cuda()
    c1, c2 = kvq8.alloc_cache(2 * batch, nkv), kvq8.alloc_cache(2 * batch, nkv)
    for c in (c1, c2):
        for t in c:
            t.zero_()
    kvq8.quantize_append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), start, td, c1)
    k_stage, v_stage = torch.empty(k.shape, device="cuda"), torch.empty(v.shape, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    kvq8.quantize_append_host(torch.from_numpy(k).pin_memory(), torch.from_numpy(v).pin_memory(),
                              k_stage, v_stage, start, td, c2, stream=stream)
    stream.synchronize()
    for x, y in zip(c1, c2):
        assert torch.equal(x, y)


@pytest.mark.slow
def test_decode_step_full_size_qwen3_2b(gpu_lib):
    cfg = wl.QWEN3_2B_28L_8K
    case = StepCase(cfg, spare_blocks=0)
    out = case.step()
    rng = np.random.default_rng(5)
    G = cfg.group
    for b, h in {(int(rng.integers(cfg.batch)), int(rng.integers(cfg.nkv))) for _ in range(5)}:
        assert_close(out[b, h * G:(h + 1) * G], case.oracle_unit(b, h), f"full step b={b} h={h}")
    assert case.status_bits() == 0
