"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

Nothing here retypes the oracle's formulas: each check is an invariant the
pages state (half-step error, one scale per row, amplitude invariance, byte
count, single pass == three pass), a hand-worked fixture under
tests/golden/, a closed form or special case, brute force on tiny inputs, or
a library routine (torch's scaled_dot_product_attention in fp64) that must
agree with the oracle where the method reduces to it.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from int8_quantized_kv_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
HD = 128
SM = np.float32(1.0 / math.sqrt(128.0))


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rows(seed, n, scale=1.0, hd=HD):
    return (np.random.default_rng(seed).standard_normal((n, hd)) * scale).astype(np.float32)


# ---------------------------------------------------------------------------
# K/V per-(token, head) quantisation
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("amp", [1.0, 1e-3, 37.0, 1e4])
def test_kv_error_at_most_half_step(amp):
    # Day 9-3 §3: each dequantised value is off by at most half a step (= scale/2).
    x = _rows(1, 500, amp)
    q, s = oracle.kv_quantize_rows(x)
    err = np.abs(q.astype(np.float64) * s[:, None].astype(np.float64) - x.astype(np.float64))
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 1e-5))
    assert q.min() >= -127 and q.max() <= 127


def test_kv_max_abs_element_maps_to_pm127_and_scale_is_step():
    x = _rows(2, 300, 3.0)
    q, s = oracle.kv_quantize_rows(x)
    idx = np.argmax(np.abs(x), axis=1)
    top = q[np.arange(len(x)), idx]
    assert np.array_equal(top, np.where(x[np.arange(len(x)), idx] > 0, 127, -127))
    m = np.abs(x).max(axis=1).astype(np.float64)
    # scale * 127 reproduces max_abs to fp32 precision (one step = max_abs/127)
    assert np.all(np.abs(s.astype(np.float64) * 127.0 - m) <= m * 2.0 ** -22)


def test_kv_round_half_even_fixture():
    g = _golden("kv_round_half_even_rows.json")
    for row in g["kv_rows"]:
        x = np.zeros(HD, np.float32)
        x[:len(row["values"])] = row["values"]
        q, s = oracle.kv_quantize_rows(x[None])
        assert s[0] == np.float32(row["scale"])
        want = np.zeros(HD, np.int8)
        want[:len(row["codes"])] = row["codes"]
        assert np.array_equal(q[0], want)


def test_kv_zero_row_and_sign_symmetry():
    x = np.zeros((1, HD), np.float32)
    q, s = oracle.kv_quantize_rows(x)
    assert s[0] == 0.0 and not q.any()
    y = _rows(3, 50)
    qa, sa = oracle.kv_quantize_rows(y)
    qb, sb = oracle.kv_quantize_rows(-y)
    assert np.array_equal(qa, -qb) and np.array_equal(sa, sb)


def test_kv_one_scale_per_row_rows_independent():
    # Day 9-3 §4 B / Day 9-1 §2: one scale per (token, head) row of 128 values.
    x = _rows(4, 64)
    q0, s0 = oracle.kv_quantize_rows(x)
    x2 = x.copy()
    x2[7] *= 1000.0
    q1, s1 = oracle.kv_quantize_rows(x2)
    keep = np.arange(64) != 7
    assert np.array_equal(q0[keep], q1[keep]) and np.array_equal(s0[keep], s1[keep])
    assert s0.shape == (64,)


def test_kv_brute_force_nearest_code_tiny():
    # Brute force: the code is the integer in [-127, 127] nearest to v/scale
    # (exact rational arithmetic); only near-ties may differ by the fp32 quotient.
    x = _rows(5, 6)
    q, s = oracle.kv_quantize_rows(x)
    for r in range(len(x)):
        sc = Fraction(float(s[r]))
        for i in range(HD):
            t = Fraction(float(x[r, i])) / sc
            best = min(range(-127, 128), key=lambda c: (abs(t - c), c % 2))
            if abs(abs(t - math.floor(t)) - Fraction(1, 2)) > Fraction(1, 10 ** 5):
                assert q[r, i] == best


def test_kv_amplitude_x3_invariance():
    # Day 9-3 §4 A: scaling K/V by 3 scales the step, relative error unchanged.
    x = _rows(6, 2000)
    q1, s1 = oracle.kv_quantize_rows(x)
    q3, s3 = oracle.kv_quantize_rows(np.float32(3.0) * x)
    mismatch = np.count_nonzero(q1 != q3)
    assert mismatch <= 1e-4 * q1.size
    assert np.all(np.abs(s3.astype(np.float64) / s1 - 3.0) <= 3 * 2.0 ** -22)


def test_kv_denormal_row_clamps():
    # Degenerate case: max_abs so small that max_abs/127 is subnormal; the clamp
    # keeps every code in [-127, 127] and the largest element at full scale.
    x = np.zeros((1, HD), np.float32)
    x[0, :4] = [1e-40, -5e-41, 2e-41, -1e-40]
    q, s = oracle.kv_quantize_rows(x)
    assert 0.0 < s[0] < np.finfo(np.float32).tiny
    assert q.min() >= -127 and q.max() <= 127
    assert q[0, 0] == 127 and q[0, 3] == -127


def test_byte_count_2112_per_token_layer():
    # Day 9-1 §2: 8 kv heads x 128: int8 K+V 2048 B + 8 heads x 2 fp32 scales = 2112 B.
    g = _golden("day9_1_byte_count.json")
    x = _rows(7, 2 * g["nkv"], hd=g["hd"])  # one token: K rows then V rows of 8 heads
    q, s = oracle.kv_quantize_rows(x)
    assert q.nbytes == g["q8_payload_bytes"]
    assert s.nbytes == g["q8_scale_bytes"]
    assert q.nbytes + s.nbytes == g["q8_bytes_per_token_layer"]
    assert g["nkv"] * g["hd"] * 2 * 2 == g["f16_bytes_per_token_layer"]
    assert round((q.nbytes + s.nbytes) / g["f16_bytes_per_token_layer"], 2) == g["ratio_q8_over_f16_rounded"]


# ---------------------------------------------------------------------------
# Q quantisation in 32-element blocks
# ---------------------------------------------------------------------------
def test_q_round_half_even_fixture():
    g = _golden("kv_round_half_even_rows.json")
    for blk in g["q_blocks"]:
        x = np.zeros(HD, np.float32)
        x[:len(blk["values"])] = blk["values"]
        qi, qsc = oracle.q_quantize_blocks(x)
        assert qsc[0] == np.float32(blk["block_scale"])
        want = np.zeros(32, np.int8)
        want[:len(blk["codes"])] = blk["codes"]
        assert np.array_equal(qi[:32], want)
        assert not qi[32:].any()


def test_q_block_max_and_error_bound():
    x = _rows(8, 40, 2.0).reshape(-1)
    qi, qsc = oracle.q_quantize_blocks(x)
    xb = x.reshape(-1, 32)
    qb = qi.reshape(-1, 32)
    i = np.argmax(np.abs(xb), axis=1)
    assert np.array_equal(np.abs(qb[np.arange(len(xb)), i]), np.full(len(xb), 127))
    err = np.abs(qb.astype(np.float64) * qsc[:, None] - xb)
    assert np.all(err <= qsc[:, None].astype(np.float64) * (0.5 + 1e-5))


def test_q_zero_and_tiny_blocks_use_unit_max():
    # Day 9-2 §2 segment 1: a block whose max is below 1e-6 is quantised as if max were 1.
    x = np.zeros(HD, np.float32)
    x[32:64] = 4e-7
    x[64] = np.float32(1e-6)       # exactly at the threshold: not replaced
    x[96] = np.nextafter(np.float32(1e-6), np.float32(0))
    qi, qsc = oracle.q_quantize_blocks(x)
    inv127 = np.float32(1.0) / np.float32(127.0)
    assert qsc[0] == inv127 and not qi[:32].any()
    assert qsc[1] == inv127 and not qi[32:64].any()   # 4e-7 * 127 rounds to 0
    assert qsc[2] == np.float32(1e-6) * inv127 and qi[64] == 127
    assert qsc[3] == inv127 and qi[96] == 0


def test_q_blocks_independent():
    x = _rows(9, 1).reshape(-1)
    a, sa = oracle.q_quantize_blocks(x)
    y = x.copy()
    y[64:96] *= 50.0
    b, sb = oracle.q_quantize_blocks(y)
    assert np.array_equal(a[:64], b[:64]) and np.array_equal(a[96:], b[96:])
    assert sa[0] == sb[0] and sa[1] == sb[1] and sa[3] == sb[3]


# ---------------------------------------------------------------------------
# scores and the two decode forms
# ---------------------------------------------------------------------------
def test_scores_block_dots_brute_force():
    rng = np.random.default_rng(10)
    qi = rng.integers(-128, 128, HD).astype(np.int8)
    kq = rng.integers(-127, 128, (9, HD)).astype(np.int8)
    qsc = np.array([1.0, 2.0, 4.0, 8.0], np.float32)   # powers of two: exact in fp64
    ks = np.ones(9, np.float32)
    s = oracle.scores_q8(qi, qsc, kq, ks, 1.0)
    for t in range(9):
        want = sum(int(qsc[b]) * sum(int(qi[i]) * int(kq[t, i]) for i in range(32 * b, 32 * b + 32))
                   for b in range(4))
        assert s[t] == want
    ks2 = np.full(9, 0.5, np.float32)
    assert np.array_equal(oracle.scores_q8(qi, qsc, kq, ks2, 0.25), s * 0.125)


def _random_unit(seed, L, G=1):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((L, HD)).astype(np.float32)
    v = rng.standard_normal((L, HD)).astype(np.float32)
    q = rng.standard_normal((G, HD)).astype(np.float32)
    return q, k, v


def test_three_pass_weights_sum_to_one():
    q, k, v = _random_unit(11, 300)
    kq, ks = oracle.kv_quantize_rows(k)
    vq, vs = oracle.kv_quantize_rows(v)
    qi, qsc = oracle.q_quantize_blocks(q[0])
    _, w = oracle.decode_q8_three_pass(qi, qsc, kq, ks, vq, vs, SM, want_weights=True)
    assert abs(w.sum() - 1.0) < 1e-12 and np.all(w > 0)


@pytest.mark.parametrize("L", [1, 2, 3, 5, 8, 300])
def test_online_single_pass_equals_three_pass(L):
    # Day 9-2 §3: the single pass and the three-pass form are functionally equal.
    q, k, v = _random_unit(12 + L, L)
    kq, ks = oracle.kv_quantize_rows(k * np.float32(2.5))
    vq, vs = oracle.kv_quantize_rows(v)
    qi, qsc = oracle.q_quantize_blocks(q[0] * np.float32(3.0))
    a = oracle.decode_q8_three_pass(qi, qsc, kq, ks, vq, vs, SM)
    b = oracle.decode_q8_online(qi, qsc, kq, ks, vq, vs, SM)
    assert np.max(np.abs(a - b)) < 1e-12


def test_length_one_returns_dequantised_v():
    q, k, v = _random_unit(13, 1)
    kq, ks = oracle.kv_quantize_rows(k)
    vq, vs = oracle.kv_quantize_rows(v)
    qi, qsc = oracle.q_quantize_blocks(q[0])
    out = oracle.decode_q8_three_pass(qi, qsc, kq, ks, vq, vs, SM)
    assert np.array_equal(out, vq[0].astype(np.float64) * np.float64(vs[0]))


def test_identical_keys_give_mean_of_v():
    q, k, v = _random_unit(14, 40)
    k[:] = k[0]
    kq, ks = oracle.kv_quantize_rows(k)
    vq, vs = oracle.kv_quantize_rows(v)
    qi, qsc = oracle.q_quantize_blocks(q[0])
    out = oracle.decode_q8_three_pass(qi, qsc, kq, ks, vq, vs, SM)
    mean = (vq.astype(np.float64) * vs[:, None]).mean(axis=0)
    assert np.max(np.abs(out - mean)) < 1e-13


def test_dominant_score_selects_its_row():
    q, k, v = _random_unit(15, 50)
    k[17] = q[0] * np.float32(40.0)   # score ~ 40*|q|^2/sqrt(128): all others negligible
    kq, ks = oracle.kv_quantize_rows(k)
    vq, vs = oracle.kv_quantize_rows(v)
    qi, qsc = oracle.q_quantize_blocks(q[0])
    out = oracle.decode_q8_three_pass(qi, qsc, kq, ks, vq, vs, SM)
    assert np.max(np.abs(out - vq[17] * np.float64(vs[17]))) < 1e-12


def _sdpa64(q, k, v, scale):
    """torch's fused attention in fp64: q [H][hd], k/v [Hk][L][hd] with GQA by
    repeating each kv head over its group of consecutive query heads."""
    H = q.shape[0]
    G = H // k.shape[0]
    kk = torch.from_numpy(np.asarray(k, np.float64)).repeat_interleave(G, dim=0)
    vv = torch.from_numpy(np.asarray(v, np.float64)).repeat_interleave(G, dim=0)
    qq = torch.from_numpy(np.asarray(q, np.float64))[:, None, :]
    o = torch.nn.functional.scaled_dot_product_attention(qq[None], kk[None], vv[None], scale=float(scale))
    return o[0, :, 0, :].numpy()


def test_q8_path_equals_library_attention_on_exact_codes():
    # Integer-valued rows whose max is 127 quantise exactly (scale 1), so the
    # q8 method must equal plain softmax attention on those integers.
    rng = np.random.default_rng(16)
    L = 77
    def exact_rows(n):
        x = rng.integers(-126, 127, (n, HD)).astype(np.float32)
        x[np.arange(n), rng.integers(0, HD, n)] = 127.0
        return x
    k, v = exact_rows(L), exact_rows(L)
    q = rng.integers(-126, 127, HD).astype(np.float32)
    q[[3, 40, 70, 100]] = [127.0, -127.0, 127.0, 127.0]  # one per 32-block
    kq, ks = oracle.kv_quantize_rows(k)
    vq, vs = oracle.kv_quantize_rows(v)
    qi, qsc = oracle.q_quantize_blocks(q)
    assert np.all(ks == 1.0) and np.all(vs == 1.0) and np.all(qsc == 1.0)
    out = oracle.decode_q8_three_pass(qi, qsc, kq, ks, vq, vs, SM)
    ref = _sdpa64(q[None], k[None], v[None], float(SM))[0]
    assert np.max(np.abs(out - ref)) <= 1e-9 * max(1.0, np.abs(ref).max())


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_unit_driver_equals_library_attention_on_dequantised_inputs(G):
    # The method's score sum_b dot_b*qsc_b*ks*scale is, in exact arithmetic, the
    # dot of the dequantised Q and K; so the whole q8 path equals fp64 softmax
    # attention over dequantised Q/K/V, with query head j reading kv head j // G.
    nkv = 2
    rng = np.random.default_rng(17 + G)
    L = 190
    q = rng.standard_normal((nkv * G, HD)).astype(np.float32)
    k = rng.standard_normal((nkv, L, HD)).astype(np.float32)
    v = rng.standard_normal((nkv, L, HD)).astype(np.float32) * np.float32(2.0)
    outs, deq_q, deq_k, deq_v = [], [], [], []
    for h in range(nkv):
        o, qz = oracle.decode_unit_q8(q[h * G:(h + 1) * G], k[h], v[h], SM)
        outs.append(o)
        deq_q.append(qz["qi"].astype(np.float64) *
                     np.repeat(qz["qsc"].astype(np.float64), 32, axis=-1))
        deq_k.append(qz["kq"].astype(np.float64) * qz["ks"][:, None])
        deq_v.append(qz["vq"].astype(np.float64) * qz["vs"][:, None])
    out = np.concatenate(outs)
    ref = _sdpa64(np.concatenate(deq_q), np.stack(deq_k), np.stack(deq_v), float(SM))
    assert np.max(np.abs(out - ref)) < 1e-12


def test_empty_context_gives_zero():
    out = oracle.decode_q8_three_pass(np.zeros(HD, np.int8), np.ones(4, np.float32),
                                      np.zeros((0, HD), np.int8), np.zeros(0, np.float32),
                                      np.zeros((0, HD), np.int8), np.zeros(0, np.float32), SM)
    assert not out.any()


# ---------------------------------------------------------------------------
# fp32 attention and the fp32-KV vs q8-KV experiment (Day 9-3 §1-§3)
# ---------------------------------------------------------------------------
def test_attention_f64_equals_library():
    q, k, v = _random_unit(18, 123)
    out = oracle.attention_f64(q[0], k, v, SM)
    ref = _sdpa64(q, k[None], v[None], float(SM))[0]
    assert np.max(np.abs(out - ref)) < 1e-13


def test_fp32_kv_vs_q8_kv_delta_order():
    # Day 9-3 §3 reports max|d_out| 0.0125, mean 0.0086 on its own ~N(0,1)
    # generator (not reproducible: parity unpinned).  On true N(0,1) the delta is
    # smaller; what is pinned is the page's reading of it: the error comes from
    # the step (mean|d| below half an average step) and stays well under the
    # output magnitude.  The measured values are recorded with the design notes.
    cfg = wl.SINGLE_HEAD_L256
    k, v = wl.unit_kv(cfg, 0, 0)
    q = wl.queries(cfg)[0, 0]
    ref = oracle.attention_f64(q, k, v, SM)
    kq, ks = oracle.kv_quantize_rows(k)
    vq, vs = oracle.kv_quantize_rows(v)
    deq = oracle.attention_f64(q, oracle.kv_dequantize_rows(kq, ks),
                               oracle.kv_dequantize_rows(vq, vs), SM)
    d = np.abs(deq - ref)
    half_step = 0.5 * float(np.mean(ks))
    assert 1e-5 < d.mean() < half_step
    assert d.max() < 0.05 and d.max() < 0.5 * np.abs(ref).max()
    # x3 amplitude on V alone scales the output delta exactly by 3 (Day 9-3 §4 A)
    vq3, vs3 = oracle.kv_quantize_rows(np.float32(3.0) * v)
    deq3 = oracle.attention_f64(q, oracle.kv_dequantize_rows(kq, ks),
                                oracle.kv_dequantize_rows(vq3, vs3), SM)
    ref3 = oracle.attention_f64(q, k, np.float32(3.0) * v, SM)
    d3 = np.abs(deq3 - ref3)
    assert abs(d3.mean() / d.mean() - 3.0) < 0.05


# ---------------------------------------------------------------------------
# asymmetric INT4 group-64 quantisation (UltraQuant §3.2)
# ---------------------------------------------------------------------------
def _int4_fixture_row(g):
    row = np.full(HD, g["row_fill_group0"], np.float32)
    row[:len(g["row_head"])] = g["row_head"]
    row[64:] = g["row_group1_constant"]
    return row


def test_int4_hand_example():
    g = _golden("int4_group64_hand_example.json")
    row = _int4_fixture_row(g)
    packed, scale, zero = oracle.int4_quantize_groups(row, g["group"])
    assert np.array_equal(scale, np.array(g["scale"], np.float32))
    assert np.array_equal(zero, np.array(g["zero"], np.float32))
    want = np.full(64, g["packed_fill_group0"], np.uint8)
    want[:len(g["packed_head"])] = g["packed_head"]
    want[32:] = g["packed_group1"]
    assert np.array_equal(packed, want)
    deq = oracle.int4_dequantize_groups(packed, scale, zero, g["group"])
    assert np.all(deq[64:] == np.float32(g["dequant_group1"]))
    codes = np.array(g["codes_head"])
    assert np.allclose(deq[:len(codes)], (codes - 5) * 0.3, atol=1e-6)


def test_int4_error_bound_and_ranges():
    x = _rows(19, 50, 2.0)
    packed, scale, zero = oracle.int4_quantize_groups(x, 64)
    deq = oracle.int4_dequantize_groups(packed, scale, zero, 64)
    err = np.abs(deq.astype(np.float64) - x).reshape(-1, 64)
    sc = scale.reshape(-1).astype(np.float64)
    assert np.all(err <= sc[:, None] * (0.5 + 1e-4))
    z = zero.reshape(-1)
    assert np.all((z >= 0) & (z <= 15))          # min <= 0 <= max here, so zero in [0, 15]
    hi, lo = packed >> 4, packed & 15
    assert hi.max() <= 15 and lo.max() <= 15


def test_int4_nibble_order_high_first():
    x = np.zeros(64, np.float32)
    x[0], x[1] = 1.0, 0.0    # group min 0, max 1: scale 1/15, zero 0; codes 15 and 0
    packed, scale, zero = oracle.int4_quantize_groups(x, 64)
    assert zero[0] == 0.0 and packed[0] == 0xF0 and not packed[1:].any()


def test_int4_round_half_even_ties():
    # [UltraQuant] §3.2 rounds with torch.round (half to even).  Group 0: min 0,
    # max 15 -> scale exactly 1, zero 0, so each code is round(x) and x = k + 0.5
    # is a tie; group 1: min -2.5, max 12.5 -> scale 1 and zero = round(2.5) = 2,
    # then code = round(x + 2).  Half away from zero would give 1, 2, 3, 4, 14,
    # 15 and zero 3.
    x = np.full(128, 7.0, np.float32)
    x[:8] = [0.0, 15.0, 0.5, 1.5, 2.5, 3.5, 13.5, 14.5]
    x[64:70] = [-2.5, 12.5, 0.5, -1.5, 1.5, 10.5]
    packed, scale, zero = oracle.int4_quantize_groups(x, 64)
    assert scale.tolist() == [1.0, 1.0] and zero.tolist() == [0.0, 2.0]
    codes = np.stack([packed >> 4, packed & 15], axis=1).reshape(-1)
    assert codes[:8].tolist() == [0, 15, 0, 2, 2, 4, 14, 14]
    assert codes[64:70].tolist() == [0, 14, 2, 0, 4, 12]    # rne(-0.5), rne(14.5), rne(2.5), rne(0.5), rne(3.5), rne(12.5)
    assert np.all(codes[8:64] == 7) and np.all(codes[70:] == 9)


def test_int4_codes_are_the_nearest_clamped_integers():
    # brute force in exact rational arithmetic on the stored fp32 scale and zero:
    # the code is the integer nearest to x/scale + zero (ties to even), clamped
    # to [0, 15]; values within 1e-5 of a half-integer are left out (there the
    # fp32 rounding of x/scale may decide either way)
    from fractions import Fraction
    x = _rows(23, 12, 3.0)
    packed, scale, zero = oracle.int4_quantize_groups(x, 64)
    codes = np.stack([packed >> 4, packed & 15], axis=-1).reshape(x.shape)
    checked = 0
    for r in range(x.shape[0]):
        for gi in range(2):
            s, z = Fraction(float(scale[r, gi])), Fraction(float(zero[r, gi]))
            for d in range(64 * gi, 64 * gi + 64):
                t = Fraction(float(x[r, d])) / s + z
                fl = t.numerator // t.denominator
                frac = t - fl
                if abs(frac - Fraction(1, 2)) < Fraction(1, 100000):
                    continue
                want = min(15, max(0, fl + (1 if frac > Fraction(1, 2) else 0)))
                assert codes[r, d] == want, (r, d, float(t))
                checked += 1
    assert checked > 0.99 * x.size


# ---------------------------------------------------------------------------
# mixed precision by token age (UltraQuant §3.3): old blocks 4-bit, recent int8
# ---------------------------------------------------------------------------
def test_mixed_with_no_old_tokens_is_the_q8_path():
    q, k, v = _random_unit(31, 700, G=2)
    mixed = oracle.decode_mixed_unit(q, k, v, 0, SM)
    ref, _ = oracle.decode_unit_q8(q, k, v, SM)
    assert np.max(np.abs(mixed - ref)) < 1e-15


def test_mixed_with_only_old_tokens_is_attention_over_requantised_rows():
    q, k, v = _random_unit(32, 512, G=2)
    kq, ks = oracle.kv_quantize_rows(k)
    vq, vs = oracle.kv_quantize_rows(v)
    k4 = oracle.int4_dequantize_groups(*oracle.int4_quantize_groups(oracle.kv_dequantize_rows(kq, ks)))
    v4 = oracle.int4_dequantize_groups(*oracle.int4_quantize_groups(oracle.kv_dequantize_rows(vq, vs)))
    mixed = oracle.decode_mixed_unit(q, k, v, 512, SM)
    ref = _sdpa64(q, k4[None], v4[None], float(SM))
    assert np.max(np.abs(mixed - ref)) < 1e-12


@pytest.mark.parametrize("n4", [256, 512, 768])
def test_mixed_equals_one_softmax_over_both_parts(n4):
    # an independent route with torch in fp64: the old tokens' logits from the
    # fp32 query and the requantised rows, the recent tokens' logits from the
    # dequantised query blocks and int8 rows (equal, exactly, to the integer
    # block dots times their scales); one softmax over the concatenation
    q, k, v = _random_unit(33, 1000, G=2)
    kq, ks = oracle.kv_quantize_rows(k)
    vq, vs = oracle.kv_quantize_rows(v)
    qi, qsc = oracle.q_quantize_blocks(q)
    T = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    k4 = oracle.int4_dequantize_groups(*oracle.int4_quantize_groups(oracle.kv_dequantize_rows(kq[:n4], ks[:n4])))
    v4 = oracle.int4_dequantize_groups(*oracle.int4_quantize_groups(oracle.kv_dequantize_rows(vq[:n4], vs[:n4])))
    qdeq = T(qi) * T(np.repeat(qsc, 32, axis=1))
    k8 = T(kq[n4:]) * T(ks[n4:])[:, None]
    v8 = T(vq[n4:]) * T(vs[n4:])[:, None]
    logits = torch.cat([T(q) @ T(k4).T, qdeq @ k8.T], dim=1) * float(SM)
    w = torch.softmax(logits, dim=1)
    ref = (w @ torch.cat([T(v4), v8], dim=0)).numpy()
    mixed = oracle.decode_mixed_unit(q, k, v, n4, SM)
    assert np.max(np.abs(mixed - ref)) < 1e-12


def test_requantised_rows_stay_within_both_half_steps():
    x = _rows(34, 200, 3.0)
    kq, ks = oracle.kv_quantize_rows(x)
    packed, sc, zr = oracle.requantize_q8_to_q4(kq, ks)
    y = oracle.int4_dequantize_groups(packed, sc, zr)
    bound = 0.5 * ks[:, None] * 1.0001 + 0.5 * np.repeat(sc, 64, axis=1) * 1.0001
    assert np.all(np.abs(y.astype(np.float64) - x) <= bound)


# --------------------------------------------------------------------------
# Non-finite inputs.  The pages give every rule for finite values only; the
# reading taken is that a unit of quantisation (K/V row, query 32-block, INT4
# group) holding a NaN or an infinity is quantised exactly as if all its
# values were zero.  Pinned to the closed forms of the zero unit.
# --------------------------------------------------------------------------
_NONFINITE = (np.nan, np.inf, -np.inf)


def test_nonfinite_kv_rows_quantise_as_the_zero_row():
    rng = np.random.default_rng(41)
    x = rng.standard_normal((7, 128)).astype(np.float32)
    bad = {1: (5, np.nan), 3: (0, np.inf), 4: (127, -np.inf), 6: (64, np.nan)}
    for r, (i, val) in bad.items():
        x[r, i] = val
    x[6, 65] = np.inf                       # two non-finite values in one row
    q, s, n = oracle.kv_quantize_rows(x, count_nonfinite=True)
    assert n == len(bad)
    for r in bad:
        # the zero row: max |v| = 0, scale +0, every code 0
        assert s[r].view(np.uint32) == 0 and not q[r].any()
    for r in (0, 2, 5):
        # finite rows keep the page's rule: the max-abs element maps to +-127,
        # scale = max|v| / 127 in fp32
        m = np.abs(x[r]).max()
        assert s[r] == np.float32(m) / np.float32(127.0)
        assert abs(int(q[r][np.argmax(np.abs(x[r]))])) == 127
    _, _, n_clean = oracle.kv_quantize_rows(x[[0, 2, 5]], count_nonfinite=True)
    assert n_clean == 0


def test_nonfinite_query_blocks_quantise_as_the_zero_block():
    rng = np.random.default_rng(42)
    x = rng.standard_normal((3, 128)).astype(np.float32)
    x[0, 40] = np.nan        # block 1 of row 0
    x[2, 127] = np.inf       # block 3 of row 2
    x[2, 0] = -np.inf        # block 0 of row 2
    qi, qsc, n = oracle.q_quantize_blocks(x, count_nonfinite=True)
    assert n == 3
    inv = np.float32(1.0) * np.float32(1.0 / 127.0)   # qm = 0 < 1e-6 -> 1
    for r, blk in ((0, 1), (2, 3), (2, 0)):
        assert qsc[r, blk] == inv and not qi[r, 32 * blk:32 * blk + 32].any()
    # the other blocks are untouched: block max -> +-127 and scale max/127
    for r, blk in ((0, 0), (0, 2), (1, 1), (2, 1)):
        b = x[r, 32 * blk:32 * blk + 32]
        assert qsc[r, blk] == np.float32(np.abs(b).max()) * np.float32(1.0 / 127.0)
        assert abs(int(qi[r, 32 * blk + np.argmax(np.abs(b))])) == 127


def test_nonfinite_int4_groups_quantise_as_the_zero_group():
    rng = np.random.default_rng(43)
    x = rng.standard_normal((4, 128)).astype(np.float32)
    x[0, 3] = np.nan          # group 0 of row 0
    x[1, 100] = np.inf        # group 1 of row 1
    x[3, 0] = -np.inf
    x[3, 127] = np.nan        # both groups of row 3
    packed, sc, zr, n = oracle.int4_quantize_groups(x, 64, count_nonfinite=True)
    assert n == 4
    neg_zero = np.float32(-0.0).view(np.uint32)
    for r, g in ((0, 0), (1, 1), (3, 0), (3, 1)):
        # the zero group: max == min -> scale 1; zero = round(-0 / 1) = -0; codes 0
        assert sc[r, g] == 1.0 and zr[r, g].view(np.uint32) == neg_zero
        assert not packed[r, 32 * g:32 * g + 32].any()
    for r, g in ((0, 1), (1, 0), (2, 0), (2, 1)):
        grp = x[r, 64 * g:64 * g + 64]
        assert sc[r, g] == (np.float32(grp.max()) - np.float32(grp.min())) / np.float32(15.0)


@pytest.mark.parametrize("val", _NONFINITE)
def test_nonfinite_rows_give_a_finite_decode(val):
    # a context with a non-finite K row and a non-finite V row decodes like the
    # same context with those rows zero (the zero K row scores 0, the zero V
    # row adds nothing), and the output is finite
    q, k, v = _random_unit(44, 300, G=2)
    k_bad, v_bad = k.copy(), v.copy()
    k_bad[17, 9] = val
    v_bad[200, 100] = val
    out, _ = oracle.decode_unit_q8(q, k_bad, v_bad, SM)
    k0, v0 = k.copy(), v.copy()
    k0[17] = 0.0
    v0[200] = 0.0
    ref, _ = oracle.decode_unit_q8(q, k0, v0, SM)
    assert np.all(np.isfinite(out)) and np.array_equal(out, ref)
