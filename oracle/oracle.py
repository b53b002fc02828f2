"""ctypes front of the C oracle (``kvq8_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use this
module.  It never imports the CUDA package, and the CUDA package never
imports it.

All arithmetic is in the C file; this module only marshals numpy arrays and
runs per-unit drivers (one unit = one sequence x one kv head with its G query
heads), in the order the pages give: quantise K/V rows, quantise Q in
32-blocks, then the three-pass decode in fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq8_oracle.c")
_HDR = os.path.join(_HERE, "kvq8_oracle.h")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
           "-fPIC", "-shared", "-Wall"]

_lib = None
_lock = threading.Lock()


def build_oracle(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH) or force or
             os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                                os.path.getmtime(_HDR)))
    if stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build_oracle())
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int
        f32 = ctypes.c_float
        sig = {
            "orc_kv_quantize_rows": (i64, [P, i64, i32, P, P]),
            "orc_kv_dequantize_rows": (None, [P, P, i64, i32, P]),
            "orc_q_quantize_blocks": (i64, [P, i64, P, P]),
            "orc_scores_q8": (None, [P, P, i32, P, P, i64, f32, P]),
            "orc_decode_q8_three_pass": (i32, [P, P, i32, P, P, P, P, i64, f32, P, P]),
            "orc_decode_q8_online": (i32, [P, P, i32, P, P, P, P, i64, f32, P]),
            "orc_attention_f64": (i32, [P, P, P, i64, i32, f32, P]),
            "orc_int4_quantize_groups": (i64, [P, i64, i32, P, P, P]),
            "orc_int4_dequantize_groups": (None, [P, P, P, i64, i32, P]),
            "orc_decode_mixed": (i32, [P, P, P, i32, P, P, i64, P, P, P, P, i64, f32, P]),
            "orc_version": (i32, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# element-level wrappers
# --------------------------------------------------------------------------
def kv_quantize_rows(x, count_nonfinite=False):
    """Per-row max-abs INT8 quantisation. x: float32 [..., hd] -> (int8 [..., hd], float32 [...]),
    plus the number of rows quantised as zeros for holding a NaN or an infinity
    when count_nonfinite."""
    x = _c(x, np.float32)
    hd = x.shape[-1]
    n = x.size // hd if hd else 0
    q = np.empty(x.shape, np.int8)
    s = np.empty(x.shape[:-1], np.float32)
    replaced = 0
    if n:
        replaced = int(_load().orc_kv_quantize_rows(_p(x), n, hd, _p(q), _p(s)))
    return (q, s, replaced) if count_nonfinite else (q, s)


def kv_dequantize_rows(q, scale):
    q = _c(q, np.int8)
    scale = _c(scale, np.float32)
    hd = q.shape[-1]
    out = np.empty(q.shape, np.float32)
    n = q.size // hd if hd else 0
    if n:
        _load().orc_kv_dequantize_rows(_p(q), _p(scale), n, hd, _p(out))
    return out


def q_quantize_blocks(x, count_nonfinite=False):
    """32-block Q quantisation. x: float32 [..., hd] -> (int8 [..., hd], float32 [..., hd/32]),
    plus the number of blocks quantised as zeros for holding a NaN or an
    infinity when count_nonfinite."""
    x = _c(x, np.float32)
    hd = x.shape[-1]
    assert hd % 32 == 0
    qi = np.empty(x.shape, np.int8)
    qsc = np.empty(x.shape[:-1] + (hd // 32,), np.float32)
    replaced = 0
    if x.size:
        replaced = int(_load().orc_q_quantize_blocks(_p(x), x.size, _p(qi), _p(qsc)))
    return (qi, qsc, replaced) if count_nonfinite else (qi, qsc)


def scores_q8(qi, qsc, kq, ks, sm_scale):
    qi, qsc = _c(qi, np.int8), _c(qsc, np.float32)
    kq, ks = _c(kq, np.int8), _c(ks, np.float32)
    L, hd = kq.shape
    s = np.empty(L, np.float64)
    if L:
        _load().orc_scores_q8(_p(qi), _p(qsc), hd, _p(kq), _p(ks), L,
                              float(sm_scale), _p(s))
    return s


def decode_q8_three_pass(qi, qsc, kq, ks, vq, vs, sm_scale, want_weights=False):
    """One query head over [L][hd] int8 K/V rows; returns fp64 [hd] (and weights)."""
    qi, qsc = _c(qi, np.int8), _c(qsc, np.float32)
    kq, ks = _c(kq, np.int8), _c(ks, np.float32)
    vq, vs = _c(vq, np.int8), _c(vs, np.float32)
    L, hd = kq.shape
    out = np.empty(hd, np.float64)
    w = np.empty(max(L, 1), np.float64) if want_weights else None
    rc = _load().orc_decode_q8_three_pass(
        _p(qi), _p(qsc), hd, _p(kq), _p(ks), _p(vq), _p(vs), L,
        float(sm_scale), _p(out), _p(w) if w is not None else None)
    if rc != 0:
        raise MemoryError("oracle scratch allocation failed")
    if want_weights:
        return out, w[:L]
    return out


def decode_q8_online(qi, qsc, kq, ks, vq, vs, sm_scale):
    qi, qsc = _c(qi, np.int8), _c(qsc, np.float32)
    kq, ks = _c(kq, np.int8), _c(ks, np.float32)
    vq, vs = _c(vq, np.int8), _c(vs, np.float32)
    L, hd = kq.shape
    out = np.empty(hd, np.float64)
    rc = _load().orc_decode_q8_online(_p(qi), _p(qsc), hd, _p(kq), _p(ks),
                                      _p(vq), _p(vs), L, float(sm_scale), _p(out))
    if rc != 0:
        raise MemoryError("oracle scratch allocation failed")
    return out


def attention_f64(q, k, v, sm_scale):
    """Plain softmax attention of one float query over float [L][hd] K/V, fp64."""
    q, k, v = _c(q, np.float32), _c(k, np.float32), _c(v, np.float32)
    L, hd = k.shape
    out = np.empty(hd, np.float64)
    rc = _load().orc_attention_f64(_p(q), _p(k), _p(v), L, hd,
                                   float(sm_scale), _p(out))
    if rc != 0:
        raise MemoryError("oracle scratch allocation failed")
    return out


def int4_quantize_groups(x, group=64, count_nonfinite=False):
    """Asymmetric INT4 per-group quantisation; returns (packed uint8, scale, zero),
    plus the number of groups quantised as zeros for holding a NaN or an
    infinity when count_nonfinite."""
    x = _c(x, np.float32)
    n = x.size
    assert n % group == 0 and group % 2 == 0
    packed = np.empty(x.shape[:-1] + (x.shape[-1] // 2,), np.uint8)
    ng = n // group
    scale = np.empty(x.shape[:-1] + (x.shape[-1] // group,), np.float32)
    zero = np.empty_like(scale)
    replaced = 0
    if n:
        replaced = int(_load().orc_int4_quantize_groups(_p(x), n, group, _p(packed),
                                                        _p(scale), _p(zero)))
    assert scale.size == ng and replaced >= 0
    return (packed, scale, zero, replaced) if count_nonfinite else (packed, scale, zero)


def int4_dequantize_groups(packed, scale, zero, group=64):
    packed = _c(packed, np.uint8)
    scale, zero = _c(scale, np.float32), _c(zero, np.float32)
    shape = packed.shape[:-1] + (packed.shape[-1] * 2,)
    out = np.empty(shape, np.float32)
    n = out.size
    if n:
        _load().orc_int4_dequantize_groups(_p(packed), _p(scale), _p(zero), n,
                                           group, _p(out))
    return out


# --------------------------------------------------------------------------
# per-unit drivers
# --------------------------------------------------------------------------
def decode_unit_q8(q_heads, k_rows, v_rows, sm_scale):
    """The q8 path for one (sequence, kv head), following the pages' order.

    q_heads: float32 [G][hd] (the query heads that read this kv head)
    k_rows, v_rows: float32 [L][hd] (the unit's context, fp32 before quantisation)
    Returns (out fp64 [G][hd], dict of the quantised intermediates).
    """
    kq, ks = kv_quantize_rows(k_rows)
    vq, vs = kv_quantize_rows(v_rows)
    qi, qsc = q_quantize_blocks(q_heads)
    G, hd = q_heads.shape
    out = np.empty((G, hd), np.float64)
    for g in range(G):
        out[g] = decode_q8_three_pass(qi[g], qsc[g], kq, ks, vq, vs, sm_scale)
    return out, dict(kq=kq, ks=ks, vq=vq, vs=vs, qi=qi, qsc=qsc)


def decode_quantized_unit(qi, qsc, kq, ks, vq, vs, sm_scale):
    """Three-pass decode of G already-quantised query heads against one kv head."""
    G, hd = qi.shape
    out = np.empty((G, hd), np.float64)
    for g in range(G):
        out[g] = decode_q8_three_pass(qi[g], qsc[g], kq, ks, vq, vs, sm_scale)
    return out


def requantize_q8_to_q4(kq, ks, group=64):
    """An int8 row's dequantised values requantised by the INT4 group rule
    ([UltraQuant] §3.3: the oldest time blocks go from 8-bit to 4-bit).
    Returns (packed, scale, zero)."""
    return int4_quantize_groups(kv_dequantize_rows(kq, ks), group)


def decode_mixed_unit(q_heads, k_rows, v_rows, n4, sm_scale):
    """Mixed precision by token age for one (sequence, kv head): every token
    is first cached as int8; the first n4 tokens (the old time blocks) are then
    requantised to INT4 group-64; the decode reads the old tokens as 4-bit and
    the recent ones as int8 (orc_decode_mixed).  Returns out fp64 [G][hd]."""
    kq, ks = kv_quantize_rows(k_rows)
    vq, vs = kv_quantize_rows(v_rows)
    qi, qsc = q_quantize_blocks(q_heads)
    n4 = int(n4)
    k4 = int4_dequantize_groups(*requantize_q8_to_q4(kq[:n4], ks[:n4]))
    v4 = int4_dequantize_groups(*requantize_q8_to_q4(vq[:n4], vs[:n4]))
    G, hd = q_heads.shape
    q_heads = _c(q_heads, np.float32)
    k4, v4 = _c(k4, np.float32), _c(v4, np.float32)
    kr, ksr = _c(kq[n4:], np.int8), _c(ks[n4:], np.float32)
    vr, vsr = _c(vq[n4:], np.int8), _c(vs[n4:], np.float32)
    out = np.empty((G, hd), np.float64)
    for g in range(G):
        row = np.empty(hd, np.float64)
        qg, qig, qscg = _c(q_heads[g], np.float32), _c(qi[g], np.int8), _c(qsc[g], np.float32)
        rc = _load().orc_decode_mixed(_p(qg), _p(qig), _p(qscg), hd, _p(k4), _p(v4), n4,
                                      _p(kr), _p(ksr), _p(vr), _p(vsr), len(kr), float(sm_scale),
                                      _p(row))
        assert rc == 0
        out[g] = row
    return out


def run_parallel(fn, items, threads: int):
    """Map fn over items on `threads` host threads (the C calls drop the GIL)."""
    if threads <= 1:
        return [fn(it) for it in items]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items))


def version() -> int:
    return int(_load().orc_version())
