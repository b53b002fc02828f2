"""Host-side checks of libkvq8: it builds for sm_103a, loads, exports every
symbol include/kvq8.h declares, and its pure-host logic (sizes, argument
validation) behaves as documented.  No call here reaches a kernel launch:
every compute call below fails validation first, so this runs without a GPU.
"""
import ctypes
import os
import re

import pytest

from int8_quantized_kv_gb300 import build as kbuild
from int8_quantized_kv_gb300 import kvq8

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq8.h")
FAKE = 1 << 20   # a 256-aligned non-null address that is never dereferenced


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kv(?:q8|q4|f32|mix)_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kvq8.load()


def test_header_declares_expected_entry_points():
    names = _declared()
    for n in ("kvq8_quantize_append", "kvq8_quantize_q", "kvq8_decode_attn",
              "kvq8_decode_split", "kvq8_decode_combine", "kvq8_decode_workspace_bytes",
              "kvq8_decode_step", "kvq8_decode_attn_noalloc", "kvq4_quantize_append",
              "kvq4_decode_attn", "kvf32_append", "kvf32_decode_attn", "kvmix_requantize",
              "kvmix_decode_attn", "kvmix_decode_workspace_bytes", "kvq8_decode_step_host",
              "kvq8_quantize_append_host", "kvq8_selftest_bounded_wait"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) <= set(kvq8.SIGNATURES)


def test_binding_does_not_import_oracle():
    import sys
    import subprocess
    code = ("import sys; import int8_quantized_kv_gb300.kvq8 as k; "
            "import int8_quantized_kv_gb300.workloads; "
            "assert not any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules)")
    subprocess.run([sys.executable, "-c", code], cwd=ROOT, check=True)


def test_status_strings(lib):
    assert kvq8.status_str(0) == "KVQ8_OK"
    assert kvq8.status_str(kvq8.ERR_WORKSPACE) == "KVQ8_ERR_WORKSPACE"
    assert kvq8.status_str(99) == "KVQ8_UNKNOWN_STATUS"
    assert lib.kvq8_abi_version() >= 1


def test_sizes_match_the_page_byte_count(lib):
    # [Day 9-1] §2: 8 kv heads x 128 dims -> 2112 bytes per token per layer
    assert kvq8.cache_bytes_per_token(8) == 2112
    assert kvq8.kv_pool_bytes(3, 8) == 3 * 8 * 256 * 128
    assert kvq8.scale_pool_bytes(3, 8) == 3 * 8 * 256 * 4
    per_token = (2 * kvq8.kv_pool_bytes(1, 8) + 2 * kvq8.scale_pool_bytes(1, 8)) // 256
    assert per_token == 2112


def test_workspace_sizes(lib):
    a = kvq8.decode_workspace_bytes(28, 16, 8, 32)
    assert a > 0 and a % 256 == 0
    assert kvq8.decode_workspace_bytes(64, 32, 8, 128) > 0
    # unsupported: group 3, hd != 128 via the raw call, bad sizes
    assert kvq8.decode_workspace_bytes(1, 6, 2, 4) == 0
    assert lib.kvq8_decode_workspace_bytes(1, 8, 8, 64, 4, 256) == 0
    assert lib.kvq8_decode_workspace_bytes(1, 8, 8, 128, 4, 128) == 0
    assert lib.kvq8_decode_workspace_bytes(1, 8, 0, 128, 4, 256) == 0
    assert lib.kvq8_decode_workspace_bytes(1, 8, 8, 128, 0, 256) == 0
    # partial results stay small next to the cache they summarise
    kv = 28 * 8192 * 2112
    assert a < 0.02 * kv


def _append(lib, **kw):
    a = dict(k=FAKE, v=FAKE, batch=1, n_new=1, nkv=1, hd=128, start=FAKE, table=FAKE,
             max_blocks=1, bs=256, num_blocks=1, kp=FAKE, vp=FAKE, ks=FAKE, vs=FAKE,
             status=None, stream=None)
    a.update(kw)
    return lib.kvq8_quantize_append(*a.values())


def test_append_validation(lib):
    assert _append(lib, hd=64) == kvq8.ERR_UNSUPPORTED
    assert _append(lib, bs=128) == kvq8.ERR_UNSUPPORTED
    assert _append(lib, k=None) == kvq8.ERR_INVALID_ARG
    assert _append(lib, kp=FAKE + 4) == kvq8.ERR_INVALID_ARG          # not 16-byte aligned
    assert _append(lib, batch=-1) == kvq8.ERR_INVALID_ARG
    assert _append(lib, nkv=0) == kvq8.ERR_INVALID_ARG
    assert _append(lib, batch=70000) == kvq8.ERR_UNSUPPORTED
    assert _append(lib, batch=0) == kvq8.OK                          # no-op, nothing launched
    assert _append(lib, n_new=0) == kvq8.OK


def _decode(lib, fn="kvq8_decode_attn", **kw):
    a = dict(q=FAKE, batch=1, nqh=8, nkv=8, hd=128, kp=FAKE, vp=FAKE, ks=FAKE, vs=FAKE,
             num_blocks=4, table=FAKE, max_blocks=4, bs=256, lens=FAKE, sm=0.088,
             out=FAKE, ws=FAKE, ws_bytes=0, status=None, stream=None)
    a.update(kw)
    if fn == "kvq8_decode_split":
        a.pop("out")
    return getattr(lib, fn)(*a.values())


def test_decode_validation(lib):
    need = kvq8.decode_workspace_bytes(1, 8, 8, 4)
    for fn in ("kvq8_decode_attn", "kvq8_decode_split"):
        assert _decode(lib, fn, hd=96) == kvq8.ERR_UNSUPPORTED
        assert _decode(lib, fn, nqh=12) == kvq8.ERR_UNSUPPORTED          # G = 1.5
        assert _decode(lib, fn, nqh=24, nkv=8) == kvq8.ERR_UNSUPPORTED   # G = 3
        assert _decode(lib, fn, nqh=128, nkv=8) == kvq8.ERR_UNSUPPORTED  # G = 16
        assert _decode(lib, fn, q=None) == kvq8.ERR_INVALID_ARG
        assert _decode(lib, fn, lens=None) == kvq8.ERR_INVALID_ARG
        assert _decode(lib, fn, num_blocks=0) == kvq8.ERR_INVALID_ARG
        assert _decode(lib, fn, sm=float("nan")) == kvq8.ERR_INVALID_ARG
        assert _decode(lib, fn, ws=None, ws_bytes=need) == kvq8.ERR_WORKSPACE
        assert _decode(lib, fn, ws=FAKE + 16, ws_bytes=need) == kvq8.ERR_WORKSPACE
        assert _decode(lib, fn, ws_bytes=need - 1) == kvq8.ERR_WORKSPACE
        assert _decode(lib, fn, batch=0) == kvq8.OK
        assert _decode(lib, fn, batch=65536) == kvq8.ERR_UNSUPPORTED     # beyond the grid's y/z limit
        assert _decode(lib, fn, max_blocks=(2**31 - 1) // 256 + 1) == kvq8.ERR_UNSUPPORTED   # positions past int32
    assert _decode(lib, out=None, ws_bytes=need) == kvq8.ERR_INVALID_ARG
    assert lib.kvq8_decode_combine(1, 8, 8, 128, 4, 256, FAKE, FAKE, need - 1, FAKE, None) \
        == kvq8.ERR_WORKSPACE
    assert lib.kvq8_decode_combine(1, 8, 8, 128, 4, 256, None, FAKE, need, FAKE, None) \
        == kvq8.ERR_INVALID_ARG


def test_noalloc_checks_arguments_like_the_regular_entry_point(lib):
    """kvq8_decode_attn_noalloc reports argument errors exactly as
    kvq8_decode_attn does, before its scratch-size check and before any device
    call: an empty batch is a no-op, a null query an argument error and a batch
    beyond the grid limit unsupported, even for sizes beyond the scratch."""
    def na(q=FAKE, batch=1, nqh=8, nkv=8, max_blocks=8, out=FAKE):
        return lib.kvq8_decode_attn_noalloc(q, batch, nqh, nkv, 128, FAKE, FAKE, FAKE, FAKE, 4, FAKE,
                                            max_blocks, 256, FAKE, 0.088, out, None, None)
    big = dict(batch=512, nqh=64, max_blocks=512)
    assert kvq8.decode_workspace_bytes(512, 64, 8, 512) > kvq8.NOALLOC_SCRATCH_BYTES
    assert na(batch=0) == kvq8.OK
    assert na(batch=0, max_blocks=0) == kvq8.ERR_INVALID_ARG
    assert na(q=None, **big) == kvq8.ERR_INVALID_ARG
    assert na(out=None, **big) == kvq8.ERR_INVALID_ARG
    assert na(nqh=24) == kvq8.ERR_UNSUPPORTED
    assert na(batch=65536) == kvq8.ERR_UNSUPPORTED
    assert na(**big) == kvq8.ERR_WORKSPACE


def test_decode_step_ex_flags(lib):
    """kvq8_decode_step_ex refuses undefined flag bits before anything else;
    with its defined flags it checks its arguments as kvq8_decode_step."""
    def step_ex(flags, q=FAKE, batch=1):
        return lib.kvq8_decode_step_ex(q, FAKE, FAKE, batch, 8, 8, 128, FAKE, FAKE, FAKE, FAKE, 4, FAKE, 4,
                                       256, FAKE, 0.088, FAKE, None, 0, None, flags, None)
    assert step_ex(0x2) == kvq8.ERR_INVALID_ARG
    assert step_ex(0x80000000) == kvq8.ERR_INVALID_ARG
    for flags in (0, kvq8.STEP_CACHE_READY):
        assert step_ex(flags, batch=0) == kvq8.OK
        assert step_ex(flags, q=None) == kvq8.ERR_INVALID_ARG
        assert step_ex(flags) == kvq8.ERR_WORKSPACE


def test_host_buffer_entry_validation(lib):
    """The host-buffer entries check every argument before queueing a copy."""
    def app(**kw):
        a = dict(kh=FAKE, vh=FAKE, k=FAKE, v=FAKE, batch=1, n_new=2, nkv=1, hd=128, start=FAKE,
                 table=FAKE, max_blocks=1, bs=256, num_blocks=1, kp=FAKE, vp=FAKE, ks=FAKE, vs=FAKE,
                 status=None, stream=None)
        a.update(kw)
        return lib.kvq8_quantize_append_host(*a.values())
    assert app(kh=None) == kvq8.ERR_INVALID_ARG
    assert app(vh=None) == kvq8.ERR_INVALID_ARG
    assert app(k=None) == kvq8.ERR_INVALID_ARG                      # device staging buffer
    assert app(v=FAKE + 4) == kvq8.ERR_INVALID_ARG
    assert app(hd=64) == kvq8.ERR_UNSUPPORTED
    assert app(kh=None, batch=0) == kvq8.OK                         # nothing to append
    assert app(kh=None, n_new=0) == kvq8.OK

    need = kvq8.decode_workspace_bytes(1, 8, 8, 4)

    def step(**kw):
        a = dict(qh=FAKE, kh=FAKE, vh=FAKE, oh=FAKE, q=FAKE, k=FAKE, v=FAKE, batch=1, nqh=8, nkv=8,
                 hd=128, kp=FAKE, vp=FAKE, ks=FAKE, vs=FAKE, num_blocks=4, table=FAKE, max_blocks=4,
                 bs=256, lens=FAKE, sm=0.088, out=FAKE, ws=FAKE, ws_bytes=need, status=None, stream=None)
        a.update(kw)
        return lib.kvq8_decode_step_host(*a.values())
    for host in ("qh", "kh", "vh", "oh"):
        assert step(**{host: None}) == kvq8.ERR_INVALID_ARG
    assert step(q=None) == kvq8.ERR_INVALID_ARG
    assert step(k=FAKE + 8) == kvq8.ERR_INVALID_ARG
    assert step(out=None) == kvq8.ERR_INVALID_ARG
    assert step(nqh=24) == kvq8.ERR_UNSUPPORTED
    assert step(ws_bytes=need - 1) == kvq8.ERR_WORKSPACE
    assert step(qh=None, batch=0) == kvq8.OK


def test_selftest_bounded_wait_validation(lib):
    f = lib.kvq8_selftest_bounded_wait
    assert f(None, 10**6, None, None) == kvq8.ERR_INVALID_ARG           # no status word
    assert f(FAKE + 2, 10**6, None, None) == kvq8.ERR_INVALID_ARG       # misaligned status word
    assert f(FAKE, 10**6, FAKE + 4, None) == kvq8.ERR_INVALID_ARG       # misaligned time word
    assert f(FAKE, 999, None, None) == kvq8.ERR_INVALID_ARG             # bound below 1 us
    assert f(FAKE, 10**10 + 1, None, None) == kvq8.ERR_INVALID_ARG      # bound above 10 s


def test_quantize_q_validation(lib):
    assert lib.kvq8_quantize_q(FAKE, 4, 64, FAKE, FAKE, None) == kvq8.ERR_UNSUPPORTED
    assert lib.kvq8_quantize_q(None, 4, 128, FAKE, FAKE, None) == kvq8.ERR_INVALID_ARG
    assert lib.kvq8_quantize_q(FAKE, -1, 128, FAKE, FAKE, None) == kvq8.ERR_INVALID_ARG
    assert lib.kvq8_quantize_q(FAKE, 0, 128, FAKE, FAKE, None) == kvq8.OK


def test_fp32_cache_sizes_and_validation(lib):
    # 8 kv heads x 128 fp32 for K and V: 8192 bytes per token per layer
    assert kvq8.cachef32_bytes_per_token(8) == 8192
    assert lib.kvf32_pool_bytes(3, 8, 128, 256) == 3 * 8 * 256 * 128 * 4
    a = dict(k=FAKE, v=FAKE, batch=1, n_new=1, nkv=1, hd=128, start=FAKE, table=FAKE,
             max_blocks=1, bs=256, num_blocks=1, kc=FAKE, vc=FAKE, status=None, stream=None)
    assert lib.kvf32_append(*dict(a, hd=64).values()) == kvq8.ERR_UNSUPPORTED
    assert lib.kvf32_append(*dict(a, kc=FAKE + 4).values()) == kvq8.ERR_INVALID_ARG
    assert lib.kvf32_append(*dict(a, v=None).values()) == kvq8.ERR_INVALID_ARG
    assert lib.kvf32_append(*dict(a, n_new=0).values()) == kvq8.OK
    need = kvq8.decode_workspace_bytes(1, 8, 8, 4)
    d = dict(q=FAKE, batch=1, nqh=8, nkv=8, hd=128, kc=FAKE, vc=FAKE, num_blocks=4, table=FAKE,
             max_blocks=4, bs=256, lens=FAKE, sm=0.088, out=FAKE, ws=FAKE, ws_bytes=need,
             status=None, stream=None)
    call = lambda **kw: lib.kvf32_decode_attn(*dict(d, **kw).values())
    assert call(nqh=24) == kvq8.ERR_UNSUPPORTED
    assert call(vc=None) == kvq8.ERR_INVALID_ARG
    assert call(kc=FAKE + 8) == kvq8.ERR_INVALID_ARG
    assert call(out=None) == kvq8.ERR_INVALID_ARG
    assert call(ws_bytes=need - 1) == kvq8.ERR_WORKSPACE
    assert call(batch=0) == kvq8.OK


def test_int4_cache_sizes_and_validation(lib):
    # 64 code bytes and 4 fp32 parameters per (token, head) for K and V
    assert kvq8.cache4_bytes_per_token(8) == 1280
    a = dict(k=FAKE, v=FAKE, batch=1, n_new=1, nkv=1, hd=128, start=FAKE, table=FAKE,
             max_blocks=1, bs=256, num_blocks=1, kc=FAKE, vc=FAKE, kp=FAKE, vp=FAKE,
             status=None, stream=None)
    assert lib.kvq4_quantize_append(*dict(a, bs=64).values()) == kvq8.ERR_UNSUPPORTED
    assert lib.kvq4_quantize_append(*dict(a, kp=FAKE + 4).values()) == kvq8.ERR_INVALID_ARG
    assert lib.kvq4_quantize_append(*dict(a, batch=0).values()) == kvq8.OK
    need = kvq8.decode_workspace_bytes(1, 8, 8, 4)
    assert lib.kvq4_decode_attn(FAKE, 1, 8, 8, 128, FAKE, FAKE, FAKE, FAKE, 4, FAKE, 4, 256,
                                FAKE, 0.088, FAKE, FAKE, need - 1, None, None) == kvq8.ERR_WORKSPACE
    assert lib.kvq4_decode_attn(FAKE, 1, 8, 8, 128, FAKE, FAKE, FAKE, FAKE, 4, FAKE, 4, 256,
                                FAKE, 0.088, None, FAKE, need, None, None) == kvq8.ERR_INVALID_ARG


def test_mixed_precision_validation(lib):
    one = kvq8.decode_workspace_bytes(1, 8, 8, 4)
    assert kvq8.mixed_workspace_bytes(1, 8, 8, 4) == 2 * one
    r = dict(batch=1, nkv=1, hd=128, kp=FAKE, vp=FAKE, ks=FAKE, vs=FAKE, nb8=2, t8=FAKE, kc=FAKE, vc=FAKE,
             kpa=FAKE, vpa=FAKE, nb4=2, t4=FAKE, max_blocks=2, bs=256, bf=FAKE, bt=FAKE, max_count=1,
             status=None, stream=None)
    assert lib.kvmix_requantize(*dict(r, hd=64).values()) == kvq8.ERR_UNSUPPORTED
    assert lib.kvmix_requantize(*dict(r, bt=None).values()) == kvq8.ERR_INVALID_ARG
    assert lib.kvmix_requantize(*dict(r, kc=FAKE + 4).values()) == kvq8.ERR_INVALID_ARG
    assert lib.kvmix_requantize(*dict(r, max_count=-1).values()) == kvq8.ERR_INVALID_ARG
    assert lib.kvmix_requantize(*dict(r, max_count=0).values()) == kvq8.OK
    d = dict(q=FAKE, batch=1, nqh=8, nkv=8, hd=128, kp=FAKE, vp=FAKE, ks=FAKE, vs=FAKE, nb8=4, t8=FAKE,
             kc=FAKE, vc=FAKE, kpa=FAKE, vpa=FAKE, nb4=4, t4=FAKE, max_blocks=4, bs=256, lens=FAKE,
             n4=FAKE, sm=0.088, out=FAKE, ws=FAKE, ws_bytes=2 * one, status=None, stream=None)
    call = lambda **kw: lib.kvmix_decode_attn(*dict(d, **kw).values())
    assert call(ws_bytes=2 * one - 1) == kvq8.ERR_WORKSPACE
    assert call(n4=None) == kvq8.ERR_INVALID_ARG
    assert call(t4=None) == kvq8.ERR_INVALID_ARG
    assert call(nqh=24) == kvq8.ERR_UNSUPPORTED
    assert call(batch=0) == kvq8.OK


def test_library_is_built_for_sm103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(kbuild.ARCH)
    assert os.path.exists(kbuild.LIB_PATH)


def test_int4_v_chunk_positions_are_a_permutation():
    # the 4-bit cache's V chunk layout places the 32 tokens of a chunk at 32
    # distinct positions of a byte column (the test readers' copy of the rule)
    from kvq8_harness import v4_pos
    import numpy as np
    pos = v4_pos(np.arange(32))
    assert sorted(pos.tolist()) == list(range(32))
    # word 2*t4 + k holds tokens 16k + 2*t4 + {0, 8, 1, 9} in bytes 0..3
    for t4 in range(4):
        for k in range(2):
            toks = [16 * k + 2 * t4 + d for d in (0, 8, 1, 9)]
            assert [int(v4_pos(t)) for t in toks] == [4 * (2 * t4 + k) + b for b in range(4)]
