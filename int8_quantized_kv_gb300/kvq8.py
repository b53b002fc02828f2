"""Python binding of libkvq8 (C ABI in include/kvq8.h), via ctypes.

Argument marshalling only: tensors are passed as device pointers plus the
sizes read from their shapes; every step of the computation runs in the
library's CUDA kernels.  torch is used for device memory and streams.  There
is no fallback: if libkvq8.so cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import NamedTuple, Optional

from . import build as _build

HEAD_DIM = 128
BLOCK_SIZE = 256
Q_BLOCK = 32
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024   # KVQ8_NOALLOC_SCRATCH_BYTES in kvq8.h

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA = range(5)
STEP_CACHE_READY = 0x1   # KVQ8_STEP_CACHE_READY
DEV_BAD_BLOCK_ID, DEV_BAD_CTX_LEN, DEV_BAD_POSITION, DEV_TIMEOUT, DEV_NONFINITE = 0x1, 0x2, 0x4, 0x8, 0x10

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/kvq8.h
SIGNATURES = {
    "kvq8_status_str": (ctypes.c_char_p, [_I]),
    "kvq8_abi_version": (_I, []),
    "kvq8_kv_pool_bytes": (_SZ, [_I, _I, _I, _I]),
    "kvq8_scale_pool_bytes": (_SZ, [_I, _I, _I]),
    "kvq8_cache_bytes_per_token": (_SZ, [_I, _I]),
    "kvq8_quantize_append": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _I, _I, _I,
                                  _P, _P, _P, _P, _P, _P]),
    "kvq8_quantize_append_host": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _I, _I,
                                       _P, _P, _P, _P, _P, _P]),
    "kvq8_quantize_q": (_I, [_P, _I64, _I, _P, _P, _P]),
    "kvq8_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "kvq8_decode_attn": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _I, _I,
                              _P, _F, _P, _P, _SZ, _P, _P]),
    "kvq8_decode_split": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _I, _I,
                               _P, _F, _P, _SZ, _P, _P]),
    "kvq8_decode_combine": (_I, [_I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P, _P]),
    "kvq8_decode_step": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _I, _I,
                              _P, _F, _P, _P, _SZ, _P, _P]),
    "kvq8_decode_step_ex": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _I, _I,
                                 _P, _F, _P, _P, _SZ, _P, ctypes.c_uint32, _P]),
    "kvq8_decode_step_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _I,
                                   _P, _I, _I, _P, _F, _P, _P, _SZ, _P, _P]),
    "kvq8_host_device_pointer": (_P, [_P]),
    "kvq8_selftest_bounded_wait": (_I, [_P, ctypes.c_uint64, _P, _P]),
    "kvq4_code_pool_bytes": (_SZ, [_I, _I, _I, _I]),
    "kvq4_param_pool_bytes": (_SZ, [_I, _I, _I]),
    "kvq4_cache_bytes_per_token": (_SZ, [_I, _I]),
    "kvq4_quantize_append": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _I, _I, _I,
                                  _P, _P, _P, _P, _P, _P]),
    "kvq4_decode_attn": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _I, _I,
                              _P, _F, _P, _P, _SZ, _P, _P]),
    "kvq4_decode_step": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _I, _I,
                              _P, _F, _P, _P, _SZ, _P, _P]),
    "kvmix_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "kvmix_requantize": (_I, [_I, _I, _I, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _P,
                              _I, _I, _P, _P, _I, _P, _P]),
    "kvmix_decode_attn": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _P,
                               _I, _I, _P, _P, _F, _P, _P, _SZ, _P, _P]),
    "kvf32_pool_bytes": (_SZ, [_I, _I, _I, _I]),
    "kvf32_cache_bytes_per_token": (_SZ, [_I, _I]),
    "kvf32_append": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _I, _I, _I, _P, _P, _P, _P]),
    "kvf32_decode_attn": (_I, [_P, _I, _I, _I, _I, _P, _P, _I, _P, _I, _I,
                               _P, _F, _P, _P, _SZ, _P, _P]),
    "kvq8_decode_attn_noalloc": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _I, _I,
                                      _P, _F, _P, _P, _P]),
}

_lib = None


class Kvq8Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_str(status)} ({status})")


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True):
    """Open libkvq8.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if build_if_missing and _build.needs_build():
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libkvq8.so not built ({path}); run int8_quantized_kv_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_str(status: int) -> str:
    return load().kvq8_status_str(status).decode()


def _check(fn: str, status: int):
    if status != OK:
        raise Kvq8Error(fn, status)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream, device=None) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _need_host(*tensors):
    for t in tensors:
        if t.is_cuda:
            raise ValueError("expected a host tensor; got one on " + str(t.device))
        if not t.is_contiguous():
            raise ValueError("kvq8 takes contiguous tensors")
        if t.dtype != _torch().float32:
            raise ValueError("host buffers are fp32")


def _torch():
    import torch
    return torch


def _need_cuda(*tensors):
    for t in tensors:
        if t is None or isinstance(t, int):
            continue
        if not t.is_cuda:
            raise ValueError("kvq8 takes device tensors; got one on " + str(t.device))
        if not t.is_contiguous():
            raise ValueError("kvq8 takes contiguous tensors")


# ------------------------------------------------------------------ sizes ---
def kv_pool_bytes(num_blocks: int, nkv: int) -> int:
    return int(load().kvq8_kv_pool_bytes(num_blocks, nkv, HEAD_DIM, BLOCK_SIZE))


def scale_pool_bytes(num_blocks: int, nkv: int) -> int:
    return int(load().kvq8_scale_pool_bytes(num_blocks, nkv, BLOCK_SIZE))


def cache_bytes_per_token(nkv: int, hd: int = HEAD_DIM) -> int:
    return int(load().kvq8_cache_bytes_per_token(nkv, hd))


def decode_workspace_bytes(batch: int, nqh: int, nkv: int, max_blocks: int) -> int:
    return int(load().kvq8_decode_workspace_bytes(batch, nqh, nkv, HEAD_DIM, max_blocks, BLOCK_SIZE))


class KVCache(NamedTuple):
    """One layer-pool of the paged cache (see the layout in include/kvq8.h)."""
    k_pool: object   # int8 [num_blocks][nkv][256][128]  token-major, 16-B chunks permuted
    v_pool: object   # int8 [num_blocks][nkv][4][128][64] dim-major per 64-token quarter
    k_scale: object  # fp32 [num_blocks][nkv][256]
    v_scale: object  # fp32 [num_blocks][nkv][256]

    @property
    def num_blocks(self) -> int:
        return self.k_pool.shape[0]

    @property
    def nkv(self) -> int:
        return self.k_pool.shape[1]


def alloc_cache(num_blocks: int, nkv: int, device="cuda") -> KVCache:
    """Allocate (uninitialised) pools with torch, sized by the library."""
    import torch
    assert kv_pool_bytes(num_blocks, nkv) == num_blocks * nkv * BLOCK_SIZE * HEAD_DIM
    k = torch.empty((num_blocks, nkv, BLOCK_SIZE, HEAD_DIM), dtype=torch.int8, device=device)
    v = torch.empty((num_blocks, nkv, BLOCK_SIZE // 64, HEAD_DIM, 64), dtype=torch.int8, device=device)
    ks = torch.empty((num_blocks, nkv, BLOCK_SIZE), dtype=torch.float32, device=device)
    vs = torch.empty((num_blocks, nkv, BLOCK_SIZE), dtype=torch.float32, device=device)
    return KVCache(k, v, ks, vs)


def alloc_workspace(batch: int, nqh: int, nkv: int, max_blocks: int, device="cuda"):
    import torch
    n = decode_workspace_bytes(batch, nqh, nkv, max_blocks)
    if n == 0:
        raise ValueError("unsupported decode sizes")
    return torch.empty(n, dtype=torch.uint8, device=device)


# ---------------------------------------------------------- entry points ---
def quantize_append(k_new, v_new, start_pos, block_table, cache: KVCache,
                    dev_status=None, stream=None):
    """k_new, v_new: fp32 [batch][n_new][nkv][128]; start_pos int32 [batch];
    block_table int32 [batch][max_blocks]."""
    _need_cuda(k_new, v_new, start_pos, block_table, *cache, dev_status)
    batch, n_new, nkv, hd = k_new.shape
    st = load().kvq8_quantize_append(
        _ptr(k_new), _ptr(v_new), batch, n_new, nkv, hd, _ptr(start_pos),
        _ptr(block_table), block_table.shape[1], BLOCK_SIZE, cache.num_blocks,
        _ptr(cache.k_pool), _ptr(cache.v_pool), _ptr(cache.k_scale), _ptr(cache.v_scale),
        _ptr(dev_status), _stream(stream))
    _check("kvq8_quantize_append", st)


def quantize_append_host(k_host, v_host, k_new, v_new, start_pos, block_table, cache: KVCache,
                         dev_status=None, stream=None):
    """quantize_append with the new rows in host memory (page-locked for full
    speed): k_host, v_host are copied into the device buffers k_new, v_new
    (fp32 [batch][n_new][nkv][128]) on the stream, then appended."""
    _need_host(k_host, v_host)
    _need_cuda(k_new, v_new, start_pos, block_table, *cache, dev_status)
    if k_host.shape != k_new.shape or v_host.shape != v_new.shape or k_new.shape != v_new.shape:
        raise ValueError("host and device row buffers differ in shape")
    batch, n_new, nkv, hd = k_new.shape
    st = load().kvq8_quantize_append_host(
        _ptr(k_host), _ptr(v_host), _ptr(k_new), _ptr(v_new), batch, n_new, nkv, hd, _ptr(start_pos),
        _ptr(block_table), block_table.shape[1], BLOCK_SIZE, cache.num_blocks,
        _ptr(cache.k_pool), _ptr(cache.v_pool), _ptr(cache.k_scale), _ptr(cache.v_scale),
        _ptr(dev_status), _stream(stream))
    _check("kvq8_quantize_append_host", st)


def quantize_q(q, q_codes, q_scales, stream=None):
    """q fp32 [..., 128] -> q_codes int8 [..., 128], q_scales fp32 [..., 4]."""
    _need_cuda(q, q_codes, q_scales)
    hd = q.shape[-1]
    n_rows = q.numel() // hd if hd else 0
    st = load().kvq8_quantize_q(_ptr(q), n_rows, hd, _ptr(q_codes), _ptr(q_scales), _stream(stream))
    _check("kvq8_quantize_q", st)


def _decode_common(q, cache: KVCache, block_table, ctx_lens):
    batch, nqh, hd = q.shape
    return batch, nqh, cache.nkv, hd, block_table.shape[1]


def decode_attn(q, cache: KVCache, block_table, ctx_lens, out, workspace,
                sm_scale: Optional[float] = None, dev_status=None, stream=None):
    """q fp32 [batch][nqh][128] -> out fp32 [batch][nqh][128]."""
    _need_cuda(q, block_table, ctx_lens, out, workspace, *cache, dev_status)
    batch, nqh, nkv, hd, max_blocks = _decode_common(q, cache, block_table, ctx_lens)
    sm = 1.0 / math.sqrt(hd) if sm_scale is None else sm_scale
    st = load().kvq8_decode_attn(
        _ptr(q), batch, nqh, nkv, hd, _ptr(cache.k_pool), _ptr(cache.v_pool),
        _ptr(cache.k_scale), _ptr(cache.v_scale), cache.num_blocks, _ptr(block_table),
        max_blocks, BLOCK_SIZE, _ptr(ctx_lens), sm, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream))
    _check("kvq8_decode_attn", st)


def decode_step(q, k_new, v_new, cache: KVCache, block_table, ctx_lens, out, workspace,
                sm_scale: Optional[float] = None, dev_status=None, stream=None, cache_ready: bool = False):
    """One decode step: append k_new/v_new (fp32 [batch][nkv][128]) at position
    ctx_lens-1 and attend over ctx_lens tokens (two launches: the split kernel,
    which also appends the token, and the combine, a programmatic dependent of
    the split).  cache_ready: KVQ8_STEP_CACHE_READY (kvq8_decode_step_ex)."""
    _need_cuda(q, k_new, v_new, block_table, ctx_lens, out, workspace, *cache, dev_status)
    batch, nqh, nkv, hd, max_blocks = _decode_common(q, cache, block_table, ctx_lens)
    sm = 1.0 / math.sqrt(hd) if sm_scale is None else sm_scale
    st = load().kvq8_decode_step_ex(
        _ptr(q), _ptr(k_new), _ptr(v_new), batch, nqh, nkv, hd, _ptr(cache.k_pool),
        _ptr(cache.v_pool), _ptr(cache.k_scale), _ptr(cache.v_scale), cache.num_blocks,
        _ptr(block_table), max_blocks, BLOCK_SIZE, _ptr(ctx_lens), sm, _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_status),
        STEP_CACHE_READY if cache_ready else 0, _stream(stream))
    _check("kvq8_decode_step_ex", st)


def decode_step_host(q_host, k_host, v_host, out_host, q, k_new, v_new, cache: KVCache, block_table,
                     ctx_lens, out, workspace, sm_scale: Optional[float] = None, dev_status=None,
                     stream=None):
    """decode_step from host memory and back, queued on the stream (synchronise
    it before reading out_host).  Page-locked host buffers are read and written
    by the kernels directly; other host buffers are copied through the device
    buffers q, k_new, v_new and out."""
    _need_host(q_host, k_host, v_host, out_host)
    _need_cuda(q, k_new, v_new, block_table, ctx_lens, out, workspace, *cache, dev_status)
    if (q_host.shape != q.shape or out_host.shape != out.shape or q.shape != out.shape or
            k_host.shape != k_new.shape or v_host.shape != v_new.shape):
        raise ValueError("host and device buffers differ in shape")
    batch, nqh, nkv, hd, max_blocks = _decode_common(q, cache, block_table, ctx_lens)
    sm = 1.0 / math.sqrt(hd) if sm_scale is None else sm_scale
    st = load().kvq8_decode_step_host(
        _ptr(q_host), _ptr(k_host), _ptr(v_host), _ptr(out_host), _ptr(q), _ptr(k_new), _ptr(v_new),
        batch, nqh, nkv, hd, _ptr(cache.k_pool), _ptr(cache.v_pool), _ptr(cache.k_scale),
        _ptr(cache.v_scale), cache.num_blocks, _ptr(block_table), max_blocks, BLOCK_SIZE,
        _ptr(ctx_lens), sm, _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _stream(stream))
    _check("kvq8_decode_step_host", st)


class HostMapped:
    """A page-locked host tensor presented to this binding's calls as device
    memory: data_ptr() is its device address (kvq8_host_device_pointer), so the
    kernels read (q, new rows) or write (out) the host memory themselves over
    the host link, with no copy.  Meant for the small per-step buffers; raises
    if the tensor is not a contiguous page-locked fp32 host tensor that the
    device can address at a 16-byte boundary."""

    is_cuda = True

    def __init__(self, t):
        _need_host(t)
        if not t.is_pinned():
            raise ValueError("HostMapped needs a page-locked (pinned) tensor")
        addr = load().kvq8_host_device_pointer(t.data_ptr())
        if not addr:
            raise ValueError("the device cannot address this host memory (or not 16-byte aligned)")
        self._t, self._addr = t, addr
        self.shape, self.dtype = t.shape, t.dtype

    def data_ptr(self) -> int:
        return self._addr

    def is_contiguous(self) -> bool:
        return True

    def numel(self) -> int:
        return self._t.numel()

    def element_size(self) -> int:
        return self._t.element_size()


class DecodeStep:
    """A decode step bound to fixed buffers: the arguments are checked and
    converted once, and each step is then one C call (bind once, run every
    step, as a serving loop does with its reused buffers).

    run() is kvq8_decode_step on the bound device buffers.  With host buffers
    bound as well (q_host, k_host, v_host, out_host), run_host() is the same
    step reading the inputs from and writing the result to them: page-locked
    host buffers are handed to the kernels directly (their device addresses
    are looked up here, once), others go through kvq8_decode_step_host and the
    bound device buffers.  Refill the bound inputs between steps; the stream
    (the current one when None) is bound too.  Synchronise it before reading
    the result."""

    def __init__(self, q, k_new, v_new, cache: KVCache, block_table, ctx_lens, out, workspace,
                 sm_scale: Optional[float] = None, dev_status=None, stream=None,
                 q_host=None, k_host=None, v_host=None, out_host=None, cache_ready: bool = False):
        _need_cuda(q, k_new, v_new, block_table, ctx_lens, out, workspace, *cache, dev_status)
        batch, nqh, nkv, hd, max_blocks = _decode_common(q, cache, block_table, ctx_lens)
        sm = 1.0 / math.sqrt(hd) if sm_scale is None else sm_scale
        lib = load()
        self._lib = lib
        st = _P(_stream(stream))
        common = [_I(batch), _I(nqh), _I(nkv), _I(hd), _P(_ptr(cache.k_pool)), _P(_ptr(cache.v_pool)),
                  _P(_ptr(cache.k_scale)), _P(_ptr(cache.v_scale)), _I(cache.num_blocks),
                  _P(_ptr(block_table)), _I(max_blocks), _I(BLOCK_SIZE), _P(_ptr(ctx_lens)), _F(sm)]
        tail = [_P(_ptr(workspace)), _SZ(workspace.numel() * workspace.element_size()), _P(_ptr(dev_status)), st]
        flags = [ctypes.c_uint32(STEP_CACHE_READY if cache_ready else 0)]
        ex_tail = tail[:-1] + flags + tail[-1:]
        self._dev_args = tuple([_P(_ptr(q)), _P(_ptr(k_new)), _P(_ptr(v_new))] + common + [_P(_ptr(out))] +
                               ex_tail)
        self._keep = (q, k_new, v_new, cache, block_table, ctx_lens, out, workspace, dev_status, stream)
        self._host_fn = None
        hosts = (q_host, k_host, v_host, out_host)
        if any(h is not None for h in hosts):
            if any(h is None for h in hosts):
                raise ValueError("bind all four host buffers or none")
            _need_host(*hosts)
            if (q_host.shape != q.shape or out_host.shape != out.shape or q.shape != out.shape or
                    k_host.shape != k_new.shape or v_host.shape != v_new.shape):
                raise ValueError("host and device buffers differ in shape")
            mapped = [lib.kvq8_host_device_pointer(_ptr(h)) for h in hosts]
            if all(mapped):
                self._host_fn = lib.kvq8_decode_step_ex
                self._host_args = tuple([_P(mapped[0]), _P(mapped[1]), _P(mapped[2])] + common +
                                        [_P(mapped[3])] + ex_tail)
            else:
                if cache_ready:
                    raise ValueError("cache_ready needs page-locked host buffers (the copying path has no flags)")
                self._host_fn = lib.kvq8_decode_step_host
                self._host_args = tuple([_P(_ptr(h)) for h in hosts] + list(self._dev_args[:3]) + common +
                                        [self._dev_args[3 + len(common)]] + tail)
            self._keep = self._keep + hosts
        self.host_direct = self._host_fn is not None and self._host_fn is lib.kvq8_decode_step_ex

    def run(self):
        _check("kvq8_decode_step_ex", self._lib.kvq8_decode_step_ex(*self._dev_args))

    def run_host(self):
        if self._host_fn is None:
            raise ValueError("no host buffers bound")
        _check("kvq8_decode_step", self._host_fn(*self._host_args))


def decode_split(q, cache: KVCache, block_table, ctx_lens, workspace,
                 sm_scale: Optional[float] = None, dev_status=None, stream=None):
    _need_cuda(q, block_table, ctx_lens, workspace, *cache, dev_status)
    batch, nqh, nkv, hd, max_blocks = _decode_common(q, cache, block_table, ctx_lens)
    sm = 1.0 / math.sqrt(hd) if sm_scale is None else sm_scale
    st = load().kvq8_decode_split(
        _ptr(q), batch, nqh, nkv, hd, _ptr(cache.k_pool), _ptr(cache.v_pool),
        _ptr(cache.k_scale), _ptr(cache.v_scale), cache.num_blocks, _ptr(block_table),
        max_blocks, BLOCK_SIZE, _ptr(ctx_lens), sm, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream))
    _check("kvq8_decode_split", st)


def decode_combine(batch: int, nqh: int, nkv: int, max_blocks: int, ctx_lens, workspace, out,
                   stream=None):
    _need_cuda(ctx_lens, workspace, out)
    st = load().kvq8_decode_combine(
        batch, nqh, nkv, HEAD_DIM, max_blocks, BLOCK_SIZE, _ptr(ctx_lens), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _stream(stream))
    _check("kvq8_decode_combine", st)


def decode_attn_noalloc(q, cache: KVCache, block_table, ctx_lens, out,
                        sm_scale: Optional[float] = None, dev_status=None, stream=None):
    """decode_attn without a workspace, for callers that cannot allocate device
    memory: the partial results live in the library's static 16 MiB device
    scratch (see kvq8_decode_attn_noalloc in kvq8.h; concurrent calls race)."""
    _need_cuda(q, block_table, ctx_lens, out, *cache, dev_status)
    batch, nqh, nkv, hd, max_blocks = _decode_common(q, cache, block_table, ctx_lens)
    sm = 1.0 / math.sqrt(hd) if sm_scale is None else sm_scale
    st = load().kvq8_decode_attn_noalloc(
        _ptr(q), batch, nqh, nkv, hd, _ptr(cache.k_pool), _ptr(cache.v_pool),
        _ptr(cache.k_scale), _ptr(cache.v_scale), cache.num_blocks, _ptr(block_table),
        max_blocks, BLOCK_SIZE, _ptr(ctx_lens), sm, _ptr(out), _ptr(dev_status),
        _stream(stream))
    _check("kvq8_decode_attn_noalloc", st)


def selftest_bounded_wait(timeout_ns: int, dev_status, waited_ns=None, stream=None):
    """One warp waits, bounded by timeout_ns, on a barrier phase that nothing
    completes (the decode kernels' wait routine): it ORs KVQ8_DEV_TIMEOUT into
    dev_status (int32 [1], device) and writes the nanoseconds it waited into
    waited_ns (int64 [1], device, optional)."""
    _need_cuda(dev_status, waited_ns)
    _check("kvq8_selftest_bounded_wait",
           load().kvq8_selftest_bounded_wait(_ptr(dev_status), int(timeout_ns), _ptr(waited_ns), _stream(stream)))


# ------------------------------------------------------------ 4-bit cache ---
class KV4Cache(NamedTuple):
    """The asymmetric INT4 group-64 cache (layout in include/kvq8.h)."""
    k_codes: object  # uint8 [num_blocks][nkv][256][64]  token-major rows
    v_codes: object  # uint8 [num_blocks][nkv][256][64]  stored as [8 chunks][64 byte columns][32]
    k_param: object  # fp32 [num_blocks][nkv][256][4]  (scale0, zero0, scale1, zero1)
    v_param: object  # fp32 [num_blocks][nkv][256][4]

    @property
    def num_blocks(self) -> int:
        return self.k_codes.shape[0]

    @property
    def nkv(self) -> int:
        return self.k_codes.shape[1]


def cache4_bytes_per_token(nkv: int, hd: int = HEAD_DIM) -> int:
    return int(load().kvq4_cache_bytes_per_token(nkv, hd))


def alloc_cache4(num_blocks: int, nkv: int, device="cuda") -> KV4Cache:
    import torch
    lib = load()
    assert lib.kvq4_code_pool_bytes(num_blocks, nkv, HEAD_DIM, BLOCK_SIZE) == num_blocks * nkv * BLOCK_SIZE * 64
    kc = torch.empty((num_blocks, nkv, BLOCK_SIZE, HEAD_DIM // 2), dtype=torch.uint8, device=device)
    vc = torch.empty_like(kc)
    kp = torch.empty((num_blocks, nkv, BLOCK_SIZE, 4), dtype=torch.float32, device=device)
    vp = torch.empty_like(kp)
    return KV4Cache(kc, vc, kp, vp)


def quantize_append4(k_new, v_new, start_pos, block_table, cache: KV4Cache, dev_status=None,
                     stream=None):
    """k_new, v_new: fp32 [batch][n_new][nkv][128] into the 4-bit cache."""
    _need_cuda(k_new, v_new, start_pos, block_table, *cache, dev_status)
    batch, n_new, nkv, hd = k_new.shape
    st = load().kvq4_quantize_append(
        _ptr(k_new), _ptr(v_new), batch, n_new, nkv, hd, _ptr(start_pos), _ptr(block_table),
        block_table.shape[1], BLOCK_SIZE, cache.num_blocks, _ptr(cache.k_codes),
        _ptr(cache.v_codes), _ptr(cache.k_param), _ptr(cache.v_param), _ptr(dev_status),
        _stream(stream))
    _check("kvq4_quantize_append", st)


def decode_attn4(q, cache: KV4Cache, block_table, ctx_lens, out, workspace,
                 sm_scale: Optional[float] = None, dev_status=None, stream=None):
    """fp32 q [batch][nqh][128] over the 4-bit cache -> out fp32 [batch][nqh][128]."""
    _need_cuda(q, block_table, ctx_lens, out, workspace, *cache, dev_status)
    batch, nqh, hd = q.shape
    sm = 1.0 / math.sqrt(hd) if sm_scale is None else sm_scale
    st = load().kvq4_decode_attn(
        _ptr(q), batch, nqh, cache.nkv, hd, _ptr(cache.k_codes), _ptr(cache.v_codes),
        _ptr(cache.k_param), _ptr(cache.v_param), cache.num_blocks, _ptr(block_table),
        block_table.shape[1], BLOCK_SIZE, _ptr(ctx_lens), sm, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream))
    _check("kvq4_decode_attn", st)


def decode_step4(q, k_new, v_new, cache: KV4Cache, block_table, ctx_lens, out, workspace,
                 sm_scale: Optional[float] = None, dev_status=None, stream=None):
    """One decode step over the 4-bit cache: append k_new/v_new (fp32
    [batch][nkv][128]) at position ctx_lens-1 and attend over ctx_lens tokens
    (two launches: the split kernel, which also appends the token, and the
    merge)."""
    _need_cuda(q, k_new, v_new, block_table, ctx_lens, out, workspace, *cache, dev_status)
    batch, nqh, hd = q.shape
    sm = 1.0 / math.sqrt(hd) if sm_scale is None else sm_scale
    st = load().kvq4_decode_step(
        _ptr(q), _ptr(k_new), _ptr(v_new), batch, nqh, cache.nkv, hd, _ptr(cache.k_codes),
        _ptr(cache.v_codes), _ptr(cache.k_param), _ptr(cache.v_param), cache.num_blocks,
        _ptr(block_table), block_table.shape[1], BLOCK_SIZE, _ptr(ctx_lens), sm, _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream))
    _check("kvq4_decode_step", st)


# ------------------------------------------------------------- fp32 cache ---
class KVF32Cache(NamedTuple):
    """The fp32 K/V cache, the comparator of the int8 one (layout in include/kvq8.h)."""
    k_cache: object  # fp32 [num_blocks][nkv][256][128]
    v_cache: object  # fp32 [num_blocks][nkv][256][128]

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]

    @property
    def nkv(self) -> int:
        return self.k_cache.shape[1]


def cachef32_bytes_per_token(nkv: int, hd: int = HEAD_DIM) -> int:
    return int(load().kvf32_cache_bytes_per_token(nkv, hd))


def alloc_cachef32(num_blocks: int, nkv: int, device="cuda") -> KVF32Cache:
    import torch
    lib = load()
    assert lib.kvf32_pool_bytes(num_blocks, nkv, HEAD_DIM, BLOCK_SIZE) == num_blocks * nkv * BLOCK_SIZE * HEAD_DIM * 4
    kc = torch.empty((num_blocks, nkv, BLOCK_SIZE, HEAD_DIM), dtype=torch.float32, device=device)
    return KVF32Cache(kc, torch.empty_like(kc))


def appendf32(k_new, v_new, start_pos, block_table, cache: KVF32Cache, dev_status=None, stream=None):
    """k_new, v_new: fp32 [batch][n_new][nkv][128] copied into the fp32 cache."""
    _need_cuda(k_new, v_new, start_pos, block_table, *cache, dev_status)
    batch, n_new, nkv, hd = k_new.shape
    st = load().kvf32_append(
        _ptr(k_new), _ptr(v_new), batch, n_new, nkv, hd, _ptr(start_pos), _ptr(block_table),
        block_table.shape[1], BLOCK_SIZE, cache.num_blocks, _ptr(cache.k_cache),
        _ptr(cache.v_cache), _ptr(dev_status), _stream(stream))
    _check("kvf32_append", st)


def decode_attnf32(q, cache: KVF32Cache, block_table, ctx_lens, out, workspace,
                   sm_scale: Optional[float] = None, dev_status=None, stream=None):
    """fp32 q [batch][nqh][128] over the fp32 cache -> out fp32 [batch][nqh][128]."""
    _need_cuda(q, block_table, ctx_lens, out, workspace, *cache, dev_status)
    batch, nqh, hd = q.shape
    sm = 1.0 / math.sqrt(hd) if sm_scale is None else sm_scale
    st = load().kvf32_decode_attn(
        _ptr(q), batch, nqh, cache.nkv, hd, _ptr(cache.k_cache), _ptr(cache.v_cache),
        cache.num_blocks, _ptr(block_table), block_table.shape[1], BLOCK_SIZE, _ptr(ctx_lens),
        sm, _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _stream(stream))
    _check("kvf32_decode_attn", st)


# ------------------------------------------ mixed precision by token age ---
def mixed_workspace_bytes(batch: int, nqh: int, nkv: int, max_blocks: int) -> int:
    return int(load().kvmix_decode_workspace_bytes(batch, nqh, nkv, HEAD_DIM, max_blocks, BLOCK_SIZE))


def alloc_mixed_workspace(batch, nqh, nkv, max_blocks, device="cuda"):
    import torch
    n = mixed_workspace_bytes(batch, nqh, nkv, max_blocks)
    if n == 0:
        raise Kvq8Error("kvmix_decode_workspace_bytes", ERR_UNSUPPORTED)
    return torch.empty(n, dtype=torch.uint8, device=device)


def requantize_blocks(cache: KVCache, table8, cache4: KV4Cache, table4, blk_from, blk_to,
                      max_count: int, dev_status=None, stream=None):
    """Requantise logical blocks [blk_from[b], blk_to[b]) of every sequence from
    the int8 cache (table8) into the 4-bit cache (table4)."""
    _need_cuda(*cache, *cache4, table8, table4, blk_from, blk_to, dev_status)
    batch, max_blocks = table8.shape
    st = load().kvmix_requantize(
        batch, cache.nkv, HEAD_DIM, _ptr(cache.k_pool), _ptr(cache.v_pool), _ptr(cache.k_scale),
        _ptr(cache.v_scale), cache.num_blocks, _ptr(table8), _ptr(cache4.k_codes),
        _ptr(cache4.v_codes), _ptr(cache4.k_param), _ptr(cache4.v_param), cache4.num_blocks,
        _ptr(table4), max_blocks, BLOCK_SIZE, _ptr(blk_from), _ptr(blk_to), int(max_count),
        _ptr(dev_status), _stream(stream))
    _check("kvmix_requantize", st)


def decode_attn_mixed(q, cache: KVCache, table8, cache4: KV4Cache, table4, ctx_lens, n4_blocks, out,
                      workspace, sm_scale: Optional[float] = None, dev_status=None, stream=None):
    """Decode over 4-bit old blocks [0, n4_blocks[b]) and int8 recent blocks."""
    _need_cuda(q, table8, table4, ctx_lens, n4_blocks, out, workspace, *cache, *cache4, dev_status)
    batch, nqh, hd = q.shape
    sm = 1.0 / math.sqrt(hd) if sm_scale is None else sm_scale
    st = load().kvmix_decode_attn(
        _ptr(q), batch, nqh, cache.nkv, hd, _ptr(cache.k_pool), _ptr(cache.v_pool),
        _ptr(cache.k_scale), _ptr(cache.v_scale), cache.num_blocks, _ptr(table8),
        _ptr(cache4.k_codes), _ptr(cache4.v_codes), _ptr(cache4.k_param), _ptr(cache4.v_param),
        cache4.num_blocks, _ptr(table4), table8.shape[1], BLOCK_SIZE, _ptr(ctx_lens),
        _ptr(n4_blocks), sm, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream))
    _check("kvmix_decode_attn", st)
