"""kvq8_decode_attn_noalloc against kvq8_decode_attn.

The allocation-free entry point serves callers that cannot allocate device
memory (they hold only their inputs, outputs and a stream), so it keeps the
split partial results in the library's static device scratch instead of a
caller workspace.  Its results must match the regular entry point's, call
after call, even though every call reuses the same scratch.  This file is
named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from int8_quantized_kv_gb300 import kvq8
from int8_quantized_kv_gb300 import workloads as wl
from kvq8_harness import Case, SM_SCALE, assert_close

pytestmark = pytest.mark.gpu


def _regular(case):
    out = torch.empty_like(case.q_d)
    ws = kvq8.alloc_workspace(case.cfg.batch, case.cfg.nqh, case.cfg.nkv, case.max_blocks)
    kvq8.decode_attn(case.q_d, case.cache, case.table_d, case.lens_d, out, ws, sm_scale=SM_SCALE)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _noalloc(case):
    out = torch.full_like(case.q_d, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq8.decode_attn_noalloc(case.q_d, case.cache, case.table_d, case.lens_d, out,
                             sm_scale=SM_SCALE, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return out.cpu().numpy()


def test_noalloc_matches_regular_decode_two_calls_in_a_row(gpu_lib):
    # two different workloads back to back: the second call finds the first
    # call's partial results in the shared scratch and must not be affected
    a = Case(wl.Workload("noalloc_a", 300, batch=5, nqh=16, nkv=4, ctx_range=(1, 3000)))
    b = Case(wl.Workload("noalloc_b", 301, batch=3, nqh=8, nkv=8, ctx_range=(200, 9000)))
    for case in (a, b):
        assert kvq8.decode_workspace_bytes(case.cfg.batch, case.cfg.nqh, case.cfg.nkv,
                                           case.max_blocks) <= kvq8.NOALLOC_SCRATCH_BYTES
    got_a = _noalloc(a)
    got_b = _noalloc(b)
    assert_close(got_a, _regular(a), "noalloc call 1")
    assert_close(got_b, _regular(b), "noalloc call 2")


def test_noalloc_rejects_sizes_beyond_its_scratch(gpu_lib):
    batch, nqh, nkv, max_blocks = 512, 64, 8, 512
    need = kvq8.decode_workspace_bytes(batch, nqh, nkv, max_blocks)
    assert need > kvq8.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the size check comes first
    st = gpu_lib.load().kvq8_decode_attn_noalloc(
        fake, batch, nqh, nkv, 128, fake, fake, fake, fake, 4, fake, max_blocks, 256, fake,
        SM_SCALE, fake, None, None)
    assert st == kvq8.ERR_WORKSPACE
