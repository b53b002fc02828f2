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
    # two different workloads back to back, the one with more split records
    # first: the second call finds the first call's partial results in the
    # shared scratch and must not be affected by them.  Both entry points run
    # the same kernels on the same grid in the same order, so the outputs are
    # equal bit for bit; each is also checked against the oracle's tolerance.
    b = Case(wl.Workload("noalloc_b", 301, batch=3, nqh=8, nkv=8, ctx_range=(200, 9000)))
    a = Case(wl.Workload("noalloc_a", 300, batch=5, nqh=16, nkv=4, ctx_range=(1, 3000)))
    for case in (a, b):
        assert kvq8.decode_workspace_bytes(case.cfg.batch, case.cfg.nqh, case.cfg.nkv,
                                           case.max_blocks) <= kvq8.NOALLOC_SCRATCH_BYTES
    assert int(b.lens.sum()) * b.cfg.nkv > int(a.lens.sum()) * a.cfg.nkv
    got_b = _noalloc(b)
    got_a = _noalloc(a)
    reg_b, reg_a = _regular(b), _regular(a)
    assert np.array_equal(got_b, reg_b), "noalloc call 1 differs from kvq8_decode_attn"
    assert np.array_equal(got_a, reg_a), "noalloc call 2 differs from kvq8_decode_attn"
    for case, got in ((b, got_b), (a, got_a)):
        for bb in range(case.cfg.batch):
            for h in range(case.cfg.nkv):
                G = case.cfg.group
                assert_close(got[bb, h * G:(h + 1) * G], case.oracle_unit(bb, h),
                             f"noalloc {case.cfg.name} b={bb} h={h}")


def test_noalloc_rejects_sizes_beyond_its_scratch(gpu_lib):
    batch, nqh, nkv, max_blocks = 512, 64, 8, 512
    need = kvq8.decode_workspace_bytes(batch, nqh, nkv, max_blocks)
    assert need > kvq8.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the size check comes first
    st = gpu_lib.load().kvq8_decode_attn_noalloc(
        fake, batch, nqh, nkv, 128, fake, fake, fake, fake, 4, fake, max_blocks, 256, fake,
        SM_SCALE, fake, None, None)
    assert st == kvq8.ERR_WORKSPACE
