"""ce_fwd_f32_noalloc: the flat cross-entropy for callers that cannot
allocate device memory (graph capture, a fixed memory budget owned by
someone else).  It must give what ce_fwd_f32 gives, call after call, while
using the library's own scratch array instead of a caller workspace.

Kept in a file of its own that pytest collects last, so a run that stops at
the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import gen

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-5, 1e-6   # the fp32 cross-entropy tolerance of the other tests


def _case(seed, T, V):
    z = torch.from_numpy(gen.normal_f32(seed, 0, (T, V))).cuda()
    t = torch.from_numpy(gen.targets(seed, 1, (T,), V)).cuda()
    return z, t


def _reference(lmho, z, t):
    return float(lmho.ce_fwd_f32(z, t).item())


def test_noalloc_matches_workspace_entry_point_twice_in_a_row(gpu_lib):
    lmho = gpu_lib
    lib = lmho.load()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [_case(21, 4096, 4096), _case(22, 777, 20000)]   # warp-per-row, then CTA-per-row
    losses = [torch.full((1,), float("nan"), device="cuda") for _ in cases]
    # two calls in a row straight through the C ABI, no sync in between
    for (z, t), out in zip(cases, losses):
        T, V = z.shape
        rc = lib.ce_fwd_f32_noalloc(ctypes.c_void_p(z.data_ptr()), ctypes.c_void_p(t.data_ptr()), T, V,
                                    ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(stream))
        assert rc == 0, lmho.strerror(rc)
    torch.cuda.synchronize()
    for (z, t), out in zip(cases, losses):
        want = _reference(lmho, z, t)
        assert float(out.item()) == pytest.approx(want, rel=RTOL, abs=ATOL)
    # and again through the binding, reusing the scratch left by the calls above
    z, t = cases[0]
    again = lmho.ce_fwd_f32_noalloc(z, t, torch.empty(1, device="cuda"))
    assert float(again.item()) == pytest.approx(_reference(lmho, z, t), rel=RTOL, abs=ATOL)


def test_noalloc_rejects_oversize_and_aliasing(gpu_lib):
    lib = gpu_lib.load()
    big_T = 65537
    # sizes are checked before any pointer is touched
    assert lib.ce_fwd_f32_noalloc(ctypes.c_void_p(0x10000000), ctypes.c_void_p(0x20000000), big_T, 8,
                                  ctypes.c_void_p(0x30000000), None) == gpu_lib.LMHO_ERR_INVALID_ARG
    z, t = _case(23, 16, 64)
    rc = lib.ce_fwd_f32_noalloc(ctypes.c_void_p(z.data_ptr()), ctypes.c_void_p(t.data_ptr()), 16, 64,
                                ctypes.c_void_p(z.data_ptr() + 8), None)
    assert rc == gpu_lib.LMHO_ERR_ALIAS
