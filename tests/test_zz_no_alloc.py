"""ce_fwd_f32_noalloc: the flat cross-entropy for callers that cannot
allocate device memory (a process that reserved its device memory up front,
a plug-in inside another framework's allocator).  It must give the loss the
oracle gives, and what ce_fwd_f32 gives, call after call, while using the
library's own scratch array instead of a caller workspace, and it must not
change the device's memory footprint.

Kept in a file of its own that pytest collects last, so a run that stops at
the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import gen
import oracle

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-5, 1e-6   # the fp32 cross-entropy tolerance of the other tests


def _case(seed, T, V):
    z = gen.normal_f32(seed, 0, (T, V))
    t = gen.targets(seed, 1, (T,), V)
    return z, t, torch.from_numpy(z).cuda(), torch.from_numpy(t).cuda()


def _call(lib, zd, td, out, stream):
    T, V = zd.shape
    return lib.ce_fwd_f32_noalloc(ctypes.c_void_p(zd.data_ptr()), ctypes.c_void_p(td.data_ptr()), T, V,
                                  ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(stream))


def test_noalloc_matches_oracle_and_workspace_entry_point_twice_in_a_row(gpu_lib):
    lmho = gpu_lib
    lib = lmho.load()
    stream = torch.cuda.current_stream().cuda_stream
    # warp per row (16 KB rows), then CTA per row (80 KB rows), then cluster per row (few long rows)
    cases = [_case(21, 4096, 4096), _case(22, 777, 20000), _case(24, 40, 70000)]
    losses = [torch.full((1,), float("nan"), device="cuda") for _ in cases]
    # calls in a row straight through the C ABI, no sync in between
    for (_, _, zd, td), out in zip(cases, losses):
        rc = _call(lib, zd, td, out, stream)
        assert rc == 0, lmho.strerror(rc)
    torch.cuda.synchronize()
    for (z, t, zd, td), out in zip(cases, losses):
        got = float(out.item())
        want, _ = oracle.ce_f32(z, t)
        assert got == pytest.approx(want, rel=RTOL, abs=ATOL)
        assert got == pytest.approx(float(lmho.ce_fwd_f32(zd, td).item()), rel=RTOL, abs=ATOL)
    # and again through the binding, reusing the scratch left by the calls above
    z, t, zd, td = cases[0]
    again = lmho.ce_fwd_f32_noalloc(zd, td, torch.empty(1, device="cuda"))
    assert float(again.item()) == pytest.approx(oracle.ce_f32(z, t)[0], rel=RTOL, abs=ATOL)


def test_noalloc_changes_no_memory_footprint(gpu_lib):
    lib = gpu_lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    _, _, zd, td = _case(25, 2048, 8192)
    out = torch.empty(1, device="cuda")
    assert _call(lib, zd, td, out, stream) == 0      # first call: address lookup, module loaded
    torch.cuda.synchronize()
    before_torch = torch.cuda.memory_allocated()
    before_free, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _call(lib, zd, td, out, stream) == 0
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == before_torch
    assert torch.cuda.mem_get_info()[0] == before_free


def test_noalloc_rejects_oversize_and_aliasing(gpu_lib):
    lib = gpu_lib.load()
    big_T = 65537
    # sizes are checked before any pointer is touched
    assert lib.ce_fwd_f32_noalloc(ctypes.c_void_p(0x10000000), ctypes.c_void_p(0x20000000), big_T, 8,
                                  ctypes.c_void_p(0x30000000), None) == gpu_lib.LMHO_ERR_INVALID_ARG
    _, _, zd, td = _case(23, 16, 64)
    rc = lib.ce_fwd_f32_noalloc(ctypes.c_void_p(zd.data_ptr()), ctypes.c_void_p(td.data_ptr()), 16, 64,
                                ctypes.c_void_p(zd.data_ptr() + 8), None)
    assert rc == gpu_lib.LMHO_ERR_ALIAS


def test_binding_rejects_tensors_on_different_devices(gpu_lib):
    _, _, zd, td = _case(26, 8, 16)
    with pytest.raises((ValueError, TypeError)):
        gpu_lib.ce_fwd_f32_noalloc(zd, td, torch.empty(1))      # loss on the host
