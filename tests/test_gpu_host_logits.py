"""The CE row calls on logits in pinned host memory: the kernels read them over
the host link instead of from HBM, and every result must equal the same call
on device copies bit for bit, for each row decomposition.  The bulk-copy ring
(cp.async.bulk copies of rows into shared memory) is only used for device
memory: forced with host logits, the call takes the automatic choice."""
import numpy as np
import pytest
import torch

import gen
from tests.helpers import to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

VARIANTS = ["auto", "warp", "cta", "cta512", "cluster2", "cluster8", "bulk"]


@pytest.fixture(autouse=True)
def _auto_variant(gpu_lib):
    gpu_lib.set_ce_variant("auto")
    yield
    gpu_lib.set_ce_variant("auto")


def pinned(t):
    return t.cpu().pin_memory()


def device_result(lmho, variant, fn):
    """The same call on device copies, with the decomposition the host call
    takes (the automatic one where the ring is forced)."""
    lmho.set_ce_variant("auto" if variant == "bulk" else variant)
    out = fn()
    lmho.set_ce_variant(variant)
    return out


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("T,V", [(300, 4096), (37, 40000)])
def test_flat_f32_from_pinned_host(gpu_lib, variant, T, V):
    z = to_dev(gen.normal_f32(60, 0, (T, V)))
    t = to_dev(gen.targets(60, 1, (T,), V))
    ws_d = gpu_lib.workspace(gpu_lib.ce_workspace_bytes(T, V))
    ref = device_result(gpu_lib, variant, lambda: gpu_lib.ce_fwd_f32(z, t, ws=ws_d).clone())
    ref_rows = gpu_lib.row_losses(ws_d, T).clone()
    gpu_lib.set_ce_variant(variant)
    ws = gpu_lib.workspace(gpu_lib.ce_workspace_bytes(T, V))
    got = gpu_lib.ce_fwd_f32(pinned(z), pinned(t), ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(got, ref) and torch.equal(gpu_lib.row_losses(ws, T), ref_rows)
    parts_d = device_result(gpu_lib, variant, lambda: gpu_lib.ce_partials_f32(z[:, 100:].contiguous(), t,
                                                                             100).clone())
    parts = gpu_lib.ce_partials_f32(pinned(z[:, 100:].contiguous()), pinned(t), 100)
    torch.cuda.synchronize()
    assert torch.equal(parts, parts_d)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("S,B,V", [(16, 4, 4096), (3, 2, 131072), (5, 3, 1001)])
def test_megatron_bf16_from_pinned_host(gpu_lib, variant, S, B, V):
    z = to_dev_bf16(gen.normal_bf16_bits(61, 0, (S, B, V), sigma=2.0))
    t = to_dev(gen.targets(61, 1, (S, B), V))
    ref = device_result(gpu_lib, variant, lambda: gpu_lib.ce_fwd_sbv_bf16(z, t).clone())
    gpu_lib.set_ce_variant(variant)
    got = gpu_lib.ce_fwd_sbv_bf16(pinned(z), pinned(t))
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    v0 = V // 3
    parts_d = device_result(gpu_lib, variant, lambda: gpu_lib.ce_partials_sbv_bf16(z[:, :, v0:].contiguous(), t,
                                                                                  v0).clone())
    parts = gpu_lib.ce_partials_sbv_bf16(pinned(z[:, :, v0:].contiguous()), pinned(t), v0)
    torch.cuda.synchronize()
    assert torch.equal(parts, parts_d)


def test_pageable_host_memory_is_rejected(gpu_lib):
    z = torch.zeros((4, 64))
    t = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(TypeError):
        gpu_lib.ce_fwd_f32(z, t)
