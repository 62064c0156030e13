"""lmho_copy_h2d: the SM-driven host -> device copy.  Every byte of a pinned
host buffer must arrive unchanged, for sizes from one 16-byte word to more
than one grid-stride round and with a ragged last round; host memory that is
not pinned, or a destination that is not device memory, is rejected; and the
copy is exact while a fused tensor-core pass runs beside it on another
stream."""
import numpy as np
import pytest
import torch

import gen
from tests.helpers import to_dev_bf16

pytestmark = pytest.mark.gpu


def pinned_bytes(seed, n):
    return torch.from_numpy(gen.normal_f32(seed, 0, (n // 4,)).view(np.uint8).copy()).pin_memory()


@pytest.mark.parametrize("nbytes", [16, 4096 + 16, 76 * 128 * 8 * 16, 76 * 128 * 8 * 16 * 3 + 48, 1 << 26])
def test_copy_is_exact(gpu_lib, nbytes):
    src = pinned_bytes(70, nbytes)
    dst = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")
    gpu_lib.copy_h2d(dst, src)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src)


def test_copy_into_a_slice_leaves_the_rest(gpu_lib):
    src = pinned_bytes(71, 1 << 20)
    big = torch.full((3 << 20,), 7, dtype=torch.uint8, device="cuda")
    gpu_lib.copy_h2d(big[1 << 20:2 << 20], src)
    torch.cuda.synchronize()
    host = big.cpu()
    assert torch.equal(host[1 << 20:2 << 20], src)
    assert bool((host[:1 << 20] == 7).all()) and bool((host[2 << 20:] == 7).all())


def test_rejections(gpu_lib):
    from lm_head_online_gb300 import LmhoError
    dst = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(TypeError):
        gpu_lib.copy_h2d(dst, torch.zeros(1024, dtype=torch.uint8))           # pageable host memory
    with pytest.raises(ValueError):
        gpu_lib.copy_h2d(dst, torch.zeros(512, dtype=torch.uint8).pin_memory())
    lib = gpu_lib.load()
    src = torch.zeros(1024, dtype=torch.uint8).pin_memory()
    pageable = torch.zeros(1024, dtype=torch.uint8)
    assert lib.lmho_copy_h2d(dst.data_ptr(), pageable.data_ptr(), 1024, None) == 1    # src not pinned
    other = torch.zeros(1024, dtype=torch.uint8).pin_memory()
    assert lib.lmho_copy_h2d(other.data_ptr(), src.data_ptr(), 1024, None) == 1      # dst in host memory
    assert lib.lmho_copy_h2d(dst.data_ptr(), src.data_ptr(), 1000, None) == 1        # not whole words
    with pytest.raises(LmhoError):
        gpu_lib.copy_h2d(dst[8:24], src[:16])                                         # dst not 16-byte aligned


def test_copy_beside_a_fused_pass(gpu_lib):
    T, H, V = 1024, 4096, 32768
    x = to_dev_bf16(gen.normal_bf16_bits(72, 2, (T, H)))
    W = to_dev_bf16(gen.normal_bf16_bits(72, 3, (V, H), sigma=0.02))
    t = torch.randint(0, V, (T,), device="cuda")
    ws = gpu_lib.workspace(gpu_lib.flce_workspace_bytes(T, H, V))
    ref = gpu_lib.flce_fwd_bf16(x, W, t, ws=ws).clone()
    src = pinned_bytes(73, 1 << 28)
    dst = torch.zeros(1 << 28, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        gpu_lib.copy_h2d(dst, src)
    loss = torch.empty(1, device="cuda")
    for _ in range(3):
        gpu_lib.flce_fwd_bf16(x, W, t, loss=loss, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src)
    assert torch.equal(loss, ref)


def test_copy_from_registered_host_memory(gpu_lib):
    # host memory made page-locked with cudaHostRegister (not allocated by CUDA):
    # the library reads it through the registration's device mapping
    cudart = torch.cuda.cudart()
    arr = np.frombuffer(gen.normal_f32(74, 0, (1 << 18,)).tobytes(), dtype=np.uint8).copy()
    host = torch.from_numpy(arr)
    assert int(cudart.cudaHostRegister(host.data_ptr(), host.numel(), 0)) == 0
    try:
        assert host.is_pinned()
        dst = torch.zeros(host.numel(), dtype=torch.uint8, device="cuda")
        gpu_lib.copy_h2d(dst, host)
        torch.cuda.synchronize()
        assert torch.equal(dst.cpu(), host)
    finally:
        torch.cuda.synchronize()
        cudart.cudaHostUnregister(host.data_ptr())
