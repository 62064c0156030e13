"""Shared helpers of the GPU parity tests: seeded inputs from ``gen`` moved to
the device unchanged, and the workloads' shapes."""
import numpy as np
import torch

import gen


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> CUDA bf16 tensor with identical bits."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def sample_rows(n_rows: int, k: int, seed: int = 0) -> np.ndarray:
    """k distinct rows, always including the first and last."""
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, max(n_rows - 1, 1)), size=min(k, max(n_rows - 2, 0)), replace=False)
    return np.unique(np.concatenate([[0, n_rows - 1], mid])).astype(np.int64)


def rows_f32(seed, stream, rows, V, sigma=1.0):
    """Selected rows of an fp32 [*, V] generator matrix, made on the host."""
    return np.stack([gen.normal_f32(seed, stream, (V,), sigma, offset=int(r) * V) for r in rows])


def rows_bf16(seed, stream, rows, V, sigma=1.0):
    return np.stack([gen.normal_bf16_bits(seed, stream, (V,), sigma, offset=int(r) * V) for r in rows])
