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


# ---------------------------------------------------------------- gradient error bounds
# The fused backward forms dZ in fp32 from the recomputed logits, rounds it to
# bf16 (round to nearest even) as the operand of the two gradient products,
# and accumulates each product in fp32 on the tensor cores (16 products per
# step) plus at most 8 fp32 slice sums of a split K.  For one element of
# dx = dZ W the error against the exact fp64 product is therefore at most
#   (u_bf16 + acc(K)) * sum_v |dZ_iv| |W_vk|      rounding of dZ, accumulation
#   + e_dz * sum_v S_iv |W_vk|                     dZ's own fp32 error
# with u_bf16 = 2^-8 (8 significant bits), acc(K) = (ceil(K/16) + 16) 2^-24,
# and S the scale of dZ's fp32 error: g * softmax for the cross-entropy
# (dZ = g (p - onehot): the error of p, relative, also at the target where
# dZ itself may be ~0), g beta P for the JSD.  e_dz = 2^-12 covers fp32 logits
# accumulated over H, ex2.approx / lg2.approx (2^-22) and the fp32 merges of
# the log-sum-exp.  dW = dZ^T x takes the same form with x and K = T.
BF16_U = 2.0 ** -8
DZ_ERR = 2.0 ** -12
F32_U = 2.0 ** -24


def acc_err(K):
    return (int(np.ceil(K / 16)) + 16) * F32_U


def grad_bounds(dz, S, x, W):
    """Per-element error bounds of dx = dZ W [T, H] and dW = dZ^T x [V, H]
    (dz, S: [T, V] fp64; x [T, H], W [V, H] as fp64 values)."""
    a, s = np.abs(dz), np.abs(S)
    Wa, xa = np.abs(W), np.abs(x)
    T, V = dz.shape
    bdx = (BF16_U + acc_err(V)) * (a @ Wa) + DZ_ERR * (s @ Wa)
    bdW = (BF16_U + acc_err(T)) * (a.T @ xa) + DZ_ERR * (s.T @ xa)
    return bdx, bdW


def ce_error_scale(dz, target, g_rows):
    """S of the cross-entropy gradient: g_i softmax(z_i) = dZ + g_i onehot(t_i)."""
    S = dz.copy()
    rows = np.arange(dz.shape[0])
    S[rows, target] += g_rows
    return S


def assert_within_bounds(got, ref, bound, what):
    err = np.abs(got - ref)
    bad = ~(err <= bound)      # a NaN anywhere fails
    if bad.any():
        worst = np.nanmax(err / np.maximum(bound, 1e-300))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside their own bound "
                             f"(worst error / bound {worst:.3g})")


def tile_samples(T, groups=(), tile=128, seed=0):
    """Tokens to check at full size: one (at a random offset) from every tile
    of `tile` tokens, the last token, and the tokens on both sides of every
    raster-group boundary of the passes involved (`groups`: token tiles per
    raster group)."""
    rng = np.random.default_rng(seed)
    n_tiles = (T + tile - 1) // tile
    picks = {T - 1}
    for m in range(n_tiles):
        lo, hi = m * tile, min(T, (m + 1) * tile)
        picks.add(int(lo + rng.integers(0, hi - lo)))
    for g in groups:
        for b in range(g * tile, T, g * tile):
            picks.update((b - 1, b))
    return np.array(sorted(picks), np.int64)
