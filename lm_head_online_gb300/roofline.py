"""Algorithmic work of each operation (the numerators of the roofline).

Cross-entropy is bandwidth-bound: its algorithmic traffic counts every
declared tensor crossing HBM exactly once, the byte model the operation pages
use for their "Estimated floor" (DRAM floor: every declared tensor crosses
HBM once at the datasheet bandwidth).  The fused-linear operations are
compute-bound: their work is the multiply-adds of the logit GEMMs, 2*T*V*H
flops per head per pass (fused linear + CE: one head, one pass; fused linear
+ JSD: two heads, two passes, since the mixture M couples both normalisers
and the logits are never stored).
"""
from __future__ import annotations


def ce_flat_bytes(T: int, V: int) -> int:
    """fp32 logits [T, V] + int64 targets [T] + fp32 loss [1]."""
    return 4 * T * V + 8 * T + 4


def ce_sbv_bytes(S: int, B: int, V: int, logit_bytes: int = 2) -> int:
    """logits [S, B, V] + int64 targets [S, B] + fp32 losses [S, B]."""
    return logit_bytes * S * B * V + 8 * S * B + 4 * S * B


def ce_flat_fwd_bwd_bytes(T: int, V: int) -> int:
    """Forward + backward: logits read once and the fp32 gradient written once."""
    return ce_flat_bytes(T, V) + 4 * T * V


def ce_sbv_fwd_bwd_bytes(S: int, B: int, V: int, with_dloss: bool = False) -> int:
    """Forward + backward, Megatron layout: bf16 logits read, bf16 gradient written."""
    return ce_sbv_bytes(S, B, V) + 2 * S * B * V + (4 * S * B if with_dloss else 0)


def flce_bytes(T: int, H: int, V: int) -> int:
    """bf16 x [T, H] + bf16 W [V, H] + int64 targets [T] + fp32 loss [1]."""
    return 2 * T * H + 2 * V * H + 8 * T + 4


def fljsd_bytes(T: int, H: int, V: int) -> int:
    """Two bf16 inputs [T, H] + two bf16 heads [V, H] + fp32 loss [1]."""
    return 2 * (2 * T * H) + 2 * (2 * V * H) + 4


def flce_flops(T: int, H: int, V: int) -> int:
    return 2 * T * V * H


def flce_fwd_bwd_flops(T: int, H: int, V: int) -> int:
    """Forward (one GEMM), the recomputation of the logit tiles for dZ, and the
    two gradient products dx = dZ W and dW = dZ^T x: four T x V x H GEMMs."""
    return 8 * T * V * H


def fljsd_flops(T: int, H: int, V: int) -> int:
    """Both passes, both heads."""
    return 8 * T * V * H


def fljsd_fwd_bwd_flops(T: int, H: int, V: int) -> int:
    """Forward (two passes over both heads), a third pass over both heads for
    the student's dZ, and the two student gradient products."""
    return 16 * T * V * H


def fljsd_pass_flops(T: int, H: int, V: int) -> int:
    """One pass over both heads (the log-sum-exp pass or the divergence pass)."""
    return 4 * T * V * H


def floor_us(nbytes: int, gbps: float) -> float:
    return nbytes / (gbps * 1e9) * 1e6
