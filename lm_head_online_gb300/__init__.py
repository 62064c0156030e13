"""GB300 (sm_103a) LM-head losses: softmax cross-entropy over a tokens x vocab
logit matrix (flat fp32 mean and Megatron-layout bf16 per token), fused
linear + cross-entropy and fused linear + generalized JSD.

This module is a thin ctypes binding over the C ABI in ``include/lmho.h``
(``liblmho.so``): it checks tensor dtypes/shapes/devices, passes raw device
pointers and the current CUDA stream, and turns status codes into exceptions.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback, and a missing library is an error.

Build the library with ``python -m lm_head_online_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# LMHO_LIB overrides the library path (to compare builds of the same sources).
LIB_PATH = os.environ.get("LMHO_LIB") or os.path.join(HERE, "_build", "liblmho.so")

LMHO_OK = 0
LMHO_ERR_INVALID_ARG = 1
LMHO_ERR_ALIAS = 2
LMHO_ERR_WORKSPACE = 3
LMHO_ERR_UNSUPPORTED = 4
LMHO_ERR_CUDA = 5
LMHO_ERR_TIMEOUT = 6

# Every symbol declared in include/lmho.h.
EXPORTS = (
    "lmho_strerror", "lmho_version", "ce_workspace_bytes", "ce_fwd_f32", "ce_fwd_f32_noalloc", "ce_fwd_sbv_bf16",
    "ce_partials_sbv_bf16", "ce_partials_f32", "ce_merge_partials",
    "ce_fwd_bwd_f32", "ce_fwd_bwd_sbv_bf16",
    "flce_workspace_bytes", "flce_fwd_bf16", "flce_bwd_workspace_bytes", "flce_fwd_bwd_bf16", "fljsd_workspace_bytes", "fljsd_fwd_bf16", "fljsd_fwd_bf16_ex",
    "fljsd_bwd_workspace_bytes", "fljsd_fwd_bwd_bf16",
    "flce_cpo_workspace_bytes", "flce_cpo_fwd_bf16", "flce_cpo_bwd_workspace_bytes", "flce_cpo_fwd_bwd_bf16",
    "flce_partials_bf16", "flce_shard_bwd_bf16", "flce_shard_bwd_rows_bf16", "cpo_combine_workspace_bytes",
    "cpo_combine_rows", "fljsd_lse_partials_bf16", "lse_merge_partials", "fljsd_terms_bf16", "fljsd_shard_bwd_bf16", "jsd_merge_terms",
    "rows_mean_f32",
    "lmho_ws_status", "lmho_probe_read", "lmho_copy_h2d", "lmho_set_ce_variant", "lmho_set_raster_group", "lmho_set_launch_events", "lmho_set_wait_timeout_ns", "lmho_selftest_wait_timeout",
)

CE_VARIANTS = {"auto": 0, "warp": 1, "cta": 2, "cta512": 3, "cluster2": 4, "cluster4": 5, "cluster8": 6, "bulk": 7}

_lock = threading.Lock()
_lib = None


class LmhoError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status}: {strerror(status)}")


def load():
    """Load liblmho.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m lm_head_online_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i64, sz, f32, u64, ci = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float,
                                     ctypes.c_uint64, ctypes.c_int)
        lib.lmho_strerror.argtypes = [ci]
        lib.lmho_strerror.restype = ctypes.c_char_p
        lib.lmho_version.restype = ci
        lib.ce_workspace_bytes.argtypes = [i64, i64]
        lib.ce_workspace_bytes.restype = sz
        lib.ce_fwd_f32.argtypes = [vp, vp, i64, i64, vp, vp, sz, vp]
        lib.ce_fwd_f32.restype = ci
        lib.ce_fwd_f32_noalloc.argtypes = [vp, vp, i64, i64, vp, vp]
        lib.ce_fwd_f32_noalloc.restype = ci
        lib.ce_fwd_sbv_bf16.argtypes = [vp, vp, i64, i64, i64, vp, vp]
        lib.ce_fwd_sbv_bf16.restype = ci
        lib.ce_partials_sbv_bf16.argtypes = [vp, vp, i64, i64, i64, i64, vp, vp]
        lib.ce_partials_sbv_bf16.restype = ci
        lib.ce_partials_f32.argtypes = [vp, vp, i64, i64, i64, vp, vp]
        lib.ce_partials_f32.restype = ci
        lib.ce_merge_partials.argtypes = [vp, i64, vp, i64, i64, i64, vp, vp]
        lib.ce_merge_partials.restype = ci
        lib.ce_fwd_bwd_f32.argtypes = [vp, vp, i64, i64, f32, vp, vp, vp, sz, vp]
        lib.ce_fwd_bwd_f32.restype = ci
        lib.ce_fwd_bwd_sbv_bf16.argtypes = [vp, vp, i64, i64, i64, vp, f32, vp, vp, vp]
        lib.ce_fwd_bwd_sbv_bf16.restype = ci
        lib.flce_workspace_bytes.argtypes = [i64, i64, i64]
        lib.flce_workspace_bytes.restype = sz
        lib.flce_fwd_bf16.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, sz, vp]
        lib.flce_fwd_bf16.restype = ci
        lib.flce_bwd_workspace_bytes.argtypes = [i64, i64, i64]
        lib.flce_bwd_workspace_bytes.restype = sz
        lib.flce_fwd_bwd_bf16.argtypes = [vp, vp, vp, i64, i64, i64, f32, vp, vp, vp, vp, sz, vp]
        lib.flce_fwd_bwd_bf16.restype = ci
        lib.fljsd_workspace_bytes.argtypes = [i64, i64, i64]
        lib.fljsd_workspace_bytes.restype = sz
        lib.fljsd_fwd_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, f32, vp, vp, sz, vp]
        lib.fljsd_fwd_bf16.restype = ci
        lib.fljsd_fwd_bf16_ex.argtypes = [vp, vp, vp, vp, i64, i64, i64, f32, f32, vp, vp, vp, sz, vp]
        lib.fljsd_fwd_bf16_ex.restype = ci
        lib.fljsd_bwd_workspace_bytes.argtypes = [i64, i64, i64]
        lib.fljsd_bwd_workspace_bytes.restype = sz
        lib.fljsd_fwd_bwd_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, f32, f32, vp, f32, vp, vp, vp, vp, sz, vp]
        lib.fljsd_fwd_bwd_bf16.restype = ci
        lib.flce_cpo_workspace_bytes.argtypes = [i64, i64, i64, i64]
        lib.flce_cpo_workspace_bytes.restype = sz
        lib.flce_cpo_fwd_bf16.argtypes = [vp, vp, vp, i64, i64, i64, i64, f32, f32, vp, vp, vp, sz, vp]
        lib.flce_cpo_fwd_bf16.restype = ci
        lib.flce_cpo_bwd_workspace_bytes.argtypes = [i64, i64, i64, i64]
        lib.flce_cpo_bwd_workspace_bytes.restype = sz
        lib.flce_cpo_fwd_bwd_bf16.argtypes = [vp, vp, vp, i64, i64, i64, i64, f32, f32, f32, vp, vp, vp, vp, vp, sz,
                                              vp]
        lib.flce_cpo_fwd_bwd_bf16.restype = ci
        lib.flce_partials_bf16.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, vp, sz, vp]
        lib.flce_partials_bf16.restype = ci
        lib.flce_shard_bwd_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, vp, vp, vp, sz, vp]
        lib.flce_shard_bwd_bf16.restype = ci
        lib.flce_shard_bwd_rows_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, vp, f32, vp, vp, vp,
                                                 sz, vp]
        lib.flce_shard_bwd_rows_bf16.restype = ci
        lib.cpo_combine_workspace_bytes.argtypes = [i64]
        lib.cpo_combine_workspace_bytes.restype = sz
        lib.cpo_combine_rows.argtypes = [vp, i64, i64, f32, f32, vp, vp, vp, vp, sz, vp]
        lib.cpo_combine_rows.restype = ci
        lib.fljsd_lse_partials_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, f32, vp, vp, sz, vp]
        lib.fljsd_lse_partials_bf16.restype = ci
        lib.lse_merge_partials.argtypes = [vp, i64, i64, vp, vp]
        lib.lse_merge_partials.restype = ci
        lib.fljsd_terms_bf16.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, f32, f32, vp, vp, vp, sz, vp]
        lib.fljsd_terms_bf16.restype = ci
        lib.fljsd_shard_bwd_bf16.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, f32, f32, f32, vp, vp, vp, sz,
                                             vp]
        lib.fljsd_shard_bwd_bf16.restype = ci
        lib.jsd_merge_terms.argtypes = [vp, i64, i64, vp, vp, vp, vp]
        lib.jsd_merge_terms.restype = ci
        lib.rows_mean_f32.argtypes = [vp, i64, vp, vp, vp]
        lib.rows_mean_f32.restype = ci
        lib.lmho_probe_read.argtypes = [vp, i64, i64, vp, vp]
        lib.lmho_probe_read.restype = ci
        lib.lmho_copy_h2d.argtypes = [vp, vp, i64, vp]
        lib.lmho_copy_h2d.restype = ci
        lib.lmho_ws_status.argtypes = [vp, sz, vp]
        lib.lmho_ws_status.restype = ci
        lib.lmho_set_ce_variant.argtypes = [ci]
        lib.lmho_set_ce_variant.restype = ci
        lib.lmho_set_raster_group.argtypes = [ci]
        lib.lmho_set_raster_group.restype = ci
        lib.lmho_set_launch_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ci]
        lib.lmho_set_launch_events.restype = None
        lib.lmho_set_wait_timeout_ns.argtypes = [u64]
        lib.lmho_set_wait_timeout_ns.restype = None
        lib.lmho_selftest_wait_timeout.argtypes = [vp, sz, u64, vp]
        lib.lmho_selftest_wait_timeout.restype = ci
        _lib = lib
    return _lib


def strerror(status: int) -> str:
    try:
        return load().lmho_strerror(int(status)).decode()
    except RuntimeError:
        return "library not loaded"


def _check(status: int, where: str):
    if status != LMHO_OK:
        raise LmhoError(status, where)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, name: str, dtype, ndim=None):
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _host_or_dev(t: torch.Tensor, name: str, dtype, ndim=None):
    """Pointer of a CUDA tensor or of a tensor in pinned host memory (which the
    GPU reads directly over the host link: the CE row calls accept it for their
    logits and targets)."""
    if isinstance(t, torch.Tensor) and t.device.type == "cpu":
        if not t.is_pinned():
            raise TypeError(f"{name} must be a CUDA tensor or in pinned host memory")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if ndim is not None and t.dim() != ndim:
            raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return t.data_ptr()
    return _dev(t, name, dtype, ndim)


def _cuda_device(*tensors):
    """Where a call's outputs go: the device of its first CUDA tensor, else the
    current CUDA device (all inputs in pinned host memory)."""
    for t in tensors:
        if t is not None and t.device.type == "cuda":
            return t.device
    return torch.device("cuda", torch.cuda.current_device())


def _on(*tensors):
    """Context in which a call runs: the device of its CUDA tensors, which must
    all be on one device (the kernels are launched on the current device, with
    the current stream of that device).  Pinned host tensors are skipped."""
    cuda = [t for t in tensors if t is not None and t.device.type == "cuda"]
    if not cuda:
        raise ValueError("a call needs at least one CUDA tensor")
    dev = cuda[0].device
    for t in cuda[1:]:
        if t.device != dev:
            raise ValueError(f"tensors on different devices: {dev} and {t.device}")
    return torch.cuda.device(dev)


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """Zero-filled device workspace (torch allocations are 512-byte aligned)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


# ---------------------------------------------------------------- sizes
def ce_workspace_bytes(T: int, V: int) -> int:
    return int(load().ce_workspace_bytes(T, V))


def flce_workspace_bytes(T: int, H: int, V: int) -> int:
    return int(load().flce_workspace_bytes(T, H, V))


def fljsd_workspace_bytes(T: int, H: int, V: int) -> int:
    return int(load().fljsd_workspace_bytes(T, H, V))


# ---------------------------------------------------------------- ops
def ce_fwd_f32(logits, target, loss=None, ws=None, stream=None):
    """Mean cross-entropy of fp32 logits [T, V] against int64 targets [T] -> fp32 [1].

    After the stream reaches this call's end, ``ws[:4*T]`` viewed as float32
    holds the per-token losses.  logits and target may be CUDA tensors or in
    pinned host memory (read directly over the host link).
    """
    lib = load()
    pl = _host_or_dev(logits, "logits", torch.float32, 2)
    T, V = logits.shape
    pt = _host_or_dev(target, "target", torch.int64, 1)
    if target.shape[0] != T:
        raise ValueError("target must have T entries")
    dev = _cuda_device(loss, ws, logits, target)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(lib.ce_workspace_bytes(T, V), dev)
    with _on(logits, target, loss, ws):
        _check(lib.ce_fwd_f32(pl, pt, T, V, _dev(loss, "loss", torch.float32), _dev(ws, "ws", torch.uint8),
                              ws.numel(), _stream(stream)), "ce_fwd_f32")
    return loss


def ce_fwd_f32_noalloc(logits, target, loss, stream=None):
    """ce_fwd_f32 for callers that cannot allocate device memory (a fixed
    device-memory budget owned by someone else): no workspace argument, the
    library's own scratch (at most 65536 tokens) is used instead.  ``loss``
    (fp32 [1], on the device) must be supplied by the caller, since this call
    allocates nothing.  Calls that overlap on the GPU share the scratch and
    race: serialise them."""
    lib = load()
    pl = _dev(logits, "logits", torch.float32, 2)
    T, V = logits.shape
    pt = _dev(target, "target", torch.int64, 1)
    if target.shape[0] != T:
        raise ValueError("target must have T entries")
    pd = _dev(loss, "loss", torch.float32)
    with _on(logits, target, loss):
        _check(lib.ce_fwd_f32_noalloc(pl, pt, T, V, pd, _stream(stream)), "ce_fwd_f32_noalloc")
    return loss


def ce_fwd_sbv_bf16(logits, target, loss=None, stream=None):
    """Per-token cross-entropy of bf16 logits [S, B, V] -> fp32 [S, B].
    logits and target may be CUDA tensors or in pinned host memory."""
    lib = load()
    pl = _host_or_dev(logits, "logits", torch.bfloat16, 3)
    S, B, V = logits.shape
    pt = _host_or_dev(target, "target", torch.int64, 2)
    if tuple(target.shape) != (S, B):
        raise ValueError("target must be [S, B]")
    if loss is None:
        loss = torch.empty((S, B), dtype=torch.float32, device=_cuda_device(logits, target))
    with _on(logits, target, loss):
        _check(lib.ce_fwd_sbv_bf16(pl, pt, S, B, V, _dev(loss, "loss", torch.float32), _stream(stream)),
               "ce_fwd_sbv_bf16")
    return loss


def ce_partials_sbv_bf16(logits_local, target, vocab_start, partials=None, stream=None):
    """One vocabulary shard of the vocab-parallel Megatron cross-entropy.

    logits_local: bf16 [S, B, V_local], the global vocab columns
    [vocab_start, vocab_start + V_local); target: int64 [S, B] global indices.
    Returns fp32 [3, S, B]: the shard's max, sum of exp(z - max), and the
    target logit (-inf where the target is not in this shard).  logits_local
    and target may be CUDA tensors or in pinned host memory."""
    lib = load()
    pl = _host_or_dev(logits_local, "logits_local", torch.bfloat16, 3)
    S, B, Vl = logits_local.shape
    pt = _host_or_dev(target, "target", torch.int64, 2)
    if tuple(target.shape) != (S, B):
        raise ValueError("target must be [S, B]")
    if partials is None:
        partials = torch.empty((3, S, B), dtype=torch.float32, device=_cuda_device(logits_local, target))
    if tuple(partials.shape) != (3, S, B):
        raise ValueError("partials must be [3, S, B]")
    with _on(logits_local, target, partials):
        _check(lib.ce_partials_sbv_bf16(pl, pt, S, B, Vl, int(vocab_start), _dev(partials, "partials", torch.float32, 3),
                                        _stream(stream)), "ce_partials_sbv_bf16")
    return partials


def ce_partials_f32(logits_local, target, vocab_start, partials=None, stream=None):
    """One vocabulary shard of the flat fp32 cross-entropy: logits_local fp32
    [T, V_local] = the global columns [vocab_start, vocab_start + V_local),
    target int64 [T] global.  Returns fp32 [3, T] (max, sum of exp, target
    logit or -inf); merge with ce_merge_partials(p.view(k, 3, T, 1), ...).
    logits_local and target may be CUDA tensors or in pinned host memory."""
    lib = load()
    pl = _host_or_dev(logits_local, "logits_local", torch.float32, 2)
    T, Vl = logits_local.shape
    pt = _host_or_dev(target, "target", torch.int64, 1)
    if target.shape[0] != T:
        raise ValueError("target must be [T]")
    if partials is None:
        partials = torch.empty((3, T), dtype=torch.float32, device=_cuda_device(logits_local, target))
    if tuple(partials.shape) != (3, T):
        raise ValueError("partials must be [3, T]")
    with _on(logits_local, target, partials):
        _check(lib.ce_partials_f32(pl, pt, T, Vl, int(vocab_start), _dev(partials, "partials", torch.float32, 2),
                                   _stream(stream)), "ce_partials_f32")
    return partials


def ce_merge_partials(partials, target, V, loss=None, stream=None):
    """Per-token losses fp32 [S, B] from the partials of every vocabulary
    shard, fp32 [shards, 3, S, B] in shard order; V = global vocabulary size."""
    lib = load()
    pp = _dev(partials, "partials", torch.float32, 4)
    k, three, S, B = partials.shape
    if three != 3:
        raise ValueError("partials must be [shards, 3, S, B]")
    pt = _dev(target, "target", torch.int64, 2)
    if tuple(target.shape) != (S, B):
        raise ValueError("target must be [S, B]")
    if loss is None:
        loss = torch.empty((S, B), dtype=torch.float32, device=partials.device)
    with _on(partials, target, loss):
        _check(lib.ce_merge_partials(pp, k, pt, S, B, int(V), _dev(loss, "loss", torch.float32, 2), _stream(stream)),
               "ce_merge_partials")
    return loss


def ce_fwd_bwd_f32(logits, target, grad_scale=1.0, loss=None, dlogits=None, ws=None, stream=None):
    """Mean cross-entropy of fp32 logits [T, V] and its gradient (times
    grad_scale) with respect to the logits, in one pass.  Returns (loss, dlogits)."""
    lib = load()
    pl = _dev(logits, "logits", torch.float32, 2)
    T, V = logits.shape
    pt = _dev(target, "target", torch.int64, 1)
    if target.shape[0] != T:
        raise ValueError("target must have T entries")
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=logits.device)
    if dlogits is None:
        dlogits = torch.empty_like(logits)
    if tuple(dlogits.shape) != (T, V):
        raise ValueError("dlogits must be [T, V]")
    if ws is None:
        ws = workspace(lib.ce_workspace_bytes(T, V), logits.device)
    with _on(logits, target, loss, dlogits, ws):
        _check(lib.ce_fwd_bwd_f32(pl, pt, T, V, float(grad_scale), _dev(loss, "loss", torch.float32),
                                  _dev(dlogits, "dlogits", torch.float32), _dev(ws, "ws", torch.uint8), ws.numel(),
                                  _stream(stream)), "ce_fwd_bwd_f32")
    return loss, dlogits


def ce_fwd_bwd_sbv_bf16(logits, target, dloss=None, grad_scale=1.0, loss=None, dlogits=None, stream=None):
    """Per-token cross-entropy of bf16 logits [S, B, V] and the gradient of
    grad_scale * sum(dloss * loss) with respect to the logits (bf16).
    Returns (loss [S, B] fp32, dlogits [S, B, V] bf16)."""
    lib = load()
    pl = _dev(logits, "logits", torch.bfloat16, 3)
    S, B, V = logits.shape
    pt = _dev(target, "target", torch.int64, 2)
    if tuple(target.shape) != (S, B):
        raise ValueError("target must be [S, B]")
    pd = None
    if dloss is not None:
        pd = _dev(dloss, "dloss", torch.float32, 2)
        if tuple(dloss.shape) != (S, B):
            raise ValueError("dloss must be [S, B]")
    if loss is None:
        loss = torch.empty((S, B), dtype=torch.float32, device=logits.device)
    if dlogits is None:
        dlogits = torch.empty_like(logits)
    with _on(logits, target, loss, dlogits, dloss):
        _check(lib.ce_fwd_bwd_sbv_bf16(pl, pt, S, B, V, pd, float(grad_scale), _dev(loss, "loss", torch.float32),
                                       _dev(dlogits, "dlogits", torch.bfloat16, 3), _stream(stream)),
               "ce_fwd_bwd_sbv_bf16")
    return loss, dlogits


def flce_fwd_bf16(x, W, target, loss=None, ws=None, stream=None):
    """Mean cross-entropy of z = x W^T (never materialised) -> fp32 [1].

    x is [T, H] or [batch, seq, H] bf16, W [V, H] bf16, target [T] or
    [batch, seq] int64.  ``ws[:4*T]`` (float32) holds the per-token losses.
    """
    lib = load()
    if x.dim() == 3:
        x = x.reshape(-1, x.shape[-1])
    if target.dim() == 2:
        target = target.reshape(-1)
    px = _dev(x, "x", torch.bfloat16, 2)
    pw = _dev(W, "W", torch.bfloat16, 2)
    pt = _dev(target, "target", torch.int64, 1)
    T, H = x.shape
    V = W.shape[0]
    if W.shape[1] != H or target.shape[0] != T:
        raise ValueError("shape mismatch: x [T,H], W [V,H], target [T]")
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(lib.flce_workspace_bytes(T, H, V), x.device)
    with _on(x, W, target, loss, ws):
        _check(lib.flce_fwd_bf16(px, pw, pt, T, H, V, _dev(loss, "loss", torch.float32), _dev(ws, "ws", torch.uint8),
                                 ws.numel(), _stream(stream)), "flce_fwd_bf16")
    return loss


def flce_bwd_workspace_bytes(T: int, H: int, V: int) -> int:
    return int(load().flce_bwd_workspace_bytes(T, H, V))


def flce_fwd_bwd_bf16(x, W, target, grad_scale=1.0, loss=None, dx=None, dW=None, ws=None, stream=None):
    """Mean cross-entropy of z = x W^T and the gradients of grad_scale * loss:
    returns (loss fp32 [1], dx fp32 [T, H], dW fp32 [V, H])."""
    lib = load()
    if x.dim() == 3:
        x = x.reshape(-1, x.shape[-1])
    if target.dim() == 2:
        target = target.reshape(-1)
    px = _dev(x, "x", torch.bfloat16, 2)
    pw = _dev(W, "W", torch.bfloat16, 2)
    pt = _dev(target, "target", torch.int64, 1)
    T, H = x.shape
    V = W.shape[0]
    if W.shape[1] != H or target.shape[0] != T:
        raise ValueError("shape mismatch: x [T,H], W [V,H], target [T]")
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=x.device)
    if dx is None:
        dx = torch.empty((T, H), dtype=torch.float32, device=x.device)
    if dW is None:
        dW = torch.empty((V, H), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(lib.flce_bwd_workspace_bytes(T, H, V), x.device)
    with _on(x, W, target, loss, dx, dW, ws):
        _check(lib.flce_fwd_bwd_bf16(px, pw, pt, T, H, V, float(grad_scale), _dev(loss, "loss", torch.float32),
                                     _dev(dx, "dx", torch.float32, 2), _dev(dW, "dW", torch.float32, 2),
                                     _dev(ws, "ws", torch.uint8), ws.numel(), _stream(stream)), "flce_fwd_bwd_bf16")
    return loss, dx, dW


def flce_cpo_workspace_bytes(B: int, S: int, H: int, V: int) -> int:
    return int(load().flce_cpo_workspace_bytes(B, S, H, V))


def flce_cpo_bwd_workspace_bytes(B: int, S: int, H: int, V: int) -> int:
    return int(load().flce_cpo_bwd_workspace_bytes(B, S, H, V))


def _cpo_shapes(x, W, target):
    if x.dim() != 3 or target.dim() != 2:
        raise ValueError("x must be [B, S, H] and target [B, S] (chosen = first B/2 sequences)")
    B, S, H = x.shape
    V = W.shape[0]
    if W.dim() != 2 or W.shape[1] != H or tuple(target.shape) != (B, S):
        raise ValueError("shape mismatch: x [B,S,H], W [V,H], target [B,S]")
    return B, S, H, V


def flce_cpo_fwd_bf16(x, W, target, beta=0.1, alpha=1.0, loss=None, logps=None, ws=None, stream=None):
    """CPO loss of the fused linear + CE (chosen = first half of the batch):
    returns (loss fp32 [1], sequence log-likelihoods fp32 [B])."""
    lib = load()
    B, S, H, V = _cpo_shapes(x, W, target)
    px = _dev(x, "x", torch.bfloat16, 3)
    pw = _dev(W, "W", torch.bfloat16, 2)
    pt = _dev(target, "target", torch.int64, 2)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=x.device)
    if logps is None:
        logps = torch.empty(B, dtype=torch.float32, device=x.device)
    if logps.numel() != B or loss.numel() < 1:
        raise ValueError("logps must hold B floats, loss at least one")
    if ws is None:
        ws = workspace(lib.flce_cpo_workspace_bytes(B, S, H, V), x.device)
    with _on(x, W, target, loss, logps, ws):
        _check(lib.flce_cpo_fwd_bf16(px, pw, pt, B, S, H, V, float(beta), float(alpha), _dev(loss, "loss", torch.float32),
                                     _dev(logps, "logps", torch.float32, 1), _dev(ws, "ws", torch.uint8), ws.numel(),
                                     _stream(stream)), "flce_cpo_fwd_bf16")
    return loss, logps


def flce_cpo_fwd_bwd_bf16(x, W, target, beta=0.1, alpha=1.0, grad_scale=1.0, loss=None, logps=None, dx=None, dW=None,
                          ws=None, stream=None):
    """CPO loss and the gradients of grad_scale * loss: returns (loss [1],
    logps [B], dx fp32 [B, S, H], dW fp32 [V, H])."""
    lib = load()
    B, S, H, V = _cpo_shapes(x, W, target)
    px = _dev(x, "x", torch.bfloat16, 3)
    pw = _dev(W, "W", torch.bfloat16, 2)
    pt = _dev(target, "target", torch.int64, 2)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=x.device)
    if logps is None:
        logps = torch.empty(B, dtype=torch.float32, device=x.device)
    if dx is None:
        dx = torch.empty((B, S, H), dtype=torch.float32, device=x.device)
    if dW is None:
        dW = torch.empty((V, H), dtype=torch.float32, device=x.device)
    if logps.numel() != B or loss.numel() < 1 or tuple(dx.shape) != (B, S, H) or tuple(dW.shape) != (V, H):
        raise ValueError("output shapes: loss [1], logps [B], dx [B, S, H], dW [V, H]")
    if ws is None:
        ws = workspace(lib.flce_cpo_bwd_workspace_bytes(B, S, H, V), x.device)
    with _on(x, W, target, loss, logps, dx, dW, ws):
        _check(lib.flce_cpo_fwd_bwd_bf16(px, pw, pt, B, S, H, V, float(beta), float(alpha), float(grad_scale),
                                         _dev(loss, "loss", torch.float32), _dev(logps, "logps", torch.float32, 1),
                                         _dev(dx, "dx", torch.float32, 3), _dev(dW, "dW", torch.float32, 2),
                                         _dev(ws, "ws", torch.uint8), ws.numel(), _stream(stream)),
               "flce_cpo_fwd_bwd_bf16")
    return loss, logps, dx, dW


def fljsd_fwd_bf16(xs, Ws, xt, Wt, beta=0.5, loss=None, ws=None, stream=None):
    """Batchmean generalized JSD between softmax(xs Ws^T) (student, P) and
    softmax(xt Wt^T) (teacher, Q) -> fp32 [1].  ``ws[:4*T]`` holds per-token JSD."""
    lib = load()
    p1 = _dev(xs, "xs", torch.bfloat16, 2)
    p2 = _dev(Ws, "Ws", torch.bfloat16, 2)
    p3 = _dev(xt, "xt", torch.bfloat16, 2)
    p4 = _dev(Wt, "Wt", torch.bfloat16, 2)
    T, H = xs.shape
    V = Ws.shape[0]
    if tuple(xt.shape) != (T, H) or tuple(Ws.shape) != (V, H) or tuple(Wt.shape) != (V, H):
        raise ValueError("shape mismatch: xs, xt [T,H]; Ws, Wt [V,H]")
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=xs.device)
    if ws is None:
        ws = workspace(lib.fljsd_workspace_bytes(T, H, V), xs.device)
    with _on(xs, Ws, xt, Wt, loss, ws):
        _check(lib.fljsd_fwd_bf16(p1, p2, p3, p4, T, H, V, float(beta), _dev(loss, "loss", torch.float32),
                                  _dev(ws, "ws", torch.uint8), ws.numel(), _stream(stream)), "fljsd_fwd_bf16")
    return loss


def fljsd_fwd_bf16_ex(xs, Ws, xt, Wt, beta=0.5, temperature=1.0, keep=None, loss=None, ws=None, stream=None):
    """fljsd_fwd_bf16 with logits divided by `temperature` and an optional
    per-token keep mask (CUDA bool/uint8 [T]); the batchmean divides by the
    number of kept tokens."""
    lib = load()
    p1 = _dev(xs, "xs", torch.bfloat16, 2)
    p2 = _dev(Ws, "Ws", torch.bfloat16, 2)
    p3 = _dev(xt, "xt", torch.bfloat16, 2)
    p4 = _dev(Wt, "Wt", torch.bfloat16, 2)
    T, H = xs.shape
    V = Ws.shape[0]
    if tuple(xt.shape) != (T, H) or tuple(Ws.shape) != (V, H) or tuple(Wt.shape) != (V, H):
        raise ValueError("shape mismatch: xs, xt [T,H]; Ws, Wt [V,H]")
    pk = None
    if keep is not None:
        if keep.dtype == torch.bool:
            keep = keep.view(torch.uint8)
        pk = _dev(keep, "keep", torch.uint8, 1)
        if keep.shape[0] != T:
            raise ValueError("keep must have T entries")
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=xs.device)
    if ws is None:
        ws = workspace(lib.fljsd_workspace_bytes(T, H, V), xs.device)
    with _on(xs, Ws, xt, Wt, keep, loss, ws):
        _check(lib.fljsd_fwd_bf16_ex(p1, p2, p3, p4, T, H, V, float(beta), float(temperature), pk,
                                     _dev(loss, "loss", torch.float32), _dev(ws, "ws", torch.uint8), ws.numel(),
                                     _stream(stream)), "fljsd_fwd_bf16_ex")
    return loss


def fljsd_bwd_workspace_bytes(T: int, H: int, V: int) -> int:
    return int(load().fljsd_bwd_workspace_bytes(T, H, V))


def fljsd_fwd_bwd_bf16(xs, Ws, xt, Wt, beta=0.5, temperature=1.0, keep=None, grad_scale=1.0, loss=None, dxs=None,
                       dWs=None, ws=None, stream=None):
    """Fused linear + JSD and the student gradients of grad_scale * loss:
    returns (loss fp32 [1], dxs fp32 [T, H], dWs fp32 [V, H])."""
    lib = load()
    p1 = _dev(xs, "xs", torch.bfloat16, 2)
    p2 = _dev(Ws, "Ws", torch.bfloat16, 2)
    p3 = _dev(xt, "xt", torch.bfloat16, 2)
    p4 = _dev(Wt, "Wt", torch.bfloat16, 2)
    T, H = xs.shape
    V = Ws.shape[0]
    if tuple(xt.shape) != (T, H) or tuple(Ws.shape) != (V, H) or tuple(Wt.shape) != (V, H):
        raise ValueError("shape mismatch: xs, xt [T,H]; Ws, Wt [V,H]")
    pk = None
    if keep is not None:
        if keep.dtype == torch.bool:
            keep = keep.view(torch.uint8)
        pk = _dev(keep, "keep", torch.uint8, 1)
        if keep.shape[0] != T:
            raise ValueError("keep must have T entries")
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=xs.device)
    if dxs is None:
        dxs = torch.empty((T, H), dtype=torch.float32, device=xs.device)
    if dWs is None:
        dWs = torch.empty((V, H), dtype=torch.float32, device=xs.device)
    if ws is None:
        ws = workspace(lib.fljsd_bwd_workspace_bytes(T, H, V), xs.device)
    with _on(xs, Ws, xt, Wt, keep, loss, dxs, dWs, ws):
        _check(lib.fljsd_fwd_bwd_bf16(p1, p2, p3, p4, T, H, V, float(beta), float(temperature), pk, float(grad_scale),
                                      _dev(loss, "loss", torch.float32), _dev(dxs, "dxs", torch.float32, 2),
                                      _dev(dWs, "dWs", torch.float32, 2), _dev(ws, "ws", torch.uint8), ws.numel(),
                                      _stream(stream)), "fljsd_fwd_bwd_bf16")
    return loss, dxs, dWs


# ---------------------------------------------------------------- vocab-parallel fused losses
def _shard_pair(xs, Ws_local, xt, Wt_local):
    pxs = _dev(xs, "xs", torch.bfloat16, 2)
    pws = _dev(Ws_local, "Ws_local", torch.bfloat16, 2)
    pxt = _dev(xt, "xt", torch.bfloat16, 2)
    pwt = _dev(Wt_local, "Wt_local", torch.bfloat16, 2)
    T, H = xs.shape
    Vl = Ws_local.shape[0]
    if tuple(xt.shape) != (T, H) or tuple(Ws_local.shape) != (Vl, H) or tuple(Wt_local.shape) != (Vl, H):
        raise ValueError("shape mismatch: xs, xt [T,H], Ws_local, Wt_local [V_local,H]")
    return (pxs, pws, pxt, pwt), T, H, Vl


def _keep_ptr(keep, T):
    """Device pointer of a token mask (CUDA uint8 or bool [T]; None = all kept)."""
    if keep is None:
        return None
    if keep.dtype == torch.bool:
        keep = keep.view(torch.uint8)
    pk = _dev(keep, "keep", torch.uint8, 1)
    if keep.shape[0] != T:
        raise ValueError("keep must be [T]")
    return pk


def flce_partials_bf16(x, W_local, target, vocab_start, partials=None, ws=None, stream=None):
    """One vocabulary shard of the fused linear + CE: W_local [V_local, H] bf16
    holds the global vocab rows [vocab_start, vocab_start + V_local); x [T, H]
    bf16; target [T] int64 global indices.  Returns fp32 [3, T]: the shard's
    max and sum of exp of x W_local^T per token, and the target logit (-inf
    where the target is not in this shard).  Merge the shards' blocks with
    ce_merge_partials(all.view(k, 3, T, 1), target.view(T, 1), V)."""
    lib = load()
    px = _dev(x, "x", torch.bfloat16, 2)
    pw = _dev(W_local, "W_local", torch.bfloat16, 2)
    pt = _dev(target, "target", torch.int64, 1)
    T, H = x.shape
    Vl = W_local.shape[0]
    if W_local.shape[1] != H or target.shape[0] != T:
        raise ValueError("shape mismatch: x [T,H], W_local [V_local,H], target [T]")
    if partials is None:
        partials = torch.empty((3, T), dtype=torch.float32, device=x.device)
    if tuple(partials.shape) != (3, T):
        raise ValueError("partials must be [3, T]")
    if ws is None:
        ws = workspace(lib.flce_workspace_bytes(T, H, Vl), x.device)
    with _on(x, W_local, target, partials, ws):
        _check(lib.flce_partials_bf16(px, pw, pt, T, H, Vl, int(vocab_start), _dev(partials, "partials", torch.float32, 2),
                                      _dev(ws, "ws", torch.uint8), ws.numel(), _stream(stream)), "flce_partials_bf16")
    return partials


def flce_shard_bwd_bf16(x, W_local, target, partials, vocab_start, V, grad_scale=1.0, dx=None, dW=None, ws=None,
                        stream=None, row_w=None):
    """Backward of one shard of the vocab-parallel fused linear + CE:
    gradients of grad_scale * mean loss.  partials: fp32 [shards, 3, T], every
    shard's flce_partials_bf16 output in shard order; V the global vocabulary.
    Returns (dx_partial fp32 [T, H], this rank's share of dx -- the ranks'
    shares sum to dx --, dW_local fp32 [V_local, H], this rank's rows of dW).
    row_w (fp32 [T], optional): a weight per token in place of the mean's 1/T
    (flce_shard_bwd_rows_bf16), e.g. cpo_combine_rows' weights."""
    lib = load()
    px = _dev(x, "x", torch.bfloat16, 2)
    pw = _dev(W_local, "W_local", torch.bfloat16, 2)
    pt = _dev(target, "target", torch.int64, 1)
    pp = _dev(partials, "partials", torch.float32, 3)
    T, H = x.shape
    Vl = W_local.shape[0]
    k = partials.shape[0]
    if W_local.shape[1] != H or target.shape[0] != T or tuple(partials.shape[1:]) != (3, T):
        raise ValueError("shape mismatch: x [T,H], W_local [V_local,H], target [T], partials [shards,3,T]")
    if dx is None:
        dx = torch.empty((T, H), dtype=torch.float32, device=x.device)
    if dW is None:
        dW = torch.empty((Vl, H), dtype=torch.float32, device=x.device)
    if tuple(dx.shape) != (T, H) or tuple(dW.shape) != (Vl, H):
        raise ValueError("dx must be [T, H] and dW [V_local, H]")
    if ws is None:
        ws = workspace(lib.flce_bwd_workspace_bytes(T, H, Vl), x.device)
    with _on(x, W_local, target, partials, dx, dW, ws, row_w):
        pdx, pdw, pws = _dev(dx, "dx", torch.float32, 2), _dev(dW, "dW", torch.float32, 2), _dev(ws, "ws", torch.uint8)
        if row_w is None:
            _check(lib.flce_shard_bwd_bf16(px, pw, pt, pp, k, T, H, Vl, int(vocab_start), int(V), float(grad_scale),
                                           pdx, pdw, pws, ws.numel(), _stream(stream)), "flce_shard_bwd_bf16")
        else:
            pr = _dev(row_w, "row_w", torch.float32, 1)
            if row_w.shape[0] != T:
                raise ValueError("row_w must be [T]")
            _check(lib.flce_shard_bwd_rows_bf16(px, pw, pt, pp, k, T, H, Vl, int(vocab_start), int(V), pr,
                                                float(grad_scale), pdx, pdw, pws, ws.numel(), _stream(stream)),
                   "flce_shard_bwd_rows_bf16")
    return dx, dW


def cpo_combine_workspace_bytes(B: int) -> int:
    return int(load().cpo_combine_workspace_bytes(B))


def cpo_combine_rows(rows, B, beta=0.1, alpha=1.0, loss=None, logps=None, row_w=None, ws=None, stream=None):
    """The CPO objective of per-token CE losses rows fp32 [B * S] (sequence
    b < B/2 chosen, b + B/2 its rejected answer): returns (loss [1], logps
    [B]); row_w (fp32 [B * S], optional) receives d loss / d rows, the weights
    of the CPO backward (flce_shard_bwd_bf16(..., row_w=row_w))."""
    lib = load()
    pr = _dev(rows, "rows", torch.float32, 1)
    n = rows.shape[0]
    if B < 2 or n % B != 0:
        raise ValueError("rows must hold B sequences of equal length")
    S = n // B
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=rows.device)
    if logps is None:
        logps = torch.empty(B, dtype=torch.float32, device=rows.device)
    pw = None
    if row_w is not None:
        pw = _dev(row_w, "row_w", torch.float32, 1)
        if row_w.shape[0] != n:
            raise ValueError("row_w must be [B * S]")
    if ws is None:
        ws = workspace(lib.cpo_combine_workspace_bytes(B), rows.device)
    with _on(rows, loss, logps, ws, row_w):
        _check(lib.cpo_combine_rows(pr, B, S, float(beta), float(alpha), _dev(loss, "loss", torch.float32),
                                    _dev(logps, "logps", torch.float32, 1), pw, _dev(ws, "ws", torch.uint8),
                                    ws.numel(), _stream(stream)), "cpo_combine_rows")
    return loss, logps


def fljsd_lse_partials_bf16(xs, Ws_local, xt, Wt_local, temperature=1.0, out=None, ws=None, stream=None):
    """Vocab-parallel fused linear + JSD, shard pass 1: fp32 [2, T], each
    head's log-sum-exp of logits / temperature over the shard's columns
    (0 = student xs Ws_local^T, 1 = teacher xt Wt_local^T)."""
    lib = load()
    ptrs, T, H, Vl = _shard_pair(xs, Ws_local, xt, Wt_local)
    if out is None:
        out = torch.empty((2, T), dtype=torch.float32, device=xs.device)
    if tuple(out.shape) != (2, T):
        raise ValueError("out must be [2, T]")
    if ws is None:
        ws = workspace(lib.fljsd_workspace_bytes(T, H, Vl), xs.device)
    with _on(xs, Ws_local, xt, Wt_local, out, ws):
        _check(lib.fljsd_lse_partials_bf16(*ptrs, T, H, Vl, float(temperature), _dev(out, "out", torch.float32, 2),
                                           _dev(ws, "ws", torch.uint8), ws.numel(), _stream(stream)),
               "fljsd_lse_partials_bf16")
    return out


def lse_merge_partials(parts, out=None, stream=None):
    """Global log-sum-exps fp32 [2, T] from every shard's [shards, 2, T] (shard order)."""
    lib = load()
    pp = _dev(parts, "parts", torch.float32, 3)
    k, two, T = parts.shape
    if two != 2:
        raise ValueError("parts must be [shards, 2, T]")
    if out is None:
        out = torch.empty((2, T), dtype=torch.float32, device=parts.device)
    if tuple(out.shape) != (2, T):
        raise ValueError("out must be [2, T]")
    with _on(parts, out):
        _check(lib.lse_merge_partials(pp, k, T, _dev(out, "out", torch.float32, 2), _stream(stream)),
               "lse_merge_partials")
    return out


def fljsd_terms_bf16(xs, Ws_local, xt, Wt_local, lse, beta=0.5, temperature=1.0, out=None, ws=None, stream=None,
                     kl_local=None):
    """Vocab-parallel fused linear + JSD, shard pass 2: with the global
    log-sum-exps lse fp32 [2, T], each token's sum of the JSD terms over the
    shard's columns, fp32 [T].  kl_local (fp32 [T], optional) receives each
    token's share of KL(P || M) over the shard, for the backward."""
    lib = load()
    ptrs, T, H, Vl = _shard_pair(xs, Ws_local, xt, Wt_local)
    pl = _dev(lse, "lse", torch.float32, 2)
    if tuple(lse.shape) != (2, T):
        raise ValueError("lse must be [2, T]")
    if out is None:
        out = torch.empty(T, dtype=torch.float32, device=xs.device)
    if tuple(out.shape) != (T,):
        raise ValueError("out must be [T]")
    pkl = None
    if kl_local is not None:
        pkl = _dev(kl_local, "kl_local", torch.float32, 1)
        if kl_local.shape[0] != T:
            raise ValueError("kl_local must be [T]")
    if ws is None:
        ws = workspace(lib.fljsd_workspace_bytes(T, H, Vl), xs.device)
    with _on(xs, Ws_local, xt, Wt_local, lse, out, ws, kl_local):
        _check(lib.fljsd_terms_bf16(*ptrs, pl, T, H, Vl, float(beta), float(temperature),
                                    _dev(out, "out", torch.float32, 1), pkl, _dev(ws, "ws", torch.uint8), ws.numel(),
                                    _stream(stream)), "fljsd_terms_bf16")
    return out


def fljsd_shard_bwd_bf16(xs, Ws_local, xt, Wt_local, lse, kl, beta=0.5, temperature=1.0, keep=None, grad_scale=1.0,
                         dx=None, dW=None, ws=None, stream=None):
    """Student backward of one shard of the vocab-parallel fused linear + JSD:
    gradients of grad_scale * loss given the global log-sum-exps lse fp32
    [2, T] and each token's KL(P || M) kl fp32 [T] (the shards' kl_local
    summed).  Returns (dxs share fp32 [T, H] -- the ranks' shares sum to the
    student's dx --, dWs rows fp32 [V_local, H])."""
    lib = load()
    ptrs, T, H, Vl = _shard_pair(xs, Ws_local, xt, Wt_local)
    pl = _dev(lse, "lse", torch.float32, 2)
    pk = _dev(kl, "kl", torch.float32, 1)
    if tuple(lse.shape) != (2, T) or kl.shape[0] != T:
        raise ValueError("lse must be [2, T] and kl [T]")
    pm = _keep_ptr(keep, T)
    if dx is None:
        dx = torch.empty((T, H), dtype=torch.float32, device=xs.device)
    if dW is None:
        dW = torch.empty((Vl, H), dtype=torch.float32, device=xs.device)
    if tuple(dx.shape) != (T, H) or tuple(dW.shape) != (Vl, H):
        raise ValueError("dx must be [T, H] and dW [V_local, H]")
    if ws is None:
        ws = workspace(lib.fljsd_bwd_workspace_bytes(T, H, Vl), xs.device)
    with _on(xs, Ws_local, xt, Wt_local, lse, kl, dx, dW, ws, keep):
        _check(lib.fljsd_shard_bwd_bf16(*ptrs, pl, pk, pm, T, H, Vl, float(beta), float(temperature),
                                        float(grad_scale), _dev(dx, "dx", torch.float32, 2),
                                        _dev(dW, "dW", torch.float32, 2), _dev(ws, "ws", torch.uint8), ws.numel(),
                                        _stream(stream)), "fljsd_shard_bwd_bf16")
    return dx, dW


def jsd_merge_terms(terms, keep=None, rows=None, loss=None, stream=None):
    """Per-token JSD fp32 [T] from every shard's term sums [shards, T] (shard
    order; 0 where keep == 0) and its batchmean over the kept tokens: returns
    (loss [1], rows [T])."""
    lib = load()
    pt = _dev(terms, "terms", torch.float32, 2)
    k, T = terms.shape
    pk = _keep_ptr(keep, T)
    if rows is None:
        rows = torch.empty(T, dtype=torch.float32, device=terms.device)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=terms.device)
    if tuple(rows.shape) != (T,):
        raise ValueError("rows must be [T]")
    with _on(terms, rows, loss, keep):
        _check(lib.jsd_merge_terms(pt, k, T, pk, _dev(rows, "rows", torch.float32, 1), _dev(loss, "loss", torch.float32),
                                   _stream(stream)), "jsd_merge_terms")
    return loss, rows


def rows_mean(rows, keep=None, out=None, stream=None):
    """Deterministic mean fp32 [1] of rows fp32 [n] (over keep != 0 when given)."""
    lib = load()
    pr = _dev(rows, "rows", torch.float32, 1)
    n = rows.shape[0]
    pk = _keep_ptr(keep, n)
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=rows.device)
    with _on(rows, out, keep):
        _check(lib.rows_mean_f32(pr, n, pk, _dev(out, "out", torch.float32), _stream(stream)), "rows_mean_f32")
    return out


def row_losses(ws: torch.Tensor, T: int) -> torch.Tensor:
    """Per-token losses (or JSD) left in the first 4*T bytes of a workspace."""
    return ws[: 4 * T].view(torch.float32)


def probe_read(data: torch.Tensor, segment_bytes: int, out=None, stream=None) -> torch.Tensor:
    """Bandwidth probe: read `data` (contiguous, CUDA) in segments of
    segment_bytes with the warp-per-row CE kernel's loads; returns the XOR of
    each segment's words (uint32 as int32 [segments])."""
    if not isinstance(data, torch.Tensor) or data.device.type != "cuda" or not data.is_contiguous():
        raise TypeError("data must be a contiguous CUDA tensor")
    nbytes = data.numel() * data.element_size()
    if segment_bytes <= 0 or nbytes % segment_bytes:
        raise ValueError("data must be a whole number of segments")
    n = nbytes // segment_bytes
    if out is None:
        out = torch.empty(n, dtype=torch.int32, device=data.device)
    _check(load().lmho_probe_read(data.data_ptr(), n, int(segment_bytes), _dev(out, "out", torch.int32, 1),
                                  _stream(stream)), "lmho_probe_read")
    return out


def copy_h2d(dst: torch.Tensor, src: torch.Tensor, stream=None) -> torch.Tensor:
    """Copy `src` (a contiguous tensor in pinned host memory) into `dst` (a
    contiguous CUDA tensor of the same size in bytes) with the library's SM
    copy kernel, on the current stream of dst's device; returns dst."""
    if not isinstance(src, torch.Tensor) or src.device.type != "cpu" or not src.is_pinned():
        raise TypeError("src must be a tensor in pinned host memory")
    if not isinstance(dst, torch.Tensor) or dst.device.type != "cuda":
        raise TypeError("dst must be a CUDA tensor")
    if not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("src and dst must be contiguous")
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("src and dst must hold the same number of bytes")
    with _on(dst):
        _check(load().lmho_copy_h2d(dst.data_ptr(), src.data_ptr(), nbytes, _stream(stream)), "lmho_copy_h2d")
    return dst


def ws_status(ws, stream=None) -> int:
    """Synchronise the stream and return (and clear) the workspace status word."""
    return int(load().lmho_ws_status(_dev(ws, "ws", torch.uint8), ws.numel(), _stream(stream)))


def set_ce_variant(name: str):
    """Row decomposition of the CE calls: auto, warp, cta, cta512, cluster2/4/8, bulk."""
    _check(load().lmho_set_ce_variant(CE_VARIANTS[name]), "lmho_set_ce_variant")


def set_raster_group(group_m: int):
    """Token tiles per raster group of the fused-linear passes (0 = automatic)."""
    _check(load().lmho_set_raster_group(int(group_m)), "lmho_set_raster_group")


def set_launch_events(events):
    """Measurement hook: a list of torch.cuda.Event (enable_timing=True) to be
    recorded around the library's own kernel launches, or None to clear."""
    if not events:
        load().lmho_set_launch_events(None, 0)
        return
    for e in events:   # torch creates the CUDA event lazily, on its first record
        if not e.cuda_event:
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    load().lmho_set_launch_events(arr, len(events))


def set_wait_timeout_ns(ns: int):
    load().lmho_set_wait_timeout_ns(int(ns))


def selftest_wait_timeout(ws, timeout_ns: int, stream=None):
    _check(load().lmho_selftest_wait_timeout(_dev(ws, "ws", torch.uint8), ws.numel(), int(timeout_ns),
                                             _stream(stream)), "lmho_selftest_wait_timeout")
