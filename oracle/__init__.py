"""ORACLE -- test infrastructure only.

ctypes wrapper over ``oracle/oracle.cpp``, the plain fp64 definitions of the
losses.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import this module; the library package never does.

Every function takes host numpy arrays (bf16 tensors as uint16 bit patterns)
and returns float64 results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.cpp")
LIB = os.path.join(HERE, "_build", "liboracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (g++, -O2, no fast-math: IEEE fp64 semantics kept)."""
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-std=c++17", "-O2", "-fno-fast-math", "-ffp-contract=off",
                               "-fPIC", "-shared", "-pthread", SRC, "-o", tmp])
        os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(LIB)
            vp, i64, dbl, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_int
            lib.oracle_ce_f64.argtypes = [vp, vp, i64, i64, vp]
            lib.oracle_ce_f64.restype = dbl
            lib.oracle_ce_f32.argtypes = [vp, vp, i64, i64, vp]
            lib.oracle_ce_f32.restype = dbl
            lib.oracle_ce_sbv_bf16.argtypes = [vp, vp, i64, i64, i64, vp]
            lib.oracle_ce_sbv_bf16.restype = None
            lib.oracle_flce_bf16.argtypes = [vp, vp, vp, i64, i64, i64, vp, ci]
            lib.oracle_flce_bf16.restype = dbl
            lib.oracle_jsd_f64.argtypes = [vp, vp, i64, i64, dbl, vp]
            lib.oracle_jsd_f64.restype = dbl
            lib.oracle_fljsd_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, vp, ci]
            lib.oracle_fljsd_bf16.restype = dbl
            lib.oracle_fljsd_ex_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, dbl, vp, vp, ci]
            lib.oracle_fljsd_ex_bf16.restype = dbl
            lib.oracle_ce_grad_f32.argtypes = [vp, vp, i64, i64, dbl, vp]
            lib.oracle_ce_grad_f32.restype = None
            lib.oracle_ce_grad_f64.argtypes = [vp, vp, i64, i64, vp, dbl, vp]
            lib.oracle_ce_grad_f64.restype = None
            lib.oracle_ce_grad_sbv_bf16.argtypes = [vp, vp, i64, i64, i64, vp, dbl, vp]
            lib.oracle_ce_grad_sbv_bf16.restype = None
            lib.oracle_flce_f64.argtypes = [vp, vp, vp, i64, i64, i64, vp]
            lib.oracle_flce_f64.restype = dbl
            lib.oracle_flce_grad_f64.argtypes = [vp, vp, vp, i64, i64, i64, dbl, vp, vp]
            lib.oracle_flce_grad_f64.restype = None
            lib.oracle_flce_grad_bf16.argtypes = [vp, vp, vp, i64, i64, i64, dbl, vp, vp]
            lib.oracle_flce_grad_bf16.restype = None
            lib.oracle_fljsd_ex_f64.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, dbl, vp, vp]
            lib.oracle_fljsd_ex_f64.restype = dbl
            lib.oracle_fljsd_grad_f64.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, dbl, vp, dbl, vp, vp]
            lib.oracle_fljsd_grad_f64.restype = None
            lib.oracle_fljsd_grad_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, dbl, vp, dbl, vp, vp]
            lib.oracle_fljsd_grad_bf16.restype = None
            lib.oracle_cpo_f64.argtypes = [vp, vp, vp, i64, i64, i64, i64, dbl, dbl, vp, vp]
            lib.oracle_cpo_f64.restype = dbl
            lib.oracle_cpo_bf16.argtypes = [vp, vp, vp, i64, i64, i64, i64, dbl, dbl, vp, vp, ci]
            lib.oracle_cpo_bf16.restype = dbl
            lib.oracle_cpo_combine.argtypes = [vp, i64, i64, dbl, dbl, vp, vp]
            lib.oracle_cpo_combine.restype = dbl
            lib.oracle_cpo_grad_f64.argtypes = [vp, vp, vp, i64, i64, i64, i64, dbl, dbl, dbl, vp, vp]
            lib.oracle_cpo_grad_f64.restype = None
            lib.oracle_cpo_grad_bf16.argtypes = [vp, vp, vp, i64, i64, i64, i64, dbl, dbl, dbl, vp, vp]
            lib.oracle_cpo_grad_bf16.restype = None
            lib.oracle_ce_partials_bf16.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp]
            lib.oracle_ce_partials_bf16.restype = None
            lib.oracle_ce_partials_f32.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp]
            lib.oracle_ce_partials_f32.restype = None
            lib.oracle_ce_merge.argtypes = [vp, vp, vp, i64, vp, i64, i64, vp]
            lib.oracle_ce_merge.restype = None
            lib.oracle_fljsd_dz_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, dbl, vp, dbl, vp, vp]
            lib.oracle_fljsd_dz_bf16.restype = None
            lib.oracle_logits_bf16.argtypes = [vp, vp, i64, i64, i64, vp]
            lib.oracle_logits_bf16.restype = None
            lib.oracle_flce_partials_bf16.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, vp, vp, ci]
            lib.oracle_flce_partials_bf16.restype = None
            lib.oracle_fljsd_lse_shard_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, vp, ci]
            lib.oracle_fljsd_lse_shard_bf16.restype = None
            lib.oracle_lse_merge.argtypes = [vp, i64, i64, vp]
            lib.oracle_lse_merge.restype = None
            lib.oracle_fljsd_terms_shard_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, dbl, vp, vp, ci]
            lib.oracle_fljsd_terms_shard_bf16.restype = None
            lib.oracle_ce_partials_lse.argtypes = [vp, vp, i64, i64, vp]
            lib.oracle_ce_partials_lse.restype = None
            lib.oracle_flce_grad_shard_bf16.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, vp, dbl, vp, vp]
            lib.oracle_flce_grad_shard_bf16.restype = None
            lib.oracle_fljsd_kl_shard_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, dbl, vp, vp, ci]
            lib.oracle_fljsd_kl_shard_bf16.restype = None
            lib.oracle_fljsd_grad_shard_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, dbl, dbl, vp, vp, vp, dbl,
                                                         vp, vp]
            lib.oracle_fljsd_grad_shard_bf16.restype = None
            lib.oracle_jsd_merge.argtypes = [vp, i64, i64, vp, vp]
            lib.oracle_jsd_merge.restype = dbl
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def _threads(threads):
    return int(threads) if threads else (os.cpu_count() or 1)


def ce_f64(z, target):
    """Cross-entropy rows of fp64 logits [T, V]. Returns (mean, per-row losses)."""
    z, pz = _c(z, np.float64)
    T, V = z.shape
    t, pt = _c(target, np.int64)
    out = np.empty(T, np.float64)
    m = _load().oracle_ce_f64(pz, pt, T, V, out.ctypes.data)
    return m, out


def ce_f32(z, target):
    """Flat fp32 logits [T, V]. Returns (mean, per-row losses)."""
    z, pz = _c(z, np.float32)
    T, V = z.shape
    t, pt = _c(target, np.int64)
    out = np.empty(T, np.float64)
    m = _load().oracle_ce_f32(pz, pt, T, V, out.ctypes.data)
    return m, out


def ce_sbv_bf16(z_bits, target):
    """Megatron layout bf16 logits [S, B, V] (uint16 bits). Returns losses [S, B]."""
    z, pz = _c(z_bits, np.uint16)
    S, B, V = z.shape
    t, pt = _c(target, np.int64)
    out = np.empty((S, B), np.float64)
    _load().oracle_ce_sbv_bf16(pz, pt, S, B, V, out.ctypes.data)
    return out


def ce_partials_bf16(z_bits, target, v0):
    """Vocab-parallel CE, one shard: bf16 logits [..., Vl] (uint16 bits) holding
    the global columns [v0, v0 + Vl), global targets [...].  Returns float64
    (m, s, zt), each shaped like target: the shard's max, sum of exp(z - m),
    and the target logit or -inf when the target is not in the shard."""
    z, pz = _c(z_bits, np.uint16)
    Vl = z.shape[-1]
    t, pt = _c(target, np.int64)
    assert z.shape[:-1] == t.shape
    rows = t.size
    m, s, zt = (np.empty(t.shape, np.float64) for _ in range(3))
    _load().oracle_ce_partials_bf16(pz, pt, rows, Vl, int(v0), m.ctypes.data, s.ctypes.data, zt.ctypes.data)
    return m, s, zt


def ce_partials_f32(z, target, v0):
    """ce_partials_bf16 for the flat layout: fp32 logits [T, Vl] holding the
    global columns [v0, v0 + Vl), global targets [T] -> float64 (m, s, zt)."""
    z, pz = _c(z, np.float32)
    Vl = z.shape[-1]
    t, pt = _c(target, np.int64)
    assert z.shape[:-1] == t.shape
    m, s, zt = (np.empty(t.shape, np.float64) for _ in range(3))
    _load().oracle_ce_partials_f32(pz, pt, t.size, Vl, int(v0), m.ctypes.data, s.ctypes.data, zt.ctypes.data)
    return m, s, zt


def ce_merge(m, s, zt, target, V):
    """Per-row losses from k shards' partials m, s, zt (each [k, ...], shard
    order), global targets [...] and the global vocabulary size V."""
    m, pm = _c(m, np.float64)
    s, ps = _c(s, np.float64)
    zt, pz = _c(zt, np.float64)
    t, pt = _c(target, np.int64)
    k = m.shape[0]
    assert m.shape == s.shape == zt.shape and m.shape[1:] == t.shape
    out = np.empty(t.shape, np.float64)
    _load().oracle_ce_merge(pm, ps, pz, k, pt, t.size, int(V), out.ctypes.data)
    return out


def flce_bf16(x_bits, W_bits, target, threads=None):
    """Fused linear + CE. x [T, H], W [V, H] bf16 bits. Returns (mean, per-token)."""
    x, px = _c(x_bits, np.uint16)
    W, pw = _c(W_bits, np.uint16)
    T, H = x.shape
    V = W.shape[0]
    assert W.shape[1] == H
    t, pt = _c(target, np.int64)
    out = np.empty(T, np.float64)
    m = _load().oracle_flce_bf16(px, pw, pt, T, H, V, out.ctypes.data, _threads(threads))
    return m, out


def jsd_f64(zs, zt, beta=0.5):
    """Generalized JSD between softmax(zs) and softmax(zt), rows of [T, V]."""
    zs, ps = _c(zs, np.float64)
    zt, pt = _c(zt, np.float64)
    assert zs.shape == zt.shape
    T, V = zs.shape
    out = np.empty(T, np.float64)
    m = _load().oracle_jsd_f64(ps, pt, T, V, float(beta), out.ctypes.data)
    return m, out


def fljsd_bf16(xs_bits, Ws_bits, xt_bits, Wt_bits, beta=0.5, threads=None):
    """Fused linear + generalized JSD (batchmean). Returns (mean, per-token)."""
    xs, p1 = _c(xs_bits, np.uint16)
    Ws, p2 = _c(Ws_bits, np.uint16)
    xt, p3 = _c(xt_bits, np.uint16)
    Wt, p4 = _c(Wt_bits, np.uint16)
    T, H = xs.shape
    V = Ws.shape[0]
    assert xt.shape == (T, H) and Ws.shape == (V, H) and Wt.shape == (V, H)
    out = np.empty(T, np.float64)
    m = _load().oracle_fljsd_bf16(p1, p2, p3, p4, T, H, V, float(beta), out.ctypes.data,
                                  _threads(threads))
    return m, out


def fljsd_ex_bf16(xs_bits, Ws_bits, xt_bits, Wt_bits, beta=0.5, temperature=1.0, keep=None, threads=None):
    """JSD variant: logits / temperature, optional keep mask (uint8 [T]);
    returns (mean over kept tokens, per-token JSD with 0 for left-out tokens)."""
    xs, p1 = _c(xs_bits, np.uint16)
    Ws, p2 = _c(Ws_bits, np.uint16)
    xt, p3 = _c(xt_bits, np.uint16)
    Wt, p4 = _c(Wt_bits, np.uint16)
    T, H = xs.shape
    V = Ws.shape[0]
    pk = None
    if keep is not None:
        keep, pk = _c(keep, np.uint8)
        assert keep.shape == (T,)
    out = np.empty(T, np.float64)
    m = _load().oracle_fljsd_ex_bf16(p1, p2, p3, p4, T, H, V, float(beta), float(temperature), pk,
                                     out.ctypes.data, _threads(threads))
    return m, out


def ce_grad_f32(z, target, scale=1.0):
    """d(scale * mean CE)/d logits for fp32 logits [T, V] -> fp64 [T, V]."""
    z, pz = _c(z, np.float32)
    T, V = z.shape
    t, pt = _c(target, np.int64)
    dz = np.empty((T, V), np.float64)
    _load().oracle_ce_grad_f32(pz, pt, T, V, float(scale), dz.ctypes.data)
    return dz


def ce_grad_f64(z, target, dloss=None, scale=1.0):
    """d(scale * sum_i dloss_i * loss_i)/d logits for fp64 logits [T, V]."""
    z, pz = _c(z, np.float64)
    T, V = z.shape
    t, pt = _c(target, np.int64)
    pd = None
    if dloss is not None:
        dloss, pd = _c(dloss, np.float64)
    dz = np.empty((T, V), np.float64)
    _load().oracle_ce_grad_f64(pz, pt, T, V, pd, float(scale), dz.ctypes.data)
    return dz


def ce_grad_sbv_bf16(z_bits, target, dloss=None, scale=1.0):
    """Megatron layout: d(scale * sum dloss[s,b] * loss[s,b])/d logits -> fp64 [S, B, V]."""
    z, pz = _c(z_bits, np.uint16)
    S, B, V = z.shape
    t, pt = _c(target, np.int64)
    pd = None
    if dloss is not None:
        dloss, pd = _c(dloss, np.float64)
    dz = np.empty((S, B, V), np.float64)
    _load().oracle_ce_grad_sbv_bf16(pz, pt, S, B, V, pd, float(scale), dz.ctypes.data)
    return dz


def flce_f64(x, W, target):
    """Fused linear + CE on fp64 inputs. Returns (mean, per-token)."""
    x, px = _c(x, np.float64)
    W, pw = _c(W, np.float64)
    T, H = x.shape
    V = W.shape[0]
    t, pt = _c(target, np.int64)
    out = np.empty(T, np.float64)
    m = _load().oracle_flce_f64(px, pw, pt, T, H, V, out.ctypes.data)
    return m, out


def flce_grad_f64(x, W, target, scale=1.0):
    """(dx, dW) of scale * mean fused-linear CE, fp64 inputs."""
    x, px = _c(x, np.float64)
    W, pw = _c(W, np.float64)
    T, H = x.shape
    V = W.shape[0]
    t, pt = _c(target, np.int64)
    dx = np.empty((T, H), np.float64)
    dW = np.empty((V, H), np.float64)
    _load().oracle_flce_grad_f64(px, pw, pt, T, H, V, float(scale), dx.ctypes.data, dW.ctypes.data)
    return dx, dW


def flce_grad_bf16(x_bits, W_bits, target, scale=1.0):
    """(dx, dW) of scale * mean fused-linear CE from bf16 inputs (uint16 bits)."""
    x, px = _c(x_bits, np.uint16)
    W, pw = _c(W_bits, np.uint16)
    T, H = x.shape
    V = W.shape[0]
    t, pt = _c(target, np.int64)
    dx = np.empty((T, H), np.float64)
    dW = np.empty((V, H), np.float64)
    _load().oracle_flce_grad_bf16(px, pw, pt, T, H, V, float(scale), dx.ctypes.data, dW.ctypes.data)
    return dx, dW


def fljsd_ex_f64(xs, Ws, xt, Wt, beta=0.5, temperature=1.0, keep=None):
    """fp64-input fused JSD (mean over kept tokens, per-token JSD)."""
    arrs = [_c(a, np.float64) for a in (xs, Ws, xt, Wt)]
    T, H = arrs[0][0].shape
    V = arrs[1][0].shape[0]
    pk = None
    if keep is not None:
        keep, pk = _c(keep, np.uint8)
    out = np.empty(T, np.float64)
    m = _load().oracle_fljsd_ex_f64(*[a[1] for a in arrs], T, H, V, float(beta), float(temperature), pk,
                                    out.ctypes.data)
    return m, out


def _fljsd_grad(fn, dtype, xs, Ws, xt, Wt, beta, temperature, keep, scale):
    arrs = [_c(a, dtype) for a in (xs, Ws, xt, Wt)]
    T, H = arrs[0][0].shape
    V = arrs[1][0].shape[0]
    pk = None
    if keep is not None:
        keep, pk = _c(keep, np.uint8)
    dxs = np.empty((T, H), np.float64)
    dWs = np.empty((V, H), np.float64)
    fn(*[a[1] for a in arrs], T, H, V, float(beta), float(temperature), pk, float(scale), dxs.ctypes.data,
       dWs.ctypes.data)
    return dxs, dWs


def fljsd_grad_f64(xs, Ws, xt, Wt, beta=0.5, temperature=1.0, keep=None, scale=1.0):
    """Student gradients (dxs, dWs) of scale * fused JSD, fp64 inputs."""
    return _fljsd_grad(_load().oracle_fljsd_grad_f64, np.float64, xs, Ws, xt, Wt, beta, temperature, keep, scale)


def fljsd_grad_bf16(xs, Ws, xt, Wt, beta=0.5, temperature=1.0, keep=None, scale=1.0):
    """Student gradients (dxs, dWs) of scale * fused JSD from bf16 bits."""
    return _fljsd_grad(_load().oracle_fljsd_grad_bf16, np.uint16, xs, Ws, xt, Wt, beta, temperature, keep, scale)


def fljsd_dz_bf16(xs, Ws, xt, Wt, beta=0.5, temperature=1.0, keep=None, scale=1.0):
    """The student's dZs [T, V] (fp64, unrounded) of scale * fused linear + JSD
    (bf16 bit inputs): the operand of its gradient products.  Returns
    (dZs, g beta P), the second being the factor of dZs besides
    ln P - ln M - KL(P || M) (g = scale / (n_kept temperature))."""
    xs, p1 = _c(xs, np.uint16)
    Ws, p2 = _c(Ws, np.uint16)
    xt, p3 = _c(xt, np.uint16)
    Wt, p4 = _c(Wt, np.uint16)
    T, H = xs.shape
    V = Ws.shape[0]
    pk = None
    if keep is not None:
        keep, pk = _c(keep, np.uint8)
    dz = np.empty((T, V), np.float64)
    gbp = np.empty((T, V), np.float64)
    _load().oracle_fljsd_dz_bf16(p1, p2, p3, p4, T, H, V, float(beta), float(temperature), pk, float(scale),
                                 dz.ctypes.data, gbp.ctypes.data)
    return dz, gbp


def logits_bf16(x_bits, W_bits):
    """z = x W^T in fp64 from bf16 bits, x [T, H], W [V, H] -> [T, V]."""
    x, px = _c(x_bits, np.uint16)
    W, pw = _c(W_bits, np.uint16)
    T, H = x.shape
    V = W.shape[0]
    z = np.empty((T, V), np.float64)
    _load().oracle_logits_bf16(px, pw, T, H, V, z.ctypes.data)
    return z


def _cpo_args(x, W, target, dtype):
    x, px = _c(x, dtype)
    W, pw = _c(W, dtype)
    B, S, H = x.shape
    V = W.shape[0]
    assert W.shape[1] == H and B % 2 == 0 and B >= 2
    t, pt = _c(target, np.int64)
    assert t.shape == (B, S)
    return px, pw, pt, B, S, H, V


def cpo_f64(x, W, target, beta=0.1, alpha=1.0):
    """CPO on the fused linear + CE, fp64 inputs x [B, S, H] (chosen = first
    B/2 sequences), W [V, H], target [B, S].  Returns (loss, per-token CE
    losses [B, S], sequence log-likelihoods [B])."""
    px, pw, pt, B, S, H, V = _cpo_args(x, W, target, np.float64)
    rows = np.empty((B, S), np.float64)
    lp = np.empty(B, np.float64)
    m = _load().oracle_cpo_f64(px, pw, pt, B, S, H, V, float(beta), float(alpha), rows.ctypes.data, lp.ctypes.data)
    return m, rows, lp


def cpo_bf16(x_bits, W_bits, target, beta=0.1, alpha=1.0, threads=None):
    """cpo_f64 from bf16 bits (uint16)."""
    px, pw, pt, B, S, H, V = _cpo_args(x_bits, W_bits, target, np.uint16)
    rows = np.empty((B, S), np.float64)
    lp = np.empty(B, np.float64)
    m = _load().oracle_cpo_bf16(px, pw, pt, B, S, H, V, float(beta), float(alpha), rows.ctypes.data, lp.ctypes.data,
                                _threads(threads))
    return m, rows, lp


def cpo_grad_f64(x, W, target, beta=0.1, alpha=1.0, scale=1.0):
    """(dx [B, S, H], dW [V, H]) of scale * CPO loss, fp64 inputs."""
    px, pw, pt, B, S, H, V = _cpo_args(x, W, target, np.float64)
    dx = np.empty((B, S, H), np.float64)
    dW = np.empty((V, H), np.float64)
    _load().oracle_cpo_grad_f64(px, pw, pt, B, S, H, V, float(beta), float(alpha), float(scale), dx.ctypes.data,
                                dW.ctypes.data)
    return dx, dW


def cpo_grad_bf16(x_bits, W_bits, target, beta=0.1, alpha=1.0, scale=1.0):
    """cpo_grad_f64 from bf16 bits (uint16)."""
    px, pw, pt, B, S, H, V = _cpo_args(x_bits, W_bits, target, np.uint16)
    dx = np.empty((B, S, H), np.float64)
    dW = np.empty((V, H), np.float64)
    _load().oracle_cpo_grad_bf16(px, pw, pt, B, S, H, V, float(beta), float(alpha), float(scale), dx.ctypes.data,
                                 dW.ctypes.data)
    return dx, dW


def cpo_combine(rows, beta=0.1, alpha=1.0):
    """The CPO combination of given per-token CE losses rows [B, S]: returns
    (loss, lp [B], d loss / d l [B, S])."""
    r, pr = _c(rows, np.float64)
    B, S = r.shape
    lp = np.empty(B, np.float64)
    w = np.empty((B, S), np.float64)
    m = _load().oracle_cpo_combine(pr, B, S, float(beta), float(alpha), lp.ctypes.data, w.ctypes.data)
    return m, lp, w


def flce_partials_bf16(x_bits, Wl_bits, target, v0, threads=None):
    """Vocab-parallel fused linear + CE, one shard: x [T, H], Wl [Vl, H] (bf16
    bits) = the global vocab rows [v0, v0 + Vl), global targets [T].  Returns
    float64 (m, s, zt) [T] of the shard's logits x Wl^T."""
    x, px = _c(x_bits, np.uint16)
    Wl, pw = _c(Wl_bits, np.uint16)
    t, pt = _c(target, np.int64)
    T, H = x.shape
    Vl = Wl.shape[0]
    assert Wl.shape[1] == H and t.shape == (T,)
    m, s, zt = (np.empty(T, np.float64) for _ in range(3))
    _load().oracle_flce_partials_bf16(px, pw, pt, T, H, Vl, int(v0), m.ctypes.data, s.ctypes.data, zt.ctypes.data,
                                      _threads(threads))
    return m, s, zt


def _two_heads(xs_bits, Wsl_bits, xt_bits, Wtl_bits):
    xs, p1 = _c(xs_bits, np.uint16)
    Ws, p2 = _c(Wsl_bits, np.uint16)
    xt, p3 = _c(xt_bits, np.uint16)
    Wt, p4 = _c(Wtl_bits, np.uint16)
    T, H = xs.shape
    Vl = Ws.shape[0]
    assert xt.shape == (T, H) and Ws.shape == (Vl, H) and Wt.shape == (Vl, H)
    return (xs, Ws, xt, Wt), (p1, p2, p3, p4), T, H, Vl


def fljsd_lse_shard_bf16(xs_bits, Wsl_bits, xt_bits, Wtl_bits, temperature=1.0, threads=None):
    """Vocab-parallel fused linear + JSD, one shard: each head's log-sum-exp
    over the shard's columns of logits / temperature -> float64 [2, T]
    (0 = student, 1 = teacher)."""
    keep_alive, ptrs, T, H, Vl = _two_heads(xs_bits, Wsl_bits, xt_bits, Wtl_bits)
    lse = np.empty((2, T), np.float64)
    _load().oracle_fljsd_lse_shard_bf16(*ptrs, T, H, Vl, float(temperature), lse.ctypes.data, _threads(threads))
    return lse


def lse_merge(parts):
    """Global log-sum-exps [2, T] from k shards' [k, 2, T], in shard order."""
    p, pp = _c(parts, np.float64)
    k, two, T = p.shape
    assert two == 2
    out = np.empty((2, T), np.float64)
    _load().oracle_lse_merge(pp, k, T, out.ctypes.data)
    return out


def fljsd_terms_shard_bf16(xs_bits, Wsl_bits, xt_bits, Wtl_bits, lse, beta=0.5, temperature=1.0, threads=None):
    """Vocab-parallel fused linear + JSD, one shard: with the global
    log-sum-exps lse [2, T], each token's sum of the JSD terms over the
    shard's columns -> float64 [T]."""
    keep_alive, ptrs, T, H, Vl = _two_heads(xs_bits, Wsl_bits, xt_bits, Wtl_bits)
    lse, pl = _c(lse, np.float64)
    assert lse.shape == (2, T)
    out = np.empty(T, np.float64)
    _load().oracle_fljsd_terms_shard_bf16(*ptrs, T, H, Vl, float(beta), float(temperature), pl, out.ctypes.data,
                                          _threads(threads))
    return out


def jsd_merge(terms, keep=None):
    """Per-token JSD [T] from k shards' term sums [k, T] (0 where keep is 0)
    and their batchmean over kept tokens: returns (mean, rows)."""
    tm, pt = _c(terms, np.float64)
    k, T = tm.shape
    pk = None
    if keep is not None:
        keep, pk = _c(keep, np.uint8)
        assert keep.shape == (T,)
    rows = np.empty(T, np.float64)
    m = _load().oracle_jsd_merge(pt, k, T, pk, rows.ctypes.data)
    return m, rows


def ce_partials_lse(m, s):
    """Each row's global log-sum-exp [...] from k shards' CE partials m, s
    (each [k, ...], shard order)."""
    m, pm = _c(m, np.float64)
    s, ps = _c(s, np.float64)
    assert m.shape == s.shape
    k = m.shape[0]
    out = np.empty(m.shape[1:], np.float64)
    _load().oracle_ce_partials_lse(pm, ps, k, out.size, out.ctypes.data)
    return out


def flce_grad_shard_bf16(x_bits, Wl_bits, target, v0, V, lse, scale=1.0):
    """Backward of one shard of the vocab-parallel fused linear + CE: with the
    tokens' global log-sum-exps lse [T], returns float64 (dx_partial [T, H],
    dWl [Vl, H]) of scale * mean loss (the shards' dx_partial sum to dx)."""
    x, px = _c(x_bits, np.uint16)
    Wl, pw = _c(Wl_bits, np.uint16)
    t, pt = _c(target, np.int64)
    lse, pl = _c(lse, np.float64)
    T, H = x.shape
    Vl = Wl.shape[0]
    assert Wl.shape[1] == H and t.shape == (T,) and lse.shape == (T,)
    dx = np.empty((T, H), np.float64)
    dW = np.empty((Vl, H), np.float64)
    _load().oracle_flce_grad_shard_bf16(px, pw, pt, T, H, Vl, int(v0), int(V), pl, float(scale), dx.ctypes.data,
                                        dW.ctypes.data)
    return dx, dW


def fljsd_kl_shard_bf16(xs_bits, Wsl_bits, xt_bits, Wtl_bits, lse, beta=0.5, temperature=1.0, threads=None):
    """Vocab-parallel fused linear + JSD backward, one shard: with the global
    log-sum-exps lse [2, T], each token's share of KL(P || M) over the shard's
    columns -> float64 [T] (the shares sum to KL)."""
    keep_alive, ptrs, T, H, Vl = _two_heads(xs_bits, Wsl_bits, xt_bits, Wtl_bits)
    lse, pl = _c(lse, np.float64)
    assert lse.shape == (2, T)
    out = np.empty(T, np.float64)
    _load().oracle_fljsd_kl_shard_bf16(*ptrs, T, H, Vl, float(beta), float(temperature), pl, out.ctypes.data,
                                       _threads(threads))
    return out


def fljsd_grad_shard_bf16(xs_bits, Wsl_bits, xt_bits, Wtl_bits, lse, kl, beta=0.5, temperature=1.0, keep=None,
                          scale=1.0):
    """Student backward of one shard of the vocab-parallel fused linear + JSD:
    with the global log-sum-exps lse [2, T] and KL(P || M) kl [T], returns
    float64 (dxs share [T, H], dWs rows [Vl, H]) of scale * loss."""
    keep_alive, ptrs, T, H, Vl = _two_heads(xs_bits, Wsl_bits, xt_bits, Wtl_bits)
    lse, pl = _c(lse, np.float64)
    kl, pk = _c(kl, np.float64)
    assert lse.shape == (2, T) and kl.shape == (T,)
    pm = None
    if keep is not None:
        keep, pm = _c(keep, np.uint8)
        assert keep.shape == (T,)
    dx = np.empty((T, H), np.float64)
    dW = np.empty((Vl, H), np.float64)
    _load().oracle_fljsd_grad_shard_bf16(*ptrs, T, H, Vl, float(beta), float(temperature), pm, pl, pk, float(scale),
                                         dx.ctypes.data, dW.ctypes.data)
    return dx, dW
