"""Host-side checks of the C-ABI library (no GPU): it loads, exports every
symbol include/lmho.h declares, and rejects bad arguments before touching a
device."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lmho.h")


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401  (loads the CUDA runtime the library links against)
    from lm_head_online_gb300 import build
    import lm_head_online_gb300 as lmho
    build.build()
    return lmho.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\**\s+\**([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("ce_fwd_f32", "ce_fwd_sbv_bf16", "flce_fwd_bf16", "fljsd_fwd_bf16",
              "ce_workspace_bytes", "flce_workspace_bytes", "fljsd_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import lm_head_online_gb300 as lmho
    names = declared_functions()
    assert set(names) == set(lmho.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_and_version(lib):
    import lm_head_online_gb300 as lmho
    assert lib.lmho_version() >= 200
    for code in range(0, 8):
        assert isinstance(lmho.strerror(code), str) and lmho.strerror(code)


def test_workspace_sizes(lib):
    import lm_head_online_gb300 as lmho
    assert lmho.ce_workspace_bytes(16384, 4096) >= 4 * 16384 + 256
    assert lmho.ce_workspace_bytes(16384, 4096) % 256 == 0
    f = lmho.flce_workspace_bytes(2048, 4096, 128256)
    assert f % 256 == 0 and f >= 4 * 2048 + 3 * 4 * 2048 * 501
    j = lmho.fljsd_workspace_bytes(1024, 4096, 128256)
    assert j % 256 == 0 and j >= 4 * 1024 * (1 + 2 * 2 * 501 + 2)


# Fake, non-dereferenced addresses: validation happens before any device use.
# Every call below must be rejected by a host-side check: one that passed them
# all would launch kernels on these addresses if a GPU were present.
A = 0x10000000
B = 0x20000000
C = 0x30000000
D = 0x40000000


def test_ce_argument_checks(lib):
    assert lib.ce_fwd_f32(None, B, 4, 4, C, D, 4096, None) == 1           # null logits
    assert lib.ce_fwd_f32(A, B, 0, 4, C, D, 4096, None) == 1              # T = 0
    assert lib.ce_fwd_f32(A, B, 4, 0, C, D, 4096, None) == 1              # V = 0
    assert lib.ce_fwd_f32(A, B, 4, 4, C, D, 16, None) == 3                # short workspace
    assert lib.ce_fwd_f32(A, B, 4, 4, C, D + 16, 4096, None) == 3         # misaligned workspace
    assert lib.ce_fwd_f32(A, B, 4, 4, A + 8, D, 4096, None) == 2          # loss inside logits
    assert lib.ce_fwd_f32(A, B, 4, 4, C, A, 4096, None) == 2              # ws over logits
    assert lib.ce_fwd_f32(A, B, 4, 4, D + 64, D, 4096, None) == 2         # loss inside ws
    assert lib.ce_fwd_sbv_bf16(A, B, 2, 2, 8, A + 4, None) == 2           # loss over logits
    assert lib.ce_fwd_sbv_bf16(A, B, 0, 2, 8, C, None) == 1


def test_fused_argument_checks(lib):
    ws = 1 << 30
    assert lib.flce_fwd_bf16(A, B, C, 4, 12, 10, D, D + 4096, ws, None) == 4   # H % 8
    assert lib.flce_fwd_bf16(A + 2, B, C, 4, 16, 10, D, D + 4096, ws, None) == 1  # x not 16-B aligned
    assert lib.flce_fwd_bf16(A, B, C, 4, 16, 10, D, D + 4096, 256, None) == 3
    assert lib.flce_fwd_bf16(A, B, C, 4, 16, 10, A, D + 4096, ws, None) == 2   # loss over x
    assert lib.fljsd_fwd_bf16(A, B, C, D, 4, 16, 10, ctypes.c_float(0.0), D + 8192, D + 16384, ws, None) == 1
    assert lib.fljsd_fwd_bf16(A, B, C, D, 4, 16, 10, ctypes.c_float(1.0), D + 8192, D + 16384, ws, None) == 1
    assert lib.fljsd_fwd_bf16(A, B, C, D, 4, 16, 10, ctypes.c_float(0.5), B + 16, 0x50000000, ws, None) == 2


def test_ce_variant_override_validation(lib):
    assert lib.lmho_set_ce_variant(8) == 1
    assert lib.lmho_set_ce_variant(7) == 0
    assert lib.lmho_set_ce_variant(-1) == 1
    assert lib.lmho_set_ce_variant(0) == 0


def test_raster_group_validation(lib):
    assert lib.lmho_set_raster_group(-1) == 1
    assert lib.lmho_set_raster_group(1025) == 1
    assert lib.lmho_set_raster_group(32) == 0
    assert lib.lmho_set_raster_group(0) == 0


def test_fljsd_ex_argument_checks(lib):
    ws = 1 << 30
    f = ctypes.c_float
    # temperature must be > 0 with a finite reciprocal
    assert lib.fljsd_fwd_bf16_ex(A, B, C, D, 4, 16, 10, f(0.5), f(0.0), None, D + 8192, D + 16384, ws, None) == 1
    assert lib.fljsd_fwd_bf16_ex(A, B, C, D, 4, 16, 10, f(0.5), f(-1.0), None, D + 8192, D + 16384, ws, None) == 1
    assert lib.fljsd_fwd_bf16_ex(A, B, C, D, 4, 16, 10, f(0.5), f(1e-45), None, D + 8192, D + 16384, ws, None) == 1
    # the mask is an input: the loss may not overlap it
    assert lib.fljsd_fwd_bf16_ex(A, B, C, D, 4, 16, 10, f(0.5), f(1.0), 0x60000000, 0x60000001, D + 16384, ws,
                                 None) == 2


def test_ce_backward_argument_checks(lib):
    nan, inf = float("nan"), float("inf")
    E = 0x50000000
    # flat: null dlogits, non-finite grad_scale, short workspace, dlogits over logits / over ws
    assert lib.ce_fwd_bwd_f32(A, B, 4, 4, 1.0, C, None, D, 4096, None) == 1
    assert lib.ce_fwd_bwd_f32(A, B, 4, 4, nan, C, E, D, 4096, None) == 1
    assert lib.ce_fwd_bwd_f32(A, B, 4, 4, inf, C, E, D, 4096, None) == 1
    assert lib.ce_fwd_bwd_f32(A, B, 4, 4, 1.0, C, E, D, 16, None) == 3
    assert lib.ce_fwd_bwd_f32(A, B, 4, 4, 1.0, C, A + 16, D, 4096, None) == 2
    assert lib.ce_fwd_bwd_f32(A, B, 4, 4, 1.0, C, D + 512, D, 4096, None) == 2
    # Megatron: dlogits over the logits, loss over dloss, sizes
    assert lib.ce_fwd_bwd_sbv_bf16(A, B, 2, 2, 8, None, 1.0, C, A + 2, None) == 2
    assert lib.ce_fwd_bwd_sbv_bf16(A, B, 2, 2, 8, E, 1.0, E + 4, C, None) == 2
    assert lib.ce_fwd_bwd_sbv_bf16(A, B, 2, 0, 8, None, 1.0, C, E, None) == 1
    assert lib.ce_fwd_bwd_sbv_bf16(A, B, 2, 2, 8, None, nan, C, E, None) == 1


def test_fused_backward_argument_checks(lib):
    ws = 1 << 30
    E, F = 0x50000000, 0x60000000
    # flce: H % 8, dx misaligned, short workspace, dx over x, dW over W, dx over dW
    assert lib.flce_fwd_bwd_bf16(A, B, C, 4, 12, 10, 1.0, D, E, F, D + 4096, ws, None) == 4
    assert lib.flce_fwd_bwd_bf16(A, B, C, 4, 16, 10, 1.0, D, E + 4, F, D + 4096, ws, None) == 1
    assert lib.flce_fwd_bwd_bf16(A, B, C, 4, 16, 10, float("inf"), D, E, F, D + 4096, ws, None) == 1
    assert lib.flce_fwd_bwd_bf16(A, B, C, 4, 16, 10, 1.0, D, E, F, D + 4096, 256, None) == 3
    assert lib.flce_fwd_bwd_bf16(A, B, C, 4, 16, 10, 1.0, D, A, F, D + 4096, ws, None) == 2
    assert lib.flce_fwd_bwd_bf16(A, B, C, 4, 16, 10, 1.0, D, E, B, D + 4096, ws, None) == 2
    assert lib.flce_fwd_bwd_bf16(A, B, C, 4, 16, 10, 1.0, D, E, E + 16, D + 4096, ws, None) == 2
    # fljsd backward: beta outside (0, 1), temperature <= 0, dWs over Wt
    args = lambda beta, tau, dws: (A, B, C, D, 4, 16, 10, beta, tau, None, 1.0, E, F, dws, 0x70000000, ws, None)  # noqa: E731
    assert lib.fljsd_fwd_bwd_bf16(*args(1.0, 1.0, 0x68000000)) == 1
    assert lib.fljsd_fwd_bwd_bf16(*args(0.5, 0.0, 0x68000000)) == 1
    assert lib.fljsd_fwd_bwd_bf16(*args(0.5, 1.0, D)) == 2


def test_cpo_argument_checks(lib):
    ws = 1 << 30
    E, F = 0x50000000, 0x60000000
    fwd = lambda Bq, S, beta, alpha: lib.flce_cpo_fwd_bf16(A, B, C, Bq, S, 16, 10, beta, alpha, D, None,  # noqa: E731
                                                           D + 4096, ws, None)
    assert fwd(3, 4, 0.1, 1.0) == 1      # odd batch: no chosen/rejected halves
    assert fwd(0, 4, 0.1, 1.0) == 1
    assert fwd(2, 0, 0.1, 1.0) == 1
    assert fwd(2, 4, 0.0, 1.0) == 1      # beta must be > 0
    assert fwd(2, 4, float("nan"), 1.0) == 1
    assert fwd(2, 4, 0.1, -1.0) == 1     # alpha must be >= 0
    assert lib.flce_cpo_fwd_bf16(A, B, C, 2, 4, 12, 10, 0.1, 1.0, D, None, D + 4096, ws, None) == 4   # H % 8
    assert lib.flce_cpo_fwd_bf16(A, B, C, 2, 4, 16, 10, 0.1, 1.0, D, A + 8, D + 4096, ws, None) == 2  # logps over x
    assert lib.flce_cpo_fwd_bf16(A, B, C, 2, 4, 16, 10, 0.1, 1.0, D, None, D + 4096, 256, None) == 3
    # backward: dW over W, non-finite grad_scale, misaligned dx
    assert lib.flce_cpo_fwd_bwd_bf16(A, B, C, 2, 4, 16, 10, 0.1, 1.0, 1.0, D, None, E, B, D + 4096, ws, None) == 2
    assert lib.flce_cpo_fwd_bwd_bf16(A, B, C, 2, 4, 16, 10, 0.1, 1.0, float("inf"), D, None, E, F, D + 4096, ws,
                                     None) == 1
    assert lib.flce_cpo_fwd_bwd_bf16(A, B, C, 2, 4, 16, 10, 0.1, 1.0, 1.0, D, None, E + 4, F, D + 4096, ws, None) == 1


def test_backward_workspace_sizes(lib):
    import lm_head_online_gb300 as lmho
    T, H, V = 2048, 4096, 128256
    fwd, bwd = lmho.flce_workspace_bytes(T, H, V), lmho.flce_bwd_workspace_bytes(T, H, V)
    # the backward keeps bf16 dZ [T, V padded to whole 256-column tiles] beyond the forward's
    assert bwd % 256 == 0 and bwd >= fwd + 2 * T * ((V + 255) // 256 * 256)
    # small T x H: room for up to 8 fp32 K slices of the [T, H] product dx
    assert lmho.flce_bwd_workspace_bytes(256, 512, 4096) >= 8 * 4 * 256 * 512
    assert lmho.fljsd_bwd_workspace_bytes(1024, H, V) >= lmho.fljsd_workspace_bytes(1024, H, V) + 2 * 1024 * V
    c, cb = lmho.flce_cpo_workspace_bytes(2, 1024, H, V), lmho.flce_cpo_bwd_workspace_bytes(2, 1024, H, V)
    assert c >= lmho.flce_workspace_bytes(2048, H, V) and cb >= lmho.flce_bwd_workspace_bytes(2048, H, V)


def test_vocab_parallel_argument_checks(lib):
    # ce_partials_sbv_bf16(logits_local, target, S, B, V_local, vocab_start, partials, stream)
    assert lib.ce_partials_sbv_bf16(None, B, 2, 2, 8, 0, C, None) == 1          # null logits
    assert lib.ce_partials_sbv_bf16(A, B, 0, 2, 8, 0, C, None) == 1             # S = 0
    assert lib.ce_partials_sbv_bf16(A, B, 2, 2, 0, 0, C, None) == 1             # V_local = 0
    assert lib.ce_partials_sbv_bf16(A, B, 2, 2, 8, -1, C, None) == 1            # negative vocab start
    assert lib.ce_partials_sbv_bf16(A, B, 2, 2, 8, 16, A + 8, None) == 2        # partials over logits
    assert lib.ce_partials_sbv_bf16(A, B, 2, 2, 8, 16, B + 24, None) == 2       # partials over target
    # ce_partials_f32(logits_local, target, T, V_local, vocab_start, partials, stream)
    assert lib.ce_partials_f32(None, B, 4, 8, 0, C, None) == 1
    assert lib.ce_partials_f32(A, B, 0, 8, 0, C, None) == 1
    assert lib.ce_partials_f32(A, B, 4, 8, -1, C, None) == 1
    assert lib.ce_partials_f32(A, B, 4, 8, 0, A + 64, None) == 2                # partials over logits
    # ce_merge_partials(partials, shards, target, S, B, V, loss, stream)
    assert lib.ce_merge_partials(None, 2, B, 2, 2, 16, C, None) == 1
    assert lib.ce_merge_partials(A, 0, B, 2, 2, 16, C, None) == 1               # no shard
    assert lib.ce_merge_partials(A, 2, B, 2, 2, 0, C, None) == 1                # V = 0
    assert lib.ce_merge_partials(A, 2, B, 2, 2, 16, A + 80, None) == 2          # loss inside partials
    assert lib.ce_merge_partials(A, 2, B, 2, 2, 16, B, None) == 2               # loss over target


def test_vocab_parallel_fused_argument_checks(lib):
    ws = 1 << 30
    f = ctypes.c_float
    E = 0x50000000
    # flce_partials_bf16(x, W_local, target, T, H, V_local, vocab_start, partials, ws, ws_bytes, stream)
    assert lib.flce_partials_bf16(None, B, C, 4, 16, 10, 0, D, E, ws, None) == 1         # null x
    assert lib.flce_partials_bf16(A, B, C, 4, 16, 0, 0, D, E, ws, None) == 1             # V_local = 0
    assert lib.flce_partials_bf16(A, B, C, 4, 16, 10, -1, D, E, ws, None) == 1           # negative vocab start
    assert lib.flce_partials_bf16(A, B, C, 4, 12, 10, 0, D, E, ws, None) == 4            # H % 8
    assert lib.flce_partials_bf16(A, B + 2, C, 4, 16, 10, 0, D, E, ws, None) == 1        # W_local unaligned
    assert lib.flce_partials_bf16(A, B, C, 4, 16, 10, 0, D, E, 256, None) == 3           # short workspace
    assert lib.flce_partials_bf16(A, B, C, 4, 16, 10, 0, C + 16, E, ws, None) == 2       # partials over target
    # flce_shard_bwd_bf16(x, W_local, target, partials, shards, T, H, V_local, vocab_start, V, grad_scale,
    #                     dx_partial, dW_local, ws, ws_bytes, stream)
    g = f(1.0)
    assert lib.flce_shard_bwd_bf16(A, B, C, None, 2, 4, 16, 10, 0, 20, g, D, D + 4096, E, ws, None) == 1
    assert lib.flce_shard_bwd_bf16(A, B, C, 0x60000000, 0, 4, 16, 10, 0, 20, g, D, D + 4096, E, ws, None) == 1
    assert lib.flce_shard_bwd_bf16(A, B, C, 0x60000000, 2, 4, 16, 10, 15, 20, g, D, D + 4096, E, ws,
                                   None) == 1                                  # shard past the vocabulary
    assert lib.flce_shard_bwd_bf16(A, B, C, 0x60000000, 2, 4, 16, 10, 0, 20, f(math.inf), D, D + 4096, E, ws,
                                   None) == 1                                  # non-finite scale
    assert lib.flce_shard_bwd_bf16(A, B, C, 0x60000000, 2, 4, 16, 10, 0, 20, g, D + 4, D + 4096, E, ws,
                                   None) == 1                                  # dx not 16-byte aligned
    assert lib.flce_shard_bwd_bf16(A, B, C, 0x60000000, 2, 4, 16, 10, 0, 20, g, D, D + 4096, E, 256,
                                   None) == 3                                  # short workspace
    assert lib.flce_shard_bwd_bf16(A, B, C, 0x60000000, 2, 4, 16, 10, 0, 20, g, 0x60000010, D + 4096, E, ws,
                                   None) == 2                                  # dx over the partials
    # flce_shard_bwd_rows_bf16(..., vocab_start, V, row_w, grad_scale, dx, dW, ws, ws_bytes, stream)
    assert lib.flce_shard_bwd_rows_bf16(A, B, C, 0x60000000, 2, 4, 16, 10, 0, 20, None, g, D, D + 4096, E, ws,
                                        None) == 1                             # null weights
    assert lib.flce_shard_bwd_rows_bf16(A, B, C, 0x60000000, 2, 4, 16, 10, 0, 20, D + 8, g, D, D + 4096, E, ws,
                                        None) == 2                             # weights over dx
    # cpo_combine_rows(rows, B, S, beta, alpha, loss, logps, row_w, ws, ws_bytes, stream)
    cw = lib.cpo_combine_workspace_bytes(4)
    assert cw >= 256 + 2 * 16 and lib.cpo_combine_workspace_bytes(0) == 256
    assert lib.cpo_combine_rows(None, 4, 8, f(0.1), f(1.0), C, None, None, E, cw, None) == 1
    assert lib.cpo_combine_rows(A, 3, 8, f(0.1), f(1.0), C, None, None, E, cw, None) == 1     # odd batch
    assert lib.cpo_combine_rows(A, 4, 8, f(0.0), f(1.0), C, None, None, E, cw, None) == 1     # beta
    assert lib.cpo_combine_rows(A, 4, 8, f(0.1), f(-1.0), C, None, None, E, cw, None) == 1    # alpha
    assert lib.cpo_combine_rows(A, 4, 1 << 62, f(0.1), f(1.0), C, None, None, E, cw, None) == 1   # B * S too large
    assert lib.cpo_combine_rows(A, 4, 8, f(0.1), f(1.0), C, None, None, E, 16, None) == 3     # short workspace
    assert lib.cpo_combine_rows(A, 4, 8, f(0.1), f(1.0), C, None, A + 64, E, cw, None) == 2   # weights over rows
    # fljsd_lse_partials_bf16(xs, Ws, xt, Wt, T, H, V_local, temperature, lse_local, ws, ws_bytes, stream)
    assert lib.fljsd_lse_partials_bf16(A, B, C, D, 4, 16, 10, f(1.0), None, E, ws, None) == 1
    assert lib.fljsd_lse_partials_bf16(A, B, C, D, 4, 16, 10, f(0.0), E + (1 << 31), E, ws, None) == 1
    assert lib.fljsd_lse_partials_bf16(A, B, C, D, 4, 16, 10, f(1.0), E + (1 << 31), E, 256, None) == 3
    assert lib.fljsd_lse_partials_bf16(A, B, C, D, 4, 16, 10, f(1.0), B + 8, E, ws, None) == 2   # over Ws
    # lse_merge_partials(parts, shards, T, lse, stream)
    assert lib.lse_merge_partials(None, 2, 4, C, None) == 1
    assert lib.lse_merge_partials(A, 0, 4, C, None) == 1
    assert lib.lse_merge_partials(A, 2, 0, C, None) == 1
    assert lib.lse_merge_partials(A, 2, 4, A + 32, None) == 2                  # lse inside parts [2][2][4]
    # fljsd_terms_bf16(xs, Ws, xt, Wt, lse, T, H, V_local, beta, temperature, terms, kl_local, ws, ws_bytes,
    #                  stream)
    assert lib.fljsd_terms_bf16(A, B, C, D, None, 4, 16, 10, f(0.5), f(1.0), E + (1 << 31), None, E, ws,
                                None) == 1
    assert lib.fljsd_terms_bf16(A, B, C, D, 0x60000000, 4, 16, 10, f(1.0), f(1.0), E + (1 << 31), None, E, ws,
                                None) == 1                                     # beta not in (0, 1)
    assert lib.fljsd_terms_bf16(A, B, C, D, 0x60000000, 4, 16, 10, f(0.5), f(1.0), 0x60000010, None, E, ws,
                                None) == 2                                     # terms over lse
    assert lib.fljsd_terms_bf16(A, B, C, D, 0x60000000, 4, 16, 10, f(0.5), f(1.0), E + (1 << 31),
                                E + (1 << 31) + 8, E, ws, None) == 2           # kl_local over terms
    # fljsd_shard_bwd_bf16(xs, Ws, xt, Wt, lse, kl, keep, T, H, V_local, beta, temperature, grad_scale, dxs, dWs,
    #                      ws, ws_bytes, stream)
    L_, K_ = 0x60000000, 0x61000000
    assert lib.fljsd_shard_bwd_bf16(A, B, C, D, L_, None, None, 4, 16, 10, f(0.5), f(1.0), f(1.0), E + (1 << 31),
                                    E + (1 << 32), E, ws, None) == 1           # null kl
    assert lib.fljsd_shard_bwd_bf16(A, B, C, D, L_, K_, None, 4, 16, 10, f(0.0), f(1.0), f(1.0), E + (1 << 31),
                                    E + (1 << 32), E, ws, None) == 1           # beta
    assert lib.fljsd_shard_bwd_bf16(A, B, C, D, L_, K_, None, 4, 16, 10, f(0.5), f(1.0), f(math.nan),
                                    E + (1 << 31), E + (1 << 32), E, ws, None) == 1   # grad scale
    assert lib.fljsd_shard_bwd_bf16(A, B, C, D, L_, K_, None, 4, 16, 10, f(0.5), f(1.0), f(1.0), E + (1 << 31),
                                    E + (1 << 32), E, 256, None) == 3          # short workspace
    assert lib.fljsd_shard_bwd_bf16(A, B, C, D, L_, K_, None, 4, 16, 10, f(0.5), f(1.0), f(1.0), K_,
                                    E + (1 << 32), E, ws, None) == 2           # dx over kl
    # jsd_merge_terms(terms, shards, T, keep, rows, loss, stream)
    assert lib.jsd_merge_terms(A, 2, 4, None, None, C, None) == 1
    assert lib.jsd_merge_terms(A, 0, 4, None, B, C, None) == 1
    assert lib.jsd_merge_terms(A, 2, 4, None, B + 4, C, None) == 1            # rows not 16-byte aligned
    assert lib.jsd_merge_terms(A, 2, 4, None, A + 16, C, None) == 2           # rows inside terms
    assert lib.jsd_merge_terms(A, 2, 4, D, B, D + 2, None) == 2               # loss over keep
    # rows_mean_f32(rows, n, keep, mean, stream)
    assert lib.rows_mean_f32(None, 4, None, C, None) == 1
    assert lib.rows_mean_f32(A, 0, None, C, None) == 1
    assert lib.rows_mean_f32(A + 4, 4, None, C, None) == 1                    # rows not 16-byte aligned
    assert lib.rows_mean_f32(A, 4, None, A + 8, None) == 2                    # mean inside rows


def test_probe_read_argument_checks(lib):
    # lmho_probe_read(data, segments, segment_bytes, out, stream)
    assert lib.lmho_probe_read(None, 4, 64, C, None) == 1
    assert lib.lmho_probe_read(A, 0, 64, C, None) == 1
    assert lib.lmho_probe_read(A, 4, 24, C, None) == 1            # segment not whole 16-byte vectors
    assert lib.lmho_probe_read(A + 8, 4, 64, C, None) == 1        # data not 16-byte aligned
    assert lib.lmho_probe_read(A, 4, 64, A + 16, None) == 2       # out inside data


def test_copy_h2d_argument_checks(lib):
    # lmho_copy_h2d(dst, src, bytes, stream)
    assert lib.lmho_copy_h2d(A, B, 0, None) == 0                  # nothing to copy: no device touched
    assert lib.lmho_copy_h2d(None, B, 64, None) == 1
    assert lib.lmho_copy_h2d(A, None, 64, None) == 1
    assert lib.lmho_copy_h2d(A, B, -16, None) == 1
    assert lib.lmho_copy_h2d(A, B, 24, None) == 1                 # not whole 16-byte words
    assert lib.lmho_copy_h2d(A + 8, B, 64, None) == 1             # dst not 16-byte aligned
    assert lib.lmho_copy_h2d(A, B + 4, 64, None) == 1             # src not 16-byte aligned
    assert lib.lmho_copy_h2d(A, A + 32, 64, None) == 2            # overlapping ranges
