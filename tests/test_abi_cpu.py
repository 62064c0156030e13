"""Host-side checks of the C-ABI library (no GPU): it loads, exports every
symbol include/lmho.h declares, and rejects bad arguments before touching a
device."""
import ctypes
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
    assert lib.lmho_version() >= 100
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
