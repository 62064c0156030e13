"""The algorithmic byte model reproduces the floors the pages print (golden
fixture tests/golden/pages_floors.txt), which fixes what the roofline
numerators count."""
import os

import pytest

from lm_head_online_gb300 import roofline as rl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_floors.txt")


def load_floors():
    out = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        op, _, bw, us, _ = [c.strip() for c in line.split("|")]
        out[op] = (float(bw), float(us))
    return out


def test_floors_match_pages():
    f = load_floors()
    got = {
        "ce_flat": rl.floor_us(rl.ce_flat_bytes(16384, 4096), f["ce_flat"][0]),
        "flce": rl.floor_us(rl.flce_bytes(2 * 1024, 4096, 128256), f["flce"][0]),
        "ce_sbv": rl.floor_us(rl.ce_sbv_bytes(2048, 4, 4096), f["ce_sbv"][0]),
        "fljsd": rl.floor_us(rl.fljsd_bytes(1024, 4096, 128256), f["fljsd"][0]),
    }
    for op, (_, us) in f.items():
        assert got[op] == pytest.approx(us, abs=0.05), op   # pages print one decimal


def test_flop_model():
    assert rl.flce_flops(2048, 4096, 128256) == 2 * 2048 * 4096 * 128256
    assert rl.fljsd_flops(1024, 4096, 128256) == 2 * rl.fljsd_pass_flops(1024, 4096, 128256)
    assert rl.fljsd_pass_flops(1, 1, 1) == 4
