"""Input generator: Philox4x32-10 known answers, slicing, determinism, moments."""
import numpy as np
import pytest

import gen


# Known-answer vectors published with Random123 (Salmon et al., SC'11) for
# Philox4x32 with 10 rounds: (counter, key) -> output.
KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", KAT)
def test_philox_known_answers(ctr, key, want):
    assert tuple(int(v) for v in gen.philox4x32_10(ctr, key)) == want


def test_slices_and_threads_agree():
    full = gen.normal_f32(0, 0, (300, 257))
    flat = full.reshape(-1)
    for off in (0, 1, 2, 255, 256, 257, 4097):
        part = gen.normal_f32(0, 0, (1031,), offset=off, threads=1)
        assert np.array_equal(part, flat[off:off + 1031])
    assert np.array_equal(full, gen.normal_f32(0, 0, (300, 257), threads=3))
    t_full = gen.targets(0, 1, (999,), 131072)
    assert np.array_equal(t_full[37:80], gen.targets(0, 1, (43,), 131072, offset=37))


def test_streams_and_seeds_differ():
    a = gen.normal_f32(0, 0, (4096,))
    assert not np.array_equal(a, gen.normal_f32(0, 2, (4096,)))
    assert not np.array_equal(a, gen.normal_f32(1, 0, (4096,)))
    assert np.array_equal(a, gen.normal_f32(0, 0, (4096,)))


def test_normal_moments_and_rounding():
    n = 1 << 20
    d = gen.normal_f64(0, 0, (n,), sigma=2.0)
    assert abs(d.mean()) < 0.01 and abs(d.std() - 2.0) < 0.01
    f = gen.normal_f32(0, 0, (n,), sigma=2.0)
    assert np.array_equal(f, d.astype(np.float32))           # RNE fp64 -> fp32
    b = gen.normal_bf16_bits(0, 0, (n,), sigma=2.0)
    w = gen.bf16_bits_to_f32(b)
    # bf16 keeps 8 significant bits: |w - f| <= half an ulp of bf16
    ulp = np.exp2(np.floor(np.log2(np.abs(f))) - 7)
    assert np.all(np.abs(w - f) <= ulp / 2 + 0.0)


def test_targets_range_and_uniformity():
    for V in (1, 2, 3, 4096, 128256, 131072):
        t = gen.targets(0, 1, (1 << 16,), V)
        assert t.min() >= 0 and t.max() < V
    t = gen.targets(0, 1, (1 << 20,), 16)
    counts = np.bincount(t, minlength=16)
    expected = (1 << 20) / 16
    chi2 = ((counts - expected) ** 2 / expected).sum()
    assert chi2 < 60  # 15 dof; p ~ 1e-7 at 60
