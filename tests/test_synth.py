"""The seeded input generator draws what the input recipe states: fp16 d / dmin uniform in
[2^-10, 2^-6], Q6_K int8 sub-block scales uniform in [-32, 31], every other byte uniform, x
= fp16(N(0, 1)), and the same seed gives the same bytes."""
import numpy as np
import pytest

from gguf_weight_only_gb300 import synth

SCALE_OFFSETS = {12: (0, 2), 13: (0, 2), 14: (208,), 23: (0,)}


def f16_at(b, off):
    return b[:, off:off + 2].copy().view(np.float16).reshape(-1).astype(np.float64)


@pytest.mark.parametrize("t", (12, 13, 14, 23))
def test_scales_in_range_and_spread(t):
    b = synth.blocks(t, 20000, [3, t])
    assert b.shape == (20000, synth.BLOCK_BYTES[t]) and b.dtype == np.uint8
    for off in SCALE_OFFSETS[t]:
        d = f16_at(b, off)
        assert d.min() >= 2.0 ** -10 and d.max() <= 2.0 ** -6
        # uniform on [2^-10, 2^-6]: mean (2^-10 + 2^-6) / 2, each quarter holds about a quarter
        assert abs(d.mean() - (2.0 ** -10 + 2.0 ** -6) / 2) < 2e-4
        q = np.histogram(d, bins=4, range=(2.0 ** -10, 2.0 ** -6))[0] / d.size
        assert np.all(np.abs(q - 0.25) < 0.02)


def test_q6k_scales_cover_minus_32_to_31_uniformly():
    b = synth.blocks(14, 20000, [4])
    sc = b[:, 192:208].copy().view(np.int8).reshape(-1).astype(np.int64)
    assert sc.min() == -32 and sc.max() == 31
    counts = np.bincount(sc + 32, minlength=64)
    assert counts.size == 64 and np.all(np.abs(counts / sc.size - 1 / 64) < 0.15 / 64)


@pytest.mark.parametrize("t", (12, 13, 14, 23))
def test_other_bytes_uniform(t):
    b = synth.blocks(t, 20000, [5, t])
    mask = np.ones(b.shape[1], bool)
    for off in SCALE_OFFSETS[t]:
        mask[off:off + 2] = False
    if t == 14:
        mask[192:208] = False
    v = b[:, mask].reshape(-1)
    counts = np.bincount(v, minlength=256)
    expected = v.size / 256
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 400          # 255 degrees of freedom: mean 255, sd about 23


def test_activations_standard_normal_fp16():
    x = synth.activations(64, 4096, [6])
    assert x.dtype == np.float16 and x.shape == (64, 4096)
    v = x.astype(np.float64)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01


def test_same_seed_same_bytes_and_row_layout():
    a = synth.weights(12, 3, 512, [7])
    assert np.array_equal(a, synth.weights(12, 3, 512, [7]))
    assert not np.array_equal(a, synth.weights(12, 3, 512, [8]))
    assert a.size == 3 * 2 * 144
    assert np.array_equal(a, synth.blocks(12, 6, [7]).reshape(-1))   # row n, superblock b at (2n + b) * 144
    with pytest.raises(ValueError):
        synth.weights(12, 3, 300, [7])
