"""Pins of the embedding-gather and greedy-head oracle (oracle/head.py) against hand-built
blocks with closed-form weights, the independent numpy decoder, constructed logits with a
known maximum, ties, and brute force on tiny shapes."""
import numpy as np
import pytest

import oracle
from oracle import head, oracle_np
from gguf_weight_only_gb300 import synth


def q4k_block(d, dmin, scale12, qs):
    b = np.zeros(144, np.uint8)
    b[0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    b[2:4] = np.frombuffer(np.float16(dmin).tobytes(), np.uint8)
    b[4:16] = scale12
    b[16:144] = qs
    return b


def test_embed_hand_built_rows():
    # row 0: sc = 1, m = 2, d = 1, dmin = 0.5, qs = 0x21 -> 0 (low nibbles) / 1 (high nibbles)
    # row 1: the same with d = 2 -> 2 q - 1: 1 (low) / 3 (high)
    r0 = q4k_block(1.0, 0.5, [1, 1, 1, 1, 2, 2, 2, 2, 0x21, 0x21, 0x21, 0x21], 0x21)
    r1 = q4k_block(2.0, 0.5, [1, 1, 1, 1, 2, 2, 2, 2, 0x21, 0x21, 0x21, 0x21], 0x21)
    W = np.concatenate([r0, r1])
    e = head.embed_rows(12, W, 2, 256, [1, 0, 1])
    lo_hi = lambda a, b: np.tile(np.r_[np.full(32, a), np.full(32, b)], 4)
    np.testing.assert_array_equal(e[0], lo_hi(1.0, 3.0))
    np.testing.assert_array_equal(e[1], lo_hi(0.0, 1.0))
    np.testing.assert_array_equal(e[2], e[0])


@pytest.mark.parametrize("t", (12, 13, 14, 23))
def test_embed_matches_numpy_decoder(t):
    N, K = 37, 512
    W = synth.weights(t, N, K, [800, t])
    ids = np.array([0, 36, 5, 5, 17])
    e = head.embed_rows(t, W, N, K, ids)
    ref = oracle_np.dequant(t, W, N, K)[ids]
    np.testing.assert_array_equal(e, ref)


def test_embed_rejects_out_of_range_ids():
    W = synth.weights(12, 4, 256, [801])
    for bad in ([4], [-1]):
        with pytest.raises(ValueError):
            head.embed_rows(12, W, 4, 256, bad)


def test_argmax_of_a_planted_row():
    # every row is zero (all bytes 0: d = dmin = 0) except row 6, whose weights are all 1:
    # sc = m = 2 in every sub-block, d = 1, dmin = 0.5, qs = 0x11 (q = 1): w = 2*1 - 0.5*2 = 1
    N, K = 9, 256
    W = np.zeros((N, 144), np.uint8)
    W[6] = q4k_block(1.0, 0.5, [2, 2, 2, 2, 2, 2, 2, 2, 0x22, 0x22, 0x22, 0x22], 0x11)
    x = np.ones((2, K), np.float16)
    x[1] *= -1
    idx, val = head.argmax(12, W.reshape(-1), N, K, x)
    assert idx[0] == 6 and val[0] == 256.0          # sum of 256 ones
    assert idx[1] == 0 and val[1] == 0.0            # row 6 gives -256; the first of the zero rows wins


def test_argmax_ties_pick_the_first_row():
    N, K = 5, 256
    blk = q4k_block(1.0, 0.5, [2, 2, 2, 2, 2, 2, 2, 2, 0x22, 0x22, 0x22, 0x22], 0x11)
    W = np.stack([np.zeros(144, np.uint8), blk, np.zeros(144, np.uint8), blk, blk])
    idx, val = head.argmax(12, W.reshape(-1), N, K, np.ones((1, K), np.float16))
    assert idx[0] == 1 and val[0] == 256.0


def test_argmax_nan_ranks_first_and_signed_zeros_tie():
    # numpy's reading of argmax: a NaN ranks above every number (the first NaN wins), and
    # -0 == +0 (the first zero wins). Row 6 as in the planted test (all weights 1, y = 256);
    # row 2 has d = NaN, so y[2] is NaN; with x = -1 row 6 gives -256 and the zero rows tie.
    N, K = 9, 256
    W = np.zeros((N, 144), np.uint8)
    W[6] = q4k_block(1.0, 0.5, [2, 2, 2, 2, 2, 2, 2, 2, 0x22, 0x22, 0x22, 0x22], 0x11)
    W[2] = q4k_block(np.nan, 0.5, [2, 2, 2, 2, 2, 2, 2, 2, 0x22, 0x22, 0x22, 0x22], 0x11)
    idx, val = head.argmax(12, W.reshape(-1), N, K, np.ones((1, K), np.float16))
    assert idx[0] == 2 and np.isnan(val[0])
    W[2] = 0
    W[0] = q4k_block(-0.0, 0.0, [2, 2, 2, 2, 2, 2, 2, 2, 0x22, 0x22, 0x22, 0x22], 0x11)   # weights -0
    idx, val = head.argmax(12, W.reshape(-1), N, K, -np.ones((1, K), np.float16))
    assert idx[0] == 0 and val[0] == 0.0


@pytest.mark.parametrize("t", (12, 13, 14, 23))
def test_argmax_brute_force_tiny(t):
    N, K, M = 8, 512, 3
    W = synth.weights(t, N, K, [802, t])
    x = synth.activations(M, K, [803, t])
    dense = x.astype(np.float64) @ oracle_np.dequant(t, W, N, K).T
    idx, val = head.argmax(t, W, N, K, x)
    np.testing.assert_array_equal(idx, np.argmax(dense, axis=1))
    np.testing.assert_allclose(val, dense.max(axis=1), rtol=1e-12, atol=0)
