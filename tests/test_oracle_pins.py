"""Pins of the fp64 oracle against facts the pages and the mathematics fix (no GPU).

Every expected value here is either printed on the pages (golden fixtures, cited), a
hand-derived literal for a hand-built block (derivation in the comments), a closed form, an
invariant, or a library routine. None comes from the CUDA path.
"""
import os

import numpy as np
import pytest

import oracle
from oracle import oracle_np
from gguf_weight_only_gb300 import synth

TYPES = (12, 13, 14, 23)


def _read_rows(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def f16_bytes(v):
    return np.array([v], np.float16).view(np.uint8)


def dq_both(t, block):
    """Decode one block with both oracle decoders; they must agree bit for bit."""
    b = np.asarray(block, np.uint8).reshape(1, -1)
    c = oracle.dequant(t, b.reshape(-1), 1, 256)[0]
    n = oracle_np.dequant_blocks(t, b)[0]
    np.testing.assert_array_equal(c.view(np.uint64), n.view(np.uint64))
    return c


# ---------------------------------------------------------------- golden fixtures

def test_block_sizes_match_pages(golden_dir):
    rows = _read_rows(os.path.join(golden_dir, "ggml_block_sizes.txt"))
    assert len(rows) == 4
    for tid, per_block, nbytes, name in rows:
        tid, per_block, nbytes = int(tid), int(per_block), int(nbytes)
        assert per_block == 256
        assert oracle.block_bytes(tid) == nbytes
        assert oracle_np.BLOCK_BYTES[tid] == nbytes
        assert synth.BLOCK_BYTES[tid] == nbytes and synth.TYPE_NAMES[tid] == name
    assert oracle.block_bytes(8) == -1


def test_iq4_codebook_and_nibble_order(golden_dir):
    """d = 1 and every 6-bit scale = 33 (ls - 32 = 1): each weight is the codebook entry,
    in the order [low nibbles of the 16 bytes, high nibbles] per group (page formula)."""
    kv = np.array([int(v) for v in _read_rows(os.path.join(golden_dir, "iq4_xs_codebook.txt"))[0]])
    assert kv.shape == (16,)
    rng = np.random.default_rng(7)
    blk = np.zeros(136, np.uint8)
    blk[0:2] = f16_bytes(1.0)
    # ls = 33 = 0b10_0001: low nibble 1 in every scales_l nibble, high bits 0b10 in every
    # 2-bit field of scales_h -> scales_l bytes 0x11, scales_h = 0xAAAA.
    blk[2:4] = [0xAA, 0xAA]
    blk[4:8] = 0x11
    qs = rng.integers(0, 256, 128, dtype=np.uint8)
    blk[8:136] = qs
    w = dq_both(23, blk)
    expect = np.concatenate([kv[np.concatenate([g & 15, g >> 4])] for g in qs.reshape(8, 16)])
    np.testing.assert_array_equal(w, expect.astype(np.float64))


# ---------------------------------------------------------------- hand-built K-quant blocks

def q4k_block(d, dmin, scale12, qs):
    b = np.zeros(144, np.uint8)
    b[0:2], b[2:4] = f16_bytes(d), f16_bytes(dmin)
    b[4:16] = scale12
    b[16:144] = qs
    return b


def test_q4k_uniform_closed_form():
    # sc = 1 and m = 2 in every sub-block: bytes 0..3 = 1, bytes 4..7 = 2 (top bits 0),
    # bytes 8..11 = 0x21 (low nibble sc[4..7] = 1, high nibble m[4..7] = 2).
    # qs = 0x21: low nibble 1, high nibble 2.  w = 1*1*q - 0.5*2 -> 0 (low) or 1 (high).
    b = q4k_block(1.0, 0.5, [1, 1, 1, 1, 2, 2, 2, 2, 0x21, 0x21, 0x21, 0x21], 0x21)
    w = dq_both(12, b)
    expect = np.tile(np.r_[np.zeros(32), np.ones(32)], 4)
    np.testing.assert_array_equal(w, expect)


def test_q4k_scale_field_all_bit_positions():
    # sc = [5, 6, 7, 8, 63, 47, 31, 16], m = [9, 10, 11, 12, 48, 33, 17, 1].
    # bytes 0..3  = sc[0..3] | (sc[4..7] >> 4) << 6 = C5 86 47 48
    # bytes 4..7  = m[0..3]  | (m[4..7]  >> 4) << 6 = C9 8A 4B 0C
    # bytes 8..11 = (sc[4..7] & 15) | (m[4..7] & 15) << 4 = 0F 1F 1F 10
    # d = 1, dmin = 0.25, qs = 0x10: even sub-blocks (low nibbles) q = 0 -> -m/4,
    # odd sub-blocks (high nibbles) q = 1 -> sc - m/4.
    S = [0xC5, 0x86, 0x47, 0x48, 0xC9, 0x8A, 0x4B, 0x0C, 0x0F, 0x1F, 0x1F, 0x10]
    w = dq_both(12, q4k_block(1.0, 0.25, S, 0x10))
    per_sub = [-2.25, 3.5, -2.75, 5.0, -12.0, 38.75, -4.25, 15.75]
    np.testing.assert_array_equal(w, np.repeat(per_sub, 32))


@pytest.mark.parametrize("pos,nib,index", [
    (0, "lo", 0), (0, "hi", 32), (31, "lo", 31), (31, "hi", 63), (32, "lo", 64),
    (33, "hi", 97), (100, "lo", 196), (100, "hi", 228), (127, "hi", 255)])
def test_q4k_nibble_position(pos, nib, index):
    # sc = 1, m = 0 everywhere (bytes 0..3 = 1, 4..7 = 0, 8..11 = 0x01), d = 1, dmin = 0.
    # Only qs[pos] is nonzero (15 in one nibble): exactly weight `index` is 15.
    qs = np.zeros(128, np.uint8)
    qs[pos] = 0x0F if nib == "lo" else 0xF0
    w = dq_both(12, q4k_block(1.0, 0.0, [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1], qs))
    expect = np.zeros(256)
    expect[index] = 15.0
    np.testing.assert_array_equal(w, expect)


def test_q5k_without_high_bits_is_q4k():
    """'Q4_K is Q5_K without the high-bit array' (commit log of explicit-dev): a Q5_K block
    with qh = 0 decodes like the Q4_K block with the same d, dmin, scales and qs."""
    rng = np.random.default_rng(3)
    for _ in range(20):
        q4 = synth.blocks(12, 1, rng.integers(1 << 30))[0]
        q5 = np.concatenate([q4[:16], np.zeros(32, np.uint8), q4[16:]])
        np.testing.assert_array_equal(dq_both(13, q5), dq_both(12, q4))


@pytest.mark.parametrize("byte,bit,index", [(5, 2, 69), (31, 7, 255), (0, 0, 0), (17, 4, 145)])
def test_q5k_high_bit_position(byte, bit, index):
    # d = 1, dmin = 0, sc = 1, qs = 0: only bit `bit` of qh[byte] set -> weight 32*bit + byte = 16.
    b = np.zeros(176, np.uint8)
    b[0:2] = f16_bytes(1.0)
    b[4:16] = [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1]
    b[16 + byte] = 1 << bit
    expect = np.zeros(256)
    expect[index] = 16.0
    np.testing.assert_array_equal(dq_both(13, b), expect)


# ---------------------------------------------------------------- hand-built Q6_K blocks

def q6k_block(ql, qh, sc, d):
    b = np.zeros(210, np.uint8)
    b[0:128], b[128:192] = ql, qh
    b[192:208] = np.asarray(sc, np.int8).view(np.uint8)
    b[208:210] = f16_bytes(d)
    return b


def test_q6k_zero_quants_give_minus_32_scale():
    sc = np.arange(1, 17)
    w = dq_both(14, q6k_block(0, 0, sc, 0.5))
    np.testing.assert_array_equal(w, -16.0 * np.repeat(sc, 16))


def test_q6k_quarter_pattern():
    # ql = 0x21, qh = 0b11_10_01_00: quarter t takes low nibble (t < 2) or high nibble, and
    # bits 2t..2t+1 of qh: q = [1, 1+16, 2+32, 2+48] -> q - 32 = [-31, -15, 2, 18].
    w = dq_both(14, q6k_block(0x21, 0xE4, np.ones(16), 1.0))
    np.testing.assert_array_equal(w, np.tile(np.repeat([-31.0, -15.0, 2.0, 18.0], 32), 2))


def test_q6k_negative_scales():
    sc = np.array([-128, -32, -1, 127] * 4)
    w = dq_both(14, q6k_block(0x21, 0xE4, sc, 2.0 ** -6))
    q = np.tile(np.repeat([-31.0, -15.0, 2.0, 18.0], 32), 2)
    np.testing.assert_array_equal(w, 2.0 ** -6 * np.repeat(sc, 16) * q)


@pytest.mark.parametrize("field,pos,val,index,value", [
    ("ql", 40, 0x01, 40, -31.0), ("ql", 70, 0x10, 198, -31.0), ("ql", 5, 0x10, 69, -31.0),
    ("ql", 127, 0x01, 191, -31.0), ("qh", 33, 0x30, 193, 16.0), ("qh", 0, 0x03, 0, 16.0),
    ("qh", 63, 0xC0, 255, 16.0)])
def test_q6k_single_positions(field, pos, val, index, value):
    # sc = 1, d = 1, everything else zero (w = -32) except one field byte.
    ql, qh = np.zeros(128, np.uint8), np.zeros(64, np.uint8)
    (ql if field == "ql" else qh)[pos] = val
    expect = np.full(256, -32.0)
    expect[index] = value
    np.testing.assert_array_equal(dq_both(14, q6k_block(ql, qh, np.ones(16), 1.0)), expect)


def test_iq4_scale_fields():
    # ls = [0, 1, 31, 32, 33, 47, 62, 63]; scales_l nibbles ls & 15 = [0,1,15,0,1,15,14,15]
    # -> bytes 0x10 0x0F 0xF1 0xFE; scales_h 2-bit fields ls >> 4 = [0,0,1,2,2,2,3,3] -> 0xFA90.
    # qs = 0x88 selects codebook entry 8 (= 1), d = 1: w = ls - 32 per sub-block.
    b = np.zeros(136, np.uint8)
    b[0:2] = f16_bytes(1.0)
    b[2:4] = [0x90, 0xFA]
    b[4:8] = [0x10, 0x0F, 0xF1, 0xFE]
    b[8:] = 0x88
    np.testing.assert_array_equal(dq_both(23, b), np.repeat([-32.0, -31, -1, 0, 1, 15, 30, 31], 32))


# ---------------------------------------------------------------- fp16 and the contraction

def test_half_decoder_matches_numpy_float16():
    bits = np.arange(1 << 16, dtype=np.uint32)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits[::7]])
    r = ref[::7]
    nan = np.isnan(r)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], r[~nan])
    for b in (0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0x7C00, 0xFC00, 0xC000):
        assert oracle.half_to_double(b) == float(np.uint16(b).view(np.float16))


@pytest.mark.parametrize("t", TYPES)
def test_decoders_agree_on_random_blocks(t):
    blk = synth.blocks(t, 64, [99, t])
    c = oracle.dequant(t, blk.reshape(-1), 64, 256)
    n = oracle_np.dequant_blocks(t, blk)
    np.testing.assert_array_equal(c.view(np.uint64), n.view(np.uint64))


@pytest.mark.parametrize("t", TYPES)
def test_brute_force_tiny(t):
    """Tiny shapes: the C oracle's y against a pure-Python triple loop over the numpy
    decoder's weights (dense fp64 matmul written out)."""
    for (N, K, M) in ((3, 256, 2), (5, 512, 3), (1, 256, 1)):
        W = synth.weights(t, N, K, [5, t, N, K])
        x = synth.activations(M, K, [6, t, M])
        w = oracle_np.dequant(t, W, N, K)
        xd = x.astype(np.float64)
        ref = np.zeros((M, N))
        for m in range(M):
            for n in range(N):
                s = 0.0
                for k in range(K):
                    s += xd[m, k] * w[n, k]
                ref[m, n] = s
        got = oracle.qlinear(t, W, N, K, x, n_threads=2)
        np.testing.assert_array_equal(got, ref)          # same order of summation in fp64
        np.testing.assert_allclose(oracle_np.qlinear_f64(t, W, N, K, x), ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("t", TYPES)
def test_unit_activation_selects_a_column(t):
    N, K = 9, 512
    W = synth.weights(t, N, K, [11, t])
    w = oracle.dequant(t, W, N, K)
    for k in (0, 1, 255, 256, 300, 511):
        x = np.zeros((1, K), np.float16)
        x[0, k] = 1.0
        np.testing.assert_array_equal(oracle.qlinear(t, W, N, K, x)[0], w[:, k])


@pytest.mark.parametrize("t", TYPES)
def test_linearity_and_exact_scaling(t):
    N, K, M = 7, 768, 3
    W = synth.weights(t, N, K, [12, t])
    x = synth.activations(M, K, [13, t])
    y = oracle.qlinear(t, W, N, K, x)
    np.testing.assert_array_equal(oracle.qlinear(t, W, N, K, (2 * x.astype(np.float32)).astype(np.float16)), 2 * y)
    # doubling every fp16 super-scale (exact: all are <= 2^-6) doubles every weight
    bb = synth.BLOCK_BYTES[t]
    blk = W.reshape(-1, bb).copy()
    offs = {12: (0, 2), 13: (0, 2), 14: (208,), 23: (0,)}[t]
    for o in offs:
        d = blk[:, o:o + 2].copy().view(np.float16) * np.float16(2)
        blk[:, o:o + 2] = d.view(np.uint8)
    np.testing.assert_array_equal(oracle.qlinear(t, blk.reshape(-1), N, K, x), 2 * y)


@pytest.mark.parametrize("t", (12, 13))
def test_zero_quants_leave_only_the_min_term(t):
    """All-zero qs (and qh): every weight of sub-block j is the same non-positive constant
    -dmin*m_j, so y = sum_j c_j * (sum of x over sub-block j)."""
    N, K = 4, 512
    blk = synth.blocks(t, N * K // 256, [14, t])
    if t == 12:
        blk[:, 16:] = 0
    else:
        blk[:, 16:] = 0
    W = blk.reshape(-1)
    w = oracle.dequant(t, W, N, K).reshape(N, -1, 32)
    assert np.all(w <= 0)
    assert np.all(w == w[:, :, :1])                      # constant within each sub-block
    x = synth.activations(2, K, [15, t])
    sx = x.astype(np.float64).reshape(2, -1, 32).sum(-1)
    np.testing.assert_allclose(oracle.qlinear(t, W, N, K, x), sx @ w[:, :, 0].T, rtol=1e-12, atol=1e-12)


def test_thread_count_does_not_change_bits():
    W = synth.weights(12, 37, 1024, [16])
    x = synth.activations(3, 1024, [17])
    a = oracle.qlinear(12, W, 37, 1024, x, n_threads=1)
    b = oracle.qlinear(12, W, 37, 1024, x, n_threads=8)
    np.testing.assert_array_equal(a.view(np.uint64), b.view(np.uint64))


def test_packed_scale_field_is_a_bijection():
    """Round trip of the 12-byte field: every 16 x 6-bit assignment packs to 12 bytes that
    decode back to it (the field has exactly 96 bits, so uniform bytes = uniform values)."""
    hypothesis = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    def pack(sc, m):
        S = np.zeros(12, np.uint8)
        for j in range(4):
            S[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
            S[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
            S[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
        return S

    @hypothesis.settings(max_examples=200, deadline=None)
    @hypothesis.given(st.lists(st.integers(0, 63), min_size=16, max_size=16))
    def check(vals):
        sc, m = vals[:8], vals[8:]
        # d = 1, dmin = 1, qs: low nibble 1 / high nibble 0 -> even sub-blocks sc - m, odd -m
        w = dq_both(12, q4k_block(1.0, 1.0, pack(sc, m), 0x01))
        per = w.reshape(8, 32)[:, 0]
        expect = [sc[j] - m[j] if j % 2 == 0 else -m[j] for j in range(8)]
        np.testing.assert_array_equal(per, expect)

    check()


def test_iq4_scale_field_is_a_bijection():
    """Round trip of IQ4_XS's scale field: every assignment of eight 6-bit ls values packs into
    scales_h (2 bytes: the high two bits of ls_j at bits 2j, 2j+1) and scales_l (4 bytes: the
    low nibble of ls_j in nibble j) and decodes back to d (ls_j - 32) on every weight of
    sub-block j. The field is exactly 48 bits, so every byte pattern is some assignment."""
    hypothesis = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    def pack(ls):
        h = 0
        low = np.zeros(4, np.uint8)
        for j, v in enumerate(ls):
            h |= (v >> 4) << (2 * j)
            low[j // 2] |= (v & 15) << (4 * (j % 2))
        return np.array([h & 0xFF, h >> 8], np.uint8), low

    @hypothesis.settings(max_examples=300, deadline=None)
    @hypothesis.given(st.lists(st.integers(0, 63), min_size=8, max_size=8), st.sampled_from([0.5, 1.0, 2.0]))
    def check(ls, d):
        sh, sl = pack(ls)
        b = np.zeros(136, np.uint8)
        b[0:2] = f16_bytes(d)
        b[2:4] = sh
        b[4:8] = sl
        b[8:] = 0x88   # codebook entry 8 (= 1) in every nibble
        np.testing.assert_array_equal(dq_both(23, b), np.repeat([d * (v - 32) for v in ls], 32))

    check()


def test_tolerance_is_positive_and_scales():
    W = synth.weights(23, 5, 512, [18])
    x = synth.activations(2, 512, [19])
    tol = oracle.tolerance(23, W, 5, 512, x)
    assert tol.shape == (2, 5) and np.all(tol > 0)
    np.testing.assert_allclose(oracle.tolerance(23, W, 5, 512, (2 * x.astype(np.float32)).astype(np.float16)), 2 * tol)


def test_tolerance_hand_computed():
    """The bound is 2e-3 * sum_k |x_k w_k| per element, not 2e-3 * |sum_k x_k w_k|. Two rows:
    row 0 has every weight 1 (d = 1, dmin = 0, sc = 1, m = 0, every nibble 1); row 1 every
    weight 0 (d = 0). With x alternating +1, -1 over K = 256: y[0] = 0 but the bound is
    2e-3 * 256 = 0.512; row 1 gets bound 0; doubling x doubles the bound; tolerance_rows
    of row 0 alone equals column 0."""
    ones = q4k_block(1.0, 0.0, [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1], 0x11)
    zeros = q4k_block(0.0, 0.0, [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1], 0x11)
    np.testing.assert_array_equal(dq_both(12, ones), np.ones(256))
    W = np.concatenate([ones, zeros])
    x = np.tile(np.array([1.0, -1.0], np.float16), 128).reshape(1, 256)
    assert oracle.qlinear(12, W, 2, 256, x)[0, 0] == 0.0
    tol = oracle.tolerance(12, W, 2, 256, x)
    np.testing.assert_allclose(tol, [[0.512, 0.0]], rtol=1e-15, atol=0)
    np.testing.assert_allclose(oracle.tolerance(12, W, 2, 256, (2 * x).astype(np.float16)), [[1.024, 0.0]], rtol=1e-15)
    np.testing.assert_array_equal(oracle.tolerance_rows(12, W, 2, 256, x, [0]), tol[:, :1])


@pytest.mark.parametrize("t", TYPES)
def test_row_sampled_oracle_matches_the_dense_product(t):
    """qlinear_rows (the sampled check at full sizes) picks row r's bytes at r * K/256 * BB:
    unsorted and repeated rows against the independent numpy decoder's dense product."""
    N, K, M = 11, 768, 2
    W = synth.weights(t, N, K, [20, t])
    x = synth.activations(M, K, [21, t])
    rows = [10, 0, 3, 3, 7]
    dense = x.astype(np.float64) @ oracle_np.dequant(t, W, N, K)[rows].T
    np.testing.assert_allclose(oracle.qlinear_rows(t, W, N, K, x, rows), dense, rtol=1e-12, atol=1e-12)


def test_bad_arguments_are_rejected():
    with pytest.raises(ValueError):
        oracle.qlinear(12, np.zeros(144, np.uint8), 1, 100, np.zeros((1, 100), np.float16))
    with pytest.raises(ValueError):
        oracle.dequant(7, np.zeros(144, np.uint8), 1, 256)
