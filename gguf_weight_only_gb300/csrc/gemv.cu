// gemv.cu -- decode-path quantized linear y[M<=8, N] = x[M, K] . dequant(W)[N, K]^T.
//
// Design (sm_103a):
//  * One CTA per 16 weight rows (one MMA row tile). Its warps split K: warp w owns a
//    contiguous range of superblocks and streams them through its own ring of shared-memory
//    stages. Each stage holds one superblock of all 16 rows plus the matching 256 columns of
//    x for every token; it is filled by bulk copies (the TMA engine, cp.async.bulk) that
//    complete on the stage's mbarrier, so HBM bytes in flight cost no registers.
//  * Every weight byte is read from HBM exactly once. Each lane decodes its share of the
//    block in registers into fp16 pairs that are EXACT small integers (sc*q for K-quants,
//    sc*(q-32) for Q6_K, (ls-32)*codebook[q] for IQ4_XS), feeds them to the legacy tensor
//    core (mma.sync m16n8k16, fp32 accumulate) with the tokens on the MMA's n = 8 side, and
//    applies the fp32 superblock scale d (and dmin for K-quants) to the per-superblock
//    fp32 partial sums. The K-quant min term dmin * sum_j m_j * sum(x over sub-block j) runs
//    through a second MMA whose A operand is the (constant per sub-block) 6-bit min.
//  * Warps' partial tiles are reduced in fixed order through shared memory (deterministic,
//    no atomics).
// MMA fragment ownership (m16n8k16): lane = 4*g + c holds rows g and g+8 of A and k-slots
// {2c, 2c+1, 2c+8, 2c+9}. The contraction does not care which real k sits in which slot, so
// each lane assigns the k's it decoded to its own slots and loads x for exactly those k's.
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace ql {

template <int TYPE>
struct GemvFmt;
template <>
struct GemvFmt<12> {   // Q4_K
    static constexpr int BB = 144;
};
template <>
struct GemvFmt<13> {   // Q5_K
    static constexpr int BB = 176;
};
template <>
struct GemvFmt<14> {   // Q6_K
    static constexpr int BB = 210;
};
template <>
struct GemvFmt<23> {   // IQ4_XS
    static constexpr int BB = 136;
};

// x segment layout inside a stage: token t, 64-column segment s at t*kXTok + s*kXSeg.
// 16 bytes of padding per 128-byte segment spread the four lanes of a row group (which read
// segments c = 0..3) over distinct banks.
constexpr uint32_t kXSeg = 144;
constexpr uint32_t kXTok = 4 * kXSeg;

// ---------------------------------------------------------------- K-quant scale constants

struct KqConsts {
    uint32_t sc_lo, n1024_lo;   // (sc, sc), (-1024 sc, ...)      sub-block 2c   (low nibbles)
    uint32_t sc16_hi, n64_hi;   // (sc/16, ...), (-64 sc, ...)     sub-block 2c+1 (high nibbles)
    uint32_t m_lo, m_hi;        // (m, m) for the two sub-blocks
};

// Scales/mins of sub-blocks 2c and 2c+1 from the 12-byte field (header words y, z, w).
__device__ __forceinline__ KqConsts kq_consts(uint4 h, int c) {
    const uint32_t A = h.y, B = h.z, C = h.w;
    const uint32_t sc_lo4 = A & 0x3F3F3F3Fu;
    const uint32_t m_lo4 = B & 0x3F3F3F3Fu;
    const uint32_t sc_hi4 = and_or(C, 0x0F0F0F0Fu, (A >> 2) & 0x30303030u);
    const uint32_t m_hi4 = and_or(C >> 4, 0x0F0F0F0Fu, (B >> 2) & 0x30303030u);
    const uint32_t sel = (2u * c) | ((2u * c + 1u) << 4);
    const uint32_t vs = prmt(sc_lo4, sc_hi4, sel);   // byte0 = sc[2c], byte1 = sc[2c+1]
    const uint32_t vm = prmt(m_lo4, m_hi4, sel);
    KqConsts k;
    const uint32_t sc0 = hsub2(prmt(vs, 0x64646464u, 0x4040u), kH2_1024);
    const uint32_t sc1 = hsub2(prmt(vs, 0x64646464u, 0x4141u), kH2_1024);
    k.sc_lo = sc0;
    k.n1024_lo = hmul2(sc0, kH2_m1024);
    k.sc16_hi = hmul2(sc1, kH2_1_16);
    k.n64_hi = hmul2(sc1, kH2_m64);
    k.m_lo = hsub2(prmt(vm, 0x64646464u, 0x4040u), kH2_1024);
    k.m_hi = hsub2(prmt(vm, 0x64646464u, 0x4141u), kH2_1024);
    return k;
}

// One qs word of a K-quant row -> the four A pairs (exact sc*q in fp16).
// w holds qs bytes [b0 b1 b2 b3] = positions l..l+3 of a 32-byte group: low nibbles are
// weights l..l+3 of sub-block 2c, high nibbles weights l..l+3 of sub-block 2c+1.
// qh (Q5_K only) holds qh[l..l+3]; bit 2c / 2c+1 of each byte is the fifth bit.
template <bool Q5>
__device__ __forceinline__ void kq_word(uint32_t w, uint32_t qh, int c, const KqConsts &k, uint32_t &lo01,
                                        uint32_t &lo23, uint32_t &hi01, uint32_t &hi23) {
    const uint32_t w2 = prmt(w, 0u, 0x3120u);   // [b0 b2 b1 b3]: half lanes hold b0|b1, then b2|b3
    const uint32_t w3 = w2 >> 8;
    uint32_t l01 = and_or(w2, 0x000F000Fu, kH2_1024);   // (1024 + q)
    uint32_t l23 = and_or(w3, 0x000F000Fu, kH2_1024);
    uint32_t h01 = and_or(w2, 0x00F000F0u, kH2_1024);   // (1024 + 16 q)
    uint32_t h23 = and_or(w3, 0x00F000F0u, kH2_1024);
    if constexpr (Q5) {
        const uint32_t q2 = prmt(qh, 0u, 0x3120u);
        const uint32_t q3 = q2 >> 8;
        const uint32_t rl = (4u - 2u * c) & 31u, rh = (7u - 2u * c) & 31u;
        l01 = or_and(l01, rotl(q2, rl), 0x00100010u);   // bit 2c   -> bit 4 (+16)
        l23 = or_and(l23, rotl(q3, rl), 0x00100010u);
        h01 = or_and(h01, rotl(q2, rh), 0x01000100u);   // bit 2c+1 -> bit 8 (+16 * 16)
        h23 = or_and(h23, rotl(q3, rh), 0x01000100u);
    }
    lo01 = hfma2(l01, k.sc_lo, k.n1024_lo);   // (1024+q)*sc - 1024 sc = q*sc (exact)
    lo23 = hfma2(l23, k.sc_lo, k.n1024_lo);
    hi01 = hfma2(h01, k.sc16_hi, k.n64_hi);   // (1024+16q)*sc/16 - 64 sc = q*sc (exact)
    hi23 = hfma2(h23, k.sc16_hi, k.n64_hi);
}

__device__ __forceinline__ uint32_t word_of(const uint4 &a, const uint4 &b, int u) {
    switch (u) {
    case 0: return a.x;
    case 1: return a.y;
    case 2: return a.z;
    case 3: return a.w;
    case 4: return b.x;
    case 5: return b.y;
    case 6: return b.z;
    default: return b.w;
    }
}
__device__ __forceinline__ uint32_t word4(const uint4 &a, int u) {
    return u == 0 ? a.x : u == 1 ? a.y : u == 2 ? a.z : a.w;
}

// ---------------------------------------------------------------- per-format superblock

// Q4_K / Q5_K: lane (g, c) decodes the 32-byte qs group c (64 weights: sub-blocks 2c, 2c+1)
// of rows g and g+8.
template <int TYPE>
__device__ __forceinline__ void superblock_kq(uint32_t blk_a, uint32_t blk_b, uint32_t xb, int c, float (&acc)[4]) {
    constexpr bool Q5 = (TYPE == 13);
    constexpr uint32_t QS = Q5 ? 48 : 16;
    const uint4 ha = lds128(blk_a), hb = lds128(blk_b);
    const KqConsts ka = kq_consts(ha, c), kb = kq_consts(hb, c);
    const uint4 qa0 = lds128(blk_a + QS + 32 * c), qa1 = lds128(blk_a + QS + 32 * c + 16);
    const uint4 qb0 = lds128(blk_b + QS + 32 * c), qb1 = lds128(blk_b + QS + 32 * c + 16);
    uint4 ha0 = make_uint4(0, 0, 0, 0), ha1 = ha0, hb0 = ha0, hb1 = ha0;
    if constexpr (Q5) {
        ha0 = lds128(blk_a + 16);
        ha1 = lds128(blk_a + 32);
        hb0 = lds128(blk_b + 16);
        hb1 = lds128(blk_b + 32);
    }
    float d1[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t xs = xb + c * kXSeg;   // segment c holds columns 64c .. 64c+63
#pragma unroll
    for (int u = 0; u < 8; u += 2) {
        const uint4 xl = lds128(xs + 8 * u);        // columns 64c + 4u .. +7   (low nibbles)
        const uint4 xh = lds128(xs + 64 + 8 * u);   // columns 64c + 32 + 4u .. (high nibbles)
#pragma unroll
        for (int v = 0; v < 2; ++v) {
            const int uu = u + v;
            uint32_t la01, la23, lh01, lh23, lb01, lb23, lbh01, lbh23;
            kq_word<Q5>(word_of(qa0, qa1, uu), word_of(ha0, ha1, uu), c, ka, la01, la23, lh01, lh23);
            kq_word<Q5>(word_of(qb0, qb1, uu), word_of(hb0, hb1, uu), c, kb, lb01, lb23, lbh01, lbh23);
            const uint32_t x0 = v ? xl.z : xl.x, x1 = v ? xl.w : xl.y;
            const uint32_t y0 = v ? xh.z : xh.x, y1 = v ? xh.w : xh.y;
            mma16816(d1, la01, lb01, la23, lb23, x0, x1);
            mma16816(d1, lh01, lbh01, lh23, lbh23, y0, y1);
            mma16816(d2, ka.m_lo, kb.m_lo, ka.m_lo, kb.m_lo, x0, x1);
            mma16816(d2, ka.m_hi, kb.m_hi, ka.m_hi, kb.m_hi, y0, y1);
        }
    }
    const float da = half_lo_to_float(ha.x), dma = half_hi_to_float(ha.x);
    const float db = half_lo_to_float(hb.x), dmb = half_hi_to_float(hb.x);
    acc[0] += da * d1[0] - dma * d2[0];
    acc[1] += da * d1[1] - dma * d2[1];
    acc[2] += db * d1[2] - dmb * d2[2];
    acc[3] += db * d1[3] - dmb * d2[3];
}

// 16 bytes at a 2-byte aligned shared address, read as aligned words and realigned.
__device__ __forceinline__ uint4 lds128_a2(uint32_t addr) {
    const uint32_t a = addr & ~3u;
    const uint32_t sel = (addr & 2u) ? 0x5432u : 0x3210u;
    const uint32_t w0 = lds32(a), w1 = lds32(a + 4), w2 = lds32(a + 8), w3 = lds32(a + 12), w4 = lds32(a + 16);
    return make_uint4(prmt(w0, w1, sel), prmt(w1, w2, sel), prmt(w2, w3, sel), prmt(w3, w4, sel));
}
__device__ __forceinline__ uint2 lds64_a2(uint32_t addr) {
    const uint32_t a = addr & ~3u;
    const uint32_t sel = (addr & 2u) ? 0x5432u : 0x3210u;
    const uint32_t w0 = lds32(a), w1 = lds32(a + 4), w2 = lds32(a + 8);
    return make_uint2(prmt(w0, w1, sel), prmt(w1, w2, sel));
}

// Q6_K: lane (g, c) takes half h = c/2 and positions l = 16*(c%2) .. +15 of that half, for
// all four quarters t (64 weights per row): ql bytes 64h+16e.. (t = 0 low / t = 2 high
// nibbles), 64h+32+16e.. (t = 1 / t = 3), qh bytes 128+32h+16e.. (bits 2t, 2t+1).
__device__ __forceinline__ void q6_row_consts(uint32_t blk, int h, int e, uint32_t (&sc)[4], float &d) {
    const uint2 s = lds64_a2(blk + 192 + 8 * h);        // int8 scales 8h .. 8h+7
    const uint32_t s0 = s.x ^ 0x80808080u, s1 = s.y ^ 0x80808080u;   // sc + 128 as unsigned bytes
    // lane needs scales 8h + e + 2t: bytes e, e+2 of s0 (t = 0, 1) and of s1 (t = 2, 3)
    const uint32_t sel0 = e ? 0x4141u : 0x4040u, sel1 = e ? 0x4343u : 0x4242u;
    const uint32_t kH2_1152 = 0x64806480u;
    sc[0] = hsub2(prmt(s0, 0x64646464u, sel0), kH2_1152);
    sc[1] = hsub2(prmt(s0, 0x64646464u, sel1), kH2_1152);
    sc[2] = hsub2(prmt(s1, 0x64646464u, sel0), kH2_1152);
    sc[3] = hsub2(prmt(s1, 0x64646464u, sel1), kH2_1152);
    d = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(blk + 208))));
}

// A pairs of quarter t for one word triple (ql word for t%2, qh word); returns (k0,k0+1)
// and (k0+2,k0+3) as exact sc*(q-32).
__device__ __forceinline__ void q6_pairs(uint32_t qlw, uint32_t qhw, int t, uint32_t sc, uint32_t &p01, uint32_t &p23) {
    const uint32_t l2 = prmt(qlw, 0u, 0x3120u);
    const uint32_t h2 = prmt(qhw, 0u, 0x3120u);
    const uint32_t l3 = l2 >> 8, h3 = h2 >> 8;
    uint32_t v01, v23;
    if (t < 2) {
        v01 = and_or(l2, 0x000F000Fu, kH2_1024);
        v23 = and_or(l3, 0x000F000Fu, kH2_1024);
    } else {
        v01 = and_or(l2 >> 4, 0x000F000Fu, kH2_1024);
        v23 = and_or(l3 >> 4, 0x000F000Fu, kH2_1024);
    }
    // bits 2t, 2t+1 of each qh byte -> bits 4, 5 of the half
    const int sh = 4 - 2 * t;
    const uint32_t b01 = sh >= 0 ? (h2 << sh) : (h2 >> -sh);
    const uint32_t b23 = sh >= 0 ? (h3 << sh) : (h3 >> -sh);
    v01 = or_and(v01, b01, 0x00300030u);
    v23 = or_and(v23, b23, 0x00300030u);
    p01 = hmul2(hsub2(v01, kH2_1056), sc);   // (q - 32) * sc
    p23 = hmul2(hsub2(v23, kH2_1056), sc);
}

__device__ __forceinline__ void superblock_q6(uint32_t blk_a, uint32_t blk_b, uint32_t xb, int c, float (&acc)[4]) {
    const int h = c >> 1, e = c & 1;
    uint32_t sca[4], scb[4];
    float da, db;
    q6_row_consts(blk_a, h, e, sca, da);
    q6_row_consts(blk_b, h, e, scb, db);
    const uint32_t offA = 64 * h + 16 * e, offB = 64 * h + 32 + 16 * e, offH = 128 + 32 * h + 16 * e;
    const uint4 qaA = lds128_a2(blk_a + offA), qaB = lds128_a2(blk_a + offB), qaH = lds128_a2(blk_a + offH);
    const uint4 qbA = lds128_a2(blk_b + offA), qbB = lds128_a2(blk_b + offB), qbH = lds128_a2(blk_b + offH);
    float d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        // columns 128h + 32t + 16e + 4u: segment 2h + t/2, offset 32(t%2) + 16e + 4u
        const uint32_t xs = xb + (2 * h + t / 2) * kXSeg + 2 * (32 * (t & 1) + 16 * e);
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
            const uint4 xv = lds128(xs + 8 * u);
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const int uu = u + v;
                uint32_t a01, a23, b01, b23;
                q6_pairs(word4((t & 1) ? qaB : qaA, uu), word4(qaH, uu), t, sca[t], a01, a23);
                q6_pairs(word4((t & 1) ? qbB : qbA, uu), word4(qbH, uu), t, scb[t], b01, b23);
                mma16816(d1, a01, b01, a23, b23, v ? xv.z : xv.x, v ? xv.w : xv.y);
            }
        }
    }
    acc[0] += da * d1[0];
    acc[1] += da * d1[1];
    acc[2] += db * d1[2];
    acc[3] += db * d1[3];
}

// IQ4_XS codebook (test/unit/test_llm_quant_cpu.py, test_unpack_lut_dot_uop) stored as
// unsigned bytes value + 128, four entries per register.
constexpr uint32_t kIq4T0 = 0x3F2D1801u;   //  -65  -83 -104 -127
constexpr uint32_t kIq4T1 = 0x766A5D4Fu;   //  -10  -22  -35  -49
constexpr uint32_t kIq4T2 = 0xA6998D81u;   //   38   25   13    1
constexpr uint32_t kIq4T3 = 0xF1D9C5B5u;   //  113   89   69   53

// Codebook lookup of the four nibbles of the low 16 bits of `s` (in nibble order) ->
// four bytes (value + 128).
__device__ __forceinline__ uint32_t iq4_lookup(uint32_t s) {
    const uint32_t s7 = s & 0x7777u;
    const uint32_t lo = prmt(kIq4T0, kIq4T1, s7);
    const uint32_t hi = prmt(kIq4T2, kIq4T3, s7);
    const uint32_t sel = ((s >> 1) & 0x4444u) | 0x3210u;   // bit 3 of each nibble picks `hi`
    return prmt(lo, hi, sel);
}

// IQ4_XS: lane (g, c) takes sub-blocks 2c and 2c+1 (qs bytes 32c .. 32c+31).
__device__ __forceinline__ void iq4_row_consts(uint32_t blk, int c, uint32_t (&ls)[2], uint32_t (&nb)[2], float &d) {
    const uint2 hd = lds64(blk);   // d | scales_h << 16, scales_l
    const uint32_t lsl = (hd.y >> (8 * c)) & 0xFFu;           // ls[2c] & 15 | (ls[2c+1] & 15) << 4
    const uint32_t lsh = (hd.x >> (16 + 4 * c)) & 0xFu;       // 2 high bits of each
    const uint32_t v0 = (lsl & 15u) | ((lsh & 3u) << 4);
    const uint32_t v1 = (lsl >> 4) | ((lsh >> 2) << 4);
    const uint32_t v = v0 | (v1 << 8);
    ls[0] = hsub2(prmt(v, 0x64646464u, 0x4040u), kH2_1056);   // ls - 32
    ls[1] = hsub2(prmt(v, 0x64646464u, 0x4141u), kH2_1056);
    nb[0] = hmul2(ls[0], kH2_m1152);
    nb[1] = hmul2(ls[1], kH2_m1152);
    d = half_lo_to_float(hd.x);
}

__device__ __forceinline__ void iq4_word(uint32_t w, uint32_t ls, uint32_t nb, uint32_t &lo01, uint32_t &lo23,
                                         uint32_t &hi01, uint32_t &hi23) {
    const uint32_t r01 = iq4_lookup(w);         // [b0.lo b0.hi b1.lo b1.hi] (+128)
    const uint32_t r23 = iq4_lookup(w >> 16);   // [b2.lo b2.hi b3.lo b3.hi]
    // (1024 + value + 128) * (ls - 32) - 1152 (ls - 32) = value * (ls - 32)
    lo01 = hfma2(prmt(r01, 0x64646464u, 0x4240u), ls, nb);
    hi01 = hfma2(prmt(r01, 0x64646464u, 0x4341u), ls, nb);
    lo23 = hfma2(prmt(r23, 0x64646464u, 0x4240u), ls, nb);
    hi23 = hfma2(prmt(r23, 0x64646464u, 0x4341u), ls, nb);
}

__device__ __forceinline__ void superblock_iq4(uint32_t blk_a, uint32_t blk_b, uint32_t xb, int c, float (&acc)[4]) {
    uint32_t lsa[2], nba[2], lsb[2], nbb[2];
    float da, db;
    iq4_row_consts(blk_a, c, lsa, nba, da);
    iq4_row_consts(blk_b, c, lsb, nbb, db);
    float d1[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t xs = xb + c * kXSeg;   // sub-blocks 2c, 2c+1 = columns 64c .. 64c+63
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t qoff = 8 + 32 * c + 16 * j;
        const uint2 a0 = lds64(blk_a + qoff), a1 = lds64(blk_a + qoff + 8);
        const uint2 b0 = lds64(blk_b + qoff), b1 = lds64(blk_b + qoff + 8);
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
            const uint4 xl = lds128(xs + 2 * (32 * j + 4 * u));        // columns 32j + 4u ..
            const uint4 xh = lds128(xs + 2 * (32 * j + 16 + 4 * u));   // columns 32j + 16 + 4u ..
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const int uu = u + v;
                const uint32_t wa = uu == 0 ? a0.x : uu == 1 ? a0.y : uu == 2 ? a1.x : a1.y;
                const uint32_t wb = uu == 0 ? b0.x : uu == 1 ? b0.y : uu == 2 ? b1.x : b1.y;
                uint32_t al01, al23, ah01, ah23, bl01, bl23, bh01, bh23;
                iq4_word(wa, lsa[j], nba[j], al01, al23, ah01, ah23);
                iq4_word(wb, lsb[j], nbb[j], bl01, bl23, bh01, bh23);
                mma16816(d1, al01, bl01, al23, bl23, v ? xl.z : xl.x, v ? xl.w : xl.y);
                mma16816(d1, ah01, bh01, ah23, bh23, v ? xh.z : xh.x, v ? xh.w : xh.y);
            }
        }
    }
    acc[0] += da * d1[0];
    acc[1] += da * d1[1];
    acc[2] += db * d1[2];
    acc[3] += db * d1[3];
}

// ---------------------------------------------------------------- the kernel

template <int TYPE>
__global__ void __launch_bounds__(512) gemv_kernel(const GemvArgs p) {
    constexpr int BB = GemvFmt<TYPE>::BB;
    extern __shared__ __align__(128) uint8_t smem[];
    const int nwarps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int row0 = blockIdx.x * 16;
    const int D = p.stages;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);               // [nwarps][D]
    float *red = reinterpret_cast<float *>(smem + p.red_offset);       // [nwarps][32][4]
    const uint32_t region = smem_u32(smem + p.region_offset) + warp * p.warp_bytes;
    const uint32_t bar0 = smem_u32(bars + warp * D);

    const int sb_begin = warp * p.sb_per_warp;
    const int sb_end = min(sb_begin + p.sb_per_warp, p.nsb);
    const int nmine = max(sb_end - sb_begin, 0);

    if (lane == 0) {
        for (int s = 0; s < D; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    const int64_t nsb = p.nsb;
    const int ncopy = 16 + 4 * p.M;

    // Fill stage buffer `s` with superblock `sb` of rows row0..row0+15 and x columns
    // 256 sb .. 256 sb + 255 of every token.
    auto issue = [&](int s, int sb) {
        const uint32_t st = region + s * p.stage_bytes;
        const uint32_t bar = bar0 + 8 * s;
        uint32_t my_bytes = 0;
        const uint8_t *src[2];
        uint32_t dst[2], nbytes[2];
        int tail_len = 0;
        uint32_t tail_dst = 0;
        const uint8_t *tail_src = nullptr;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int q = lane + 32 * r;
            nbytes[r] = 0;
            src[r] = nullptr;
            dst[r] = 0;
            if (q < 16) {
                const int row = row0 + q;
                if (row < p.N) {
                    const int64_t o = (static_cast<int64_t>(row) * nsb + sb) * BB;
                    const int64_t lo = o & ~int64_t(15);
                    int64_t hi = (o + BB + 15) & ~int64_t(15);
                    const int64_t t16 = p.total_bytes & ~int64_t(15);
                    if (hi > t16) {   // last block of a buffer whose size is not a multiple of 16
                        hi = t16;
                        tail_len = static_cast<int>(o + BB - t16);
                        tail_src = p.W + t16;
                        tail_dst = st + q * p.row_pitch + static_cast<uint32_t>(t16 - lo);
                    }
                    src[r] = p.W + lo;
                    dst[r] = st + q * p.row_pitch;
                    nbytes[r] = static_cast<uint32_t>(hi - lo);
                }
            } else if (q < ncopy) {
                const int t = (q - 16) >> 2, seg = (q - 16) & 3;
                src[r] = reinterpret_cast<const uint8_t *>(p.x + static_cast<int64_t>(t) * p.K + sb * 256 + seg * 64);
                dst[r] = st + 16 * p.row_pitch + t * kXTok + seg * kXSeg;
                nbytes[r] = 128;
            }
            my_bytes += nbytes[r];
        }
        const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, my_bytes);
        if (lane == 0) mbar_arrive_expect_tx(bar, total);
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 2; ++r)
            if (nbytes[r]) bulk_g2s(dst[r], src[r], nbytes[r], bar);
        if (tail_len > 0) {
            uint8_t *gdst = reinterpret_cast<uint8_t *>(smem) + (tail_dst - smem_u32(smem));
            for (int i = 0; i < tail_len; ++i) gdst[i] = __ldg(tail_src + i);
        }
    };

    for (int s = 0; s < D && s < nmine; ++s) issue(s, sb_begin + s);

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    bool ok = true;
    int it = 0;
    const int tok = min(g, p.M - 1);
    for (; it < nmine; ++it) {
        const int s = it % D;
        const uint32_t parity = (it / D) & 1;
        if (!mbar_wait(bar0 + 8 * s, parity)) {
            ok = false;
            break;
        }
        const int sb = sb_begin + it;
        const uint32_t st = region + s * p.stage_bytes;
        const int ra = min(row0 + g, p.N - 1), rb = min(row0 + g + 8, p.N - 1);
        const uint32_t offa = static_cast<uint32_t>(((static_cast<int64_t>(ra) * nsb + sb) * BB) & 15);
        const uint32_t offb = static_cast<uint32_t>(((static_cast<int64_t>(rb) * nsb + sb) * BB) & 15);
        const uint32_t blk_a = st + g * p.row_pitch + offa;
        const uint32_t blk_b = st + (g + 8) * p.row_pitch + offb;
        const uint32_t xb = st + 16 * p.row_pitch + tok * kXTok;
        if constexpr (TYPE == 12 || TYPE == 13) superblock_kq<TYPE>(blk_a, blk_b, xb, c, acc);
        else if constexpr (TYPE == 14) superblock_q6(blk_a, blk_b, xb, c, acc);
        else superblock_iq4(blk_a, blk_b, xb, c, acc);
        __syncwarp();
        if (it + D < nmine) {
            fence_proxy_async_smem();
            issue(s, sb_begin + it + D);
        }
    }
    if (!ok) {
        if (lane == 0) atomicOr(p.status, kStatusTimeout);
        // let copies still in flight land before the shared memory is released
        for (int j = it + 1; j < nmine && j < it + D; ++j) (void)mbar_wait(bar0 + 8 * (j % D), (j / D) & 1);
    }

    // fixed-order reduction of the warps' 16 x 8 tiles
#pragma unroll
    for (int i = 0; i < 4; ++i) red[(warp * 32 + lane) * 4 + i] = acc[i];
    __syncthreads();
    for (int t = threadIdx.x; t < 16 * p.M; t += blockDim.x) {
        const int row = t & 15, tk = t >> 4;
        const int src_lane = (row & 7) * 4 + (tk >> 1);
        const int slot = ((row >> 3) << 1) | (tk & 1);
        float s = 0.f;
        for (int w = 0; w < nwarps; ++w) s += red[(w * 32 + src_lane) * 4 + slot];
        if (row0 + row < p.N) p.y[static_cast<int64_t>(tk) * p.N + row0 + row] = s;
    }
}

// ---------------------------------------------------------------- host side

namespace {
template <int TYPE>
cudaError_t launch_t(const GemvArgs &a, int threads, size_t smem, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemv_kernel<TYPE>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int grid = (a.N + 15) / 16;
    gemv_kernel<TYPE><<<grid, threads, smem, stream>>>(a);
    return cudaGetLastError();
}
}  // namespace

int gemv_block_bytes(int type) {
    switch (type) {
    case 12: return 144;
    case 13: return 176;
    case 14: return 210;
    case 23: return 136;
    default: return -1;
    }
}

// Choose warps per CTA and pipeline depth: enough warps GPU-wide to cover HBM latency
// (about 16 per SM), no more warps than superblocks, and shared memory within budget.
GemvPlan gemv_plan(int type, int64_t N, int64_t K, int M, int num_sms) {
    GemvPlan pl{};
    const int bb = gemv_block_bytes(type);
    const int nsb = static_cast<int>(K / 256);
    const int tiles = static_cast<int>((N + 15) / 16);
    const uint32_t pitch_raw = static_cast<uint32_t>((bb + 15 + 15) & ~15);   // window incl. misalignment
    // odd multiple of 16 bytes -> row groups g, g+1 start on different bank quarters
    pl.row_pitch = ((pitch_raw / 16) % 2 == 1) ? pitch_raw : pitch_raw + 16;
    if (type == 12 || type == 13) pl.row_pitch = ((static_cast<uint32_t>(bb) / 16) % 2 == 1) ? bb : bb + 16;
    pl.stage_bytes = 16 * pl.row_pitch + M * kXTok;
    const int want_warps = 16 * num_sms;
    int w = 1;
    while (w < 16 && w * tiles < want_warps) w *= 2;
    while (w > 1 && w > nsb) w /= 2;
    int D = 4;
    auto smem_of = [&](int ww, int dd) {
        const size_t bars = ((static_cast<size_t>(ww) * dd * 8) + 127) & ~size_t(127);
        const size_t red = static_cast<size_t>(ww) * 32 * 4 * sizeof(float);
        return bars + red + static_cast<size_t>(ww) * dd * pl.stage_bytes;
    };
    const size_t budget = 200 * 1024;
    while (smem_of(w, D) > budget && D > 2) --D;
    while (smem_of(w, D) > budget && w > 1) w /= 2;
    pl.warps = w;
    pl.stages = D;
    pl.sb_per_warp = (nsb + w - 1) / w;
    pl.red_offset = static_cast<uint32_t>(((static_cast<size_t>(w) * D * 8) + 127) & ~size_t(127));
    pl.region_offset = pl.red_offset + static_cast<uint32_t>(w * 32 * 4 * sizeof(float));
    pl.warp_bytes = D * pl.stage_bytes;
    pl.smem = smem_of(w, D);
    pl.grid = tiles;
    return pl;
}

cudaError_t gemv_launch(int type, const uint8_t *W, const __half *x, float *y, int64_t N, int64_t K, int M,
                        unsigned *status, int num_sms, cudaStream_t stream) {
    const GemvPlan pl = gemv_plan(type, N, K, M, num_sms);
    GemvArgs a{};
    a.W = W;
    a.x = x;
    a.y = y;
    a.status = status;
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.M = M;
    a.nsb = static_cast<int>(K / 256);
    a.sb_per_warp = pl.sb_per_warp;
    a.stages = pl.stages;
    a.row_pitch = pl.row_pitch;
    a.stage_bytes = pl.stage_bytes;
    a.warp_bytes = pl.warp_bytes;
    a.red_offset = pl.red_offset;
    a.region_offset = pl.region_offset;
    a.total_bytes = N * (K / 256) * gemv_block_bytes(type);
    const int threads = 32 * pl.warps;
    switch (type) {
    case 12: return launch_t<12>(a, threads, pl.smem, stream);
    case 13: return launch_t<13>(a, threads, pl.smem, stream);
    case 14: return launch_t<14>(a, threads, pl.smem, stream);
    case 23: return launch_t<23>(a, threads, pl.smem, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ql
