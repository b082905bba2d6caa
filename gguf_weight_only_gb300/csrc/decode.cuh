// decode.cuh -- per-format superblock decoders shared by the decode kernels: ggml Q4_K / Q5_K /
// Q6_K / IQ4_XS blocks turned into exact fp16 integer products fed to mma.sync m16n8k16 with the
// tokens on the MMA's n side (x staged in shared memory, 128-byte swizzled rows).
//
// MMA fragment ownership (m16n8k16): lane = 4*g + c holds rows g and g+8 of A and k-slots
// {2c, 2c+1, 2c+8, 2c+9}. The contraction does not care which real k sits in which slot, so
// each lane assigns the k's it decoded to its own slots and reads x for exactly those k's.
// A 32-bit word of packed quants holds bytes b0..b3 of consecutive positions; masking it
// directly yields the half pairs (b0, b2) and (b1, b3), so x is staged with each group of
// four columns stored as [x0 x2 x1 x3] and one 8-byte read gives both B registers.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace ql {
namespace {

// ---------------------------------------------------------------- K-quant scale constants

struct KqConsts {
    uint32_t sc_lo, n1024_lo;   // (sc, sc), (-1024 sc, ...)      sub-block 2c   (low nibbles)
    uint32_t sc16_hi, n64_hi;   // (sc/16, ...), (-64 sc, ...)     sub-block 2c+1 (high nibbles)
    uint32_t m_lo, m_hi;        // (m, m) for the two sub-blocks
    uint32_t m_pair;            // (m[2c], m[2c+1])
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
    k.m_pair = hsub2(prmt(vm, 0x64646464u, 0x4140u), kH2_1024);
    return k;
}

// One qs word of a K-quant row -> the four A pairs (exact sc*q in fp16).
// w = qs bytes [b0 b1 b2 b3] at positions l..l+3 of 32-byte group c: low nibbles are weights
// of sub-block 2c, high nibbles of sub-block 2c+1. Masking w pairs the half lanes (b0, b2)
// and (b1, b3): with x stored permuted ([x0 x2 x1 x3] per group of four, PERM) that is used
// directly; otherwise w is first reordered to [b0 b2 b1 b3], giving (b0, b1) and (b2, b3).
// qh (Q5_K only) = qh[l..l+3]; bit 2c / 2c+1 of each byte is the fifth bit.
template <bool Q5, bool PERM>
__device__ __forceinline__ void kq_word(uint32_t w, uint32_t qh, int c, const KqConsts &k, uint32_t &lo01,
                                        uint32_t &lo23, uint32_t &hi01, uint32_t &hi23) {
    const uint32_t w2 = PERM ? w : prmt(w, 0u, 0x3120u), w3 = w2 >> 8;
    uint32_t l01 = and_or(w2, 0x000F000Fu, kH2_1024);   // (1024 + q)
    uint32_t l23 = and_or(w3, 0x000F000Fu, kH2_1024);
    uint32_t h01 = and_or(w2, 0x00F000F0u, kH2_1024);   // (1024 + 16 q)
    uint32_t h23 = and_or(w3, 0x00F000F0u, kH2_1024);
    if constexpr (Q5) {
        const uint32_t q2 = PERM ? qh : prmt(qh, 0u, 0x3120u), q3 = q2 >> 8;
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

// x of one stage: token t, 64-column segment R (= 4 * superblock + segment) is the 128-byte
// row t * 4S + R of a tile the TMA wrote with the 128-byte swizzle (16-byte chunk p of row r
// stored at chunk p ^ (r & 7)). xrow(r) gives the row base, chunk address = base ^ key.
struct XRow {
    uint32_t base, key;
};
__device__ __forceinline__ XRow xrow(uint32_t xst, uint32_t r) { return XRow{xst + r * 128u, (r & 7u) << 4}; }
__device__ __forceinline__ uint4 ldx(const XRow &x, uint32_t p) { return lds128(x.base + ((p << 4) ^ x.key)); }

// ---------------------------------------------------------------- per-format superblock

// Q4_K / Q5_K: lane (g, c) decodes 32-byte qs group c (sub-blocks 2c, 2c+1) of rows g, g+8.
// xr = row of columns 64c .. 64c+63 of this superblock.
// The min term sum_j dmin m_j sum_{k in j} x_k factors through the sums of x over the eight
// 32-wide sub-blocks (the group-sum idea). With XS those sums are staged (xsum = this
// superblock's 32-byte record for this lane's token: pair c holds the hi and lo fp16 halves of
// the sums of sub-blocks 2c, 2c+1) and ONE MMA with A = (m_2c, m_2c+1) in k-slots {2c, 2c+1}
// and again in {2c+8, 2c+9} against B = (hi, lo) yields sum_j m_j (hi_j + lo_j). Without XS
// every 16-wide piece runs its own MMA with A = m against x.
// swap16 = 16 swaps the two 16-byte halves of every 32-byte quant (and Q5_K high-bit) read: the
// lane then holds words 4..7 of its group first. The caller pairs it with x chunks p ^ 2 (an
// XRow whose key is XOR-ed with 32), so the contraction is unchanged; rows whose quants would share
// bank groups with the neighbouring row's (a row pitch that is a multiple of 32 bytes) use it on
// odd rows to keep the reads conflict-free.
template <int TYPE, bool PERM, bool XS>
__device__ __forceinline__ void superblock_kq(uint32_t blk_a, uint32_t blk_b, const XRow &xr, int c, float (&acc)[4],
                                              uint32_t xsum, uint32_t swap16 = 0) {
    constexpr bool Q5 = (TYPE == 13);
    constexpr uint32_t QS = Q5 ? 48 : 16;
    const uint4 ha = lds128(blk_a), hb = lds128(blk_b);
    const uint32_t q0 = QS + 32 * c + swap16, q1 = QS + 32 * c + (16u - swap16);
    const uint4 qa0 = lds128(blk_a + q0), qa1 = lds128(blk_a + q1);
    const uint4 qb0 = lds128(blk_b + q0), qb1 = lds128(blk_b + q1);
    uint4 ha0 = make_uint4(0, 0, 0, 0), ha1 = ha0, hb0 = ha0, hb1 = ha0;
    if constexpr (Q5) {
        ha0 = lds128(blk_a + 16 + swap16);
        ha1 = lds128(blk_a + 32 - swap16);
        hb0 = lds128(blk_b + 16 + swap16);
        hb1 = lds128(blk_b + 32 - swap16);
    }
    const KqConsts ka = kq_consts(ha, c), kb = kq_consts(hb, c);
    float d1[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 8; u += 2) {
        const uint4 xl = ldx(xr, u >> 1);         // columns 64c + 4u .. +7   (low nibbles)
        const uint4 xh = ldx(xr, 4 + (u >> 1));   // columns 64c + 32 + 4u .. (high nibbles)
#pragma unroll
        for (int v = 0; v < 2; ++v) {
            const int uu = u + v;
            uint32_t la01, la23, ha01, ha23, lb01, lb23, hb01, hb23;
            kq_word<Q5, PERM>(word_of(qa0, qa1, uu), word_of(ha0, ha1, uu), c, ka, la01, la23, ha01, ha23);
            kq_word<Q5, PERM>(word_of(qb0, qb1, uu), word_of(hb0, hb1, uu), c, kb, lb01, lb23, hb01, hb23);
            const uint32_t x0 = v ? xl.z : xl.x, x1 = v ? xl.w : xl.y;
            const uint32_t y0 = v ? xh.z : xh.x, y1 = v ? xh.w : xh.y;
            mma16816(d1, la01, lb01, la23, lb23, x0, x1);   // two independent accumulator chains
            mma16816(e1, ha01, hb01, ha23, hb23, y0, y1);
            if constexpr (!XS) {
                mma16816(d2, ka.m_lo, kb.m_lo, ka.m_lo, kb.m_lo, x0, x1);
                mma16816(d2, ka.m_hi, kb.m_hi, ka.m_hi, kb.m_hi, y0, y1);
            }
        }
    }
    if constexpr (XS) {
        const uint2 sums = lds64(xsum + 8u * c);   // (hi_2c, hi_2c+1), (lo_2c, lo_2c+1)
        mma16816(d2, ka.m_pair, kb.m_pair, ka.m_pair, kb.m_pair, sums.x, sums.y);
    }
    const float da = half_lo_to_float(ha.x), dma = half_hi_to_float(ha.x);
    const float db = half_lo_to_float(hb.x), dmb = half_hi_to_float(hb.x);
    acc[0] += da * (d1[0] + e1[0]) - dma * d2[0];
    acc[1] += da * (d1[1] + e1[1]) - dma * d2[1];
    acc[2] += db * (d1[2] + e1[2]) - dmb * d2[2];
    acc[3] += db * (d1[3] + e1[3]) - dmb * d2[3];
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
    const uint2 s = lds64_a2(blk + 192 + 8 * h);                       // int8 scales 8h .. 8h+7
    const uint32_t s0 = s.x ^ 0x80808080u, s1 = s.y ^ 0x80808080u;   // sc + 128 as unsigned bytes
    const uint32_t sel0 = e ? 0x4141u : 0x4040u, sel1 = e ? 0x4343u : 0x4242u;
    const uint32_t kH2_1152 = 0x64806480u;
    sc[0] = hsub2(prmt(s0, 0x64646464u, sel0), kH2_1152);   // scale 8h + e + 2t
    sc[1] = hsub2(prmt(s0, 0x64646464u, sel1), kH2_1152);
    sc[2] = hsub2(prmt(s1, 0x64646464u, sel0), kH2_1152);
    sc[3] = hsub2(prmt(s1, 0x64646464u, sel1), kH2_1152);
    d = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(blk + 208))));
}

// A pairs of quarter t for one (ql word, qh word) as sc*(q-32): columns (k0, k0+2) and
// (k0+1, k0+3) with permuted x (PERM), else (k0, k0+1) and (k0+2, k0+3).
template <bool PERM>
__device__ __forceinline__ void q6_pairs(uint32_t qlw, uint32_t qhw, int t, uint32_t sc, uint32_t &p01, uint32_t &p23) {
    uint32_t l2 = PERM ? qlw : prmt(qlw, 0u, 0x3120u);
    if (t >= 2) l2 >>= 4;
    const uint32_t h2 = PERM ? qhw : prmt(qhw, 0u, 0x3120u);
    uint32_t v01 = and_or(l2, 0x000F000Fu, kH2_1024);
    uint32_t v23 = and_or(l2 >> 8, 0x000F000Fu, kH2_1024);
    // bits 2t, 2t+1 of each qh byte -> bits 4, 5 of the half
    const int sh = 4 - 2 * t;
    const uint32_t h3 = h2 >> 8;
    v01 = or_and(v01, sh >= 0 ? (h2 << sh) : (h2 >> -sh), 0x00300030u);
    v23 = or_and(v23, sh >= 0 ? (h3 << sh) : (h3 >> -sh), 0x00300030u);
    p01 = hmul2(hsub2(v01, kH2_1056), sc);   // (q - 32) * sc
    p23 = hmul2(hsub2(v23, kH2_1056), sc);
}

// xs = x tile of this stage, r0 = token row base (tok * 4S + 4j).
// ALIGNED: blocks start on 16-byte boundaries (the 224-byte layout), so 16-byte loads need no
// realignment.
template <bool PERM, bool ALIGNED = false>
__device__ __forceinline__ void superblock_q6(uint32_t blk_a, uint32_t blk_b, uint32_t xs, uint32_t r0, int c,
                                              float (&acc)[4]) {
    const int h = c >> 1, e = c & 1;
    uint32_t sca[4], scb[4];
    float da, db;
    q6_row_consts(blk_a, h, e, sca, da);
    q6_row_consts(blk_b, h, e, scb, db);
    const uint32_t offA = 64 * h + 16 * e, offB = 64 * h + 32 + 16 * e, offH = 128 + 32 * h + 16 * e;
    auto ld16 = [](uint32_t a) { return ALIGNED ? lds128(a) : lds128_a2(a); };
    const uint4 qaA = ld16(blk_a + offA), qaB = ld16(blk_a + offB), qaH = ld16(blk_a + offH);
    const uint4 qbA = ld16(blk_b + offA), qbB = ld16(blk_b + offB), qbH = ld16(blk_b + offH);
    float d1[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        // columns 128h + 32t + 16e + 4u: segment 2h + t/2, chunk 4(t%2) + 2e + u/2
        const XRow xr = xrow(xs, r0 + 2 * h + t / 2);
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
            const uint4 xv = ldx(xr, 4 * (t & 1) + 2 * e + (u >> 1));
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const int uu = u + v;
                uint32_t a01, a23, b01, b23;
                q6_pairs<PERM>(word4((t & 1) ? qaB : qaA, uu), word4(qaH, uu), t, sca[t], a01, a23);
                q6_pairs<PERM>(word4((t & 1) ? qbB : qbA, uu), word4(qbH, uu), t, scb[t], b01, b23);
                if (v) mma16816(e1, a01, b01, a23, b23, xv.z, xv.w);
                else mma16816(d1, a01, b01, a23, b23, xv.x, xv.y);
            }
        }
    }
    acc[0] += da * (d1[0] + e1[0]);
    acc[1] += da * (d1[1] + e1[1]);
    acc[2] += db * (d1[2] + e1[2]);
    acc[3] += db * (d1[3] + e1[3]);
}

// IQ4_XS codebook (test/unit/test_llm_quant_cpu.py, test_unpack_lut_dot_uop) stored as
// unsigned bytes value + 128, four entries per register, entry 0 in the low byte.
constexpr uint32_t kIq4T0 = 0x3F2D1801u;   // -127 -104  -83  -65
constexpr uint32_t kIq4T1 = 0x766A5D4Fu;   //  -49  -35  -22  -10
constexpr uint32_t kIq4T2 = 0xA6998D81u;   //    1   13   25   38
constexpr uint32_t kIq4T3 = 0xF1D9C5B5u;   //   53   69   89  113

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

__device__ __forceinline__ void superblock_iq4(uint32_t blk_a, uint32_t blk_b, const XRow &xr, int c, float (&acc)[4]) {
    uint32_t lsa[2], nba[2], lsb[2], nbb[2];
    float da, db;
    iq4_row_consts(blk_a, c, lsa, nba, da);
    iq4_row_consts(blk_b, c, lsb, nbb, db);
    float d1[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t qoff = 8 + 32 * c + 16 * j;
        const uint2 a0 = lds64(blk_a + qoff), a1 = lds64(blk_a + qoff + 8);
        const uint2 b0 = lds64(blk_b + qoff), b1 = lds64(blk_b + qoff + 8);
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
            const uint4 xl = ldx(xr, 4 * j + (u >> 1));       // columns 64c + 32j + 4u ..
            const uint4 xh = ldx(xr, 4 * j + 2 + (u >> 1));   // columns 64c + 32j + 16 + 4u ..
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const int uu = u + v;
                const uint32_t wa = uu == 0 ? a0.x : uu == 1 ? a0.y : uu == 2 ? a1.x : a1.y;
                const uint32_t wb = uu == 0 ? b0.x : uu == 1 ? b0.y : uu == 2 ? b1.x : b1.y;
                uint32_t al01, al23, ah01, ah23, bl01, bl23, bh01, bh23;
                iq4_word(wa, lsa[j], nba[j], al01, al23, ah01, ah23);
                iq4_word(wb, lsb[j], nbb[j], bl01, bl23, bh01, bh23);
                mma16816(d1, al01, bl01, al23, bl23, v ? xl.z : xl.x, v ? xl.w : xl.y);
                mma16816(e1, ah01, bh01, ah23, bh23, v ? xh.z : xh.x, v ? xh.w : xh.y);
            }
        }
    }
    acc[0] += da * (d1[0] + e1[0]);
    acc[1] += da * (d1[1] + e1[1]);
    acc[2] += db * (d1[2] + e1[2]);
    acc[3] += db * (d1[3] + e1[3]);
}

}  // namespace
}  // namespace ql
