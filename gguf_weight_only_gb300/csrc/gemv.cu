// gemv.cu -- decode-path quantized linear y[M<=8, N] = x[M, K] . dequant(W)[N, K]^T, for one
// weight matrix or for up to four sharing x and K (projections; their row tiles form one list).
//
// Design (sm_103a):
//  * Persistent: one CTA per SM owns a contiguous run of 16-row tiles. Its warps are
//    (K slice, tile group) pairs: warp (kidx, tg) streams the superblocks of K slice kidx of
//    the CTA's tiles tg, tg + tgc, ... through its own ring of shared-memory stages. A stage
//    holds S superblocks of 16 rows and is filled by ONE 2-D TMA tensor copy (rows whose
//    byte length is a multiple of 16), else by one bulk copy per row over the 16-byte aligned
//    window around the row's span. Copies complete on the stage's mbarrier, so HBM bytes in
//    flight cost no registers, and every weight byte is read from HBM exactly once.
//  * The warp's slice of x (all tokens) lands once by TMA and is permuted in place into the
//    order the MMA fragments want (see below); for the K-quants the same pass stores the
//    sum of x over every 32-wide sub-block (fp16 hi + lo).
//  * Each lane decodes its share of a block in registers into fp16 pairs that are EXACT
//    integers (sc*q for K-quants, sc*(q-32) for Q6_K, (ls-32)*codebook[q] for IQ4_XS,
//    the last two rounded only beyond 2048) and feeds them to the legacy tensor core
//    (mma.sync m16n8k16, fp32 accumulate) with the tokens on the MMA's n = 8 side. The fp32
//    superblock scale d is applied to per-superblock fp32 partial sums; the K-quant min term
//    dmin * sum_j m_j * sum(x over sub-block j) is one MMA per superblock against the staged
//    sub-block sums.
//  * Per-tile partials of the warps go to shared memory; after a round of tiles they are
//    summed over the K slices in fixed order (deterministic).
//  * One token with K-quants or IQ4_XS (when each warp has at least 2 superblocks) takes a
//    specialised kernel that puts the eight sub-blocks on the MMA's n side instead of tokens,
//    feeds the quants as exact fp16 subnormals (IQ4_XS: codebook pairs from a byte table),
//    applies scales once per sub-block in fp32, and stages its x records straight from global
//    memory, without an x tile (see the single-token sections below). QL_GEMV_M1=0 in the
//    environment disables it (A/B timing).
//  * Variants of the launch (several projections; a fused prologue; the greedy-head epilogue)
//    are separate instantiations, so the plain kernel compiles as if they did not exist.
// Fragment ownership and the per-format decoders: decode.cuh.
#include <algorithm>
#include <cstdlib>
#include <cstdint>
#include <cuda.h>

#include "decode.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace ql {

namespace {

template <int TYPE>
struct GemvFmt;
// BB: bytes per superblock. MAXW: most warps per CTA. The decoders take 124 to 168 registers
// per thread; measured on GB300, 8 warps per SM (each with more superblocks per visit and a
// deeper share of shared memory) outrun 16, and capping registers to fit more warps loses.
template <>
struct GemvFmt<12> {   // Q4_K
    static constexpr int BB = 144, MAXW = 8;
};
template <>
struct GemvFmt<13> {   // Q5_K
    static constexpr int BB = 176, MAXW = 8;
};
template <>
struct GemvFmt<14> {   // Q6_K
    static constexpr int BB = 210, MAXW = 8;
};
template <>
struct GemvFmt<kQ6KAligned> {   // Q6_K in 224-byte blocks
    static constexpr int BB = 224, MAXW = 8;
};
template <>
struct GemvFmt<23> {   // IQ4_XS
    static constexpr int BB = 136, MAXW = 8;
};

int gemv_max_warps(int type) {
    switch (type) {
    case 12: return GemvFmt<12>::MAXW;
    case 13: return GemvFmt<13>::MAXW;
    case 14: return GemvFmt<14>::MAXW;
    case kQ6KAligned: return GemvFmt<kQ6KAligned>::MAXW;
    default: return GemvFmt<23>::MAXW;
    }
}

struct GemvArgs {
    // projections j < nproj share K and x: W[j] holds N[j] rows, y[j] is [M, N[j]], and
    // projection j owns row tiles [tile0[j], tile0[j+1]) of the concatenated tile space
    const uint8_t *W[kGemvMaxProj];
    float *y[kGemvMaxProj];
    int64_t total_bytes[kGemvMaxProj];   // bytes of W[j]
    int N[kGemvMaxProj];
    int tile0[kGemvMaxProj + 1];
    int nproj;
    const __half *x;
    unsigned *status;
    // Fused prologue (resident x only): 0 = x given; 1 = x = fp16(silu(gate) * up);
    // 2 = x = fp16(h * rsqrt(mean(h^2) + eps) * norm_w), also written to xnorm when set.
    int pro;
    const __half *gate;      // pro 1: [M, K]
    const float *up_or_h;    // pro 1: up [M, K]; pro 2: h [M, K]
    const float *norm_w;     // pro 2: [K]
    float eps;
    __half *xnorm;           // pro 2: optional [M, K] output of the normalised activations
    const float *residual;   // optional [M, N] added to y (single projection); may be y itself
    unsigned long long *best;  // greedy head: per token the largest packed (value, row) key, zeroed by the host
    int K, M, nsb;
    int S;                   // superblocks per stage
    int kw;                  // superblocks of the K slice each warp owns
    int ks, tgc;             // warp = tile group * ks + K slice: ks K slices x tgc tile groups
    int stages;              // ring depth per warp
    int xres;                // 1: x slice resident per warp; 0: x travels with each stage
    uint32_t row_pitch;      // bytes between rows inside a stage
    uint32_t w_bytes;        // weight bytes of a stage (16 * row_pitch)
    uint32_t x_bytes;        // per-stage x bytes inside a ring slot (0 when resident)
    uint32_t x_tx;           // bytes one x tensor copy delivers (all tokens)
    uint32_t x_warp_bytes;   // resident x region per warp
    uint32_t slot_bytes;     // one ring slot, rounded to 1 KB
    uint32_t red_offset, x_offset, ring_offset;
    int round_tiles;         // row tiles whose partials are reduced together (one barrier pair)
    int m1;                  // single-token kernel (sub-blocks on the MMA's n side)
    uint32_t lut_offset;     // single-token IQ4_XS: the replicated codebook byte table
    int qswap;               // single-token K-quants: odd-c lanes read their quant halves swapped
};

// Weight tensor maps, one per projection (unused entries stay zero).
struct GemvMaps {
    CUtensorMap m[kGemvMaxProj];
};

// ---------------------------------------------------------------- single-token K-quant path
//
// With one token the MMA's eight n columns would all carry the same x. Here they carry the
// eight 32-wide sub-blocks of the superblock instead: column j of B holds x only at the
// k-slots that come from sub-block j and zero elsewhere, so D[row][j] = sum over sub-block j
// of q * x, unscaled. Lane (g, c) decodes qs group c of rows g, g+8 (sub-blocks 2c from the
// low nibbles into k-slots 2c, 2c+1 and 2c+1 from the high nibbles into 2c+8, 2c+9) and holds
// exactly D[g][2c], D[g][2c+1], D[g+8][2c], D[g+8][2c+1] afterwards: its own sub-blocks. Their
// scales and mins are then applied once per sub-block in fp32, so the per-weight decode is only
// a mask: the masked nibble q (or 16 q for the high nibble) read as an fp16 bit pattern is the
// subnormal q * 2^-24 (or q * 2^-20), exact, and the tensor core multiplies subnormal fp16
// inputs exactly (checked on GB300), so D = 2^-24 sum q x (2^-20 for the high nibbles).
//
// B staging (per warp, once per launch): for superblock b of the slice and sub-block j, the
// 16 MMAs i = 2u + v (word u of the group, v = even/odd bytes) take the x pairs
// (x[32j + 4u + v], x[32j + 4u + v + 2]). Record (b, i) holds nine 8-byte slots: slot j is
// (b0, b1) for column j (the pair in b0 for even j, in b1 for odd j, the other half zero),
// slot 8 is zero. Lane (g, c) reads slot g when g >> 1 == c and slot 8 otherwise, so the
// warp's reads of one record cover 72 contiguous bytes (no bank conflicts). The fp32 sums of
// x over every sub-block (the min term) are staged after the records.

constexpr uint32_t kM1Rec = 72, kM1Sb = 16 * kM1Rec;   // record and superblock strides of the staged B

// Chunk `lane` (x[8 lane .. 8 lane + 7]) of superblock b of the slice, already in registers, laid
// out as the plain staging lays out its items 2 (lane & 3) and 2 (lane & 3) + 1 of sub-block
// lane >> 2. The sub-block sum is formed in the plain staging's order: each item's pair sums,
// then the item pair (in lane), then shuffles across the sub-block's four lanes (fp32 addition
// is commutative, so every lane of a pair holds the same sum at each step).
__device__ __forceinline__ void m1_stage_chunk(const uint4 &v, int b, uint32_t xexp, uint32_t xsums, int lane, int qswap) {
    const uint32_t j = static_cast<uint32_t>(lane) >> 2, m = static_cast<uint32_t>(lane) & 3u;
    float s2[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t vx = h ? v.z : v.x, vy = h ? v.w : v.y;
        const uint32_t u = 2u * m + static_cast<uint32_t>(h);
        const uint32_t p02 = prmt(vx, vy, 0x5410u), p13 = prmt(vx, vy, 0x7632u);
        const uint32_t us = u ^ ((qswap && ((j >> 1) & 1u)) ? 4u : 0u);
        const uint32_t e = xexp + static_cast<uint32_t>(b) * kM1Sb + (2u * us) * kM1Rec + 8u * j;
        if (j & 1u) {
            sts64(e, 0u, p02);
            sts64(e + kM1Rec, 0u, p13);
        } else {
            sts64(e, p02, 0u);
            sts64(e + kM1Rec, p13, 0u);
        }
        if (j == 0u) {
            sts64(e + 64u, 0u, 0u);
            sts64(e + kM1Rec + 64u, 0u, 0u);
        }
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&vx));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&vy));
        s2[h] = (f0.x + f0.y) + (f1.x + f1.y);
    }
    float sum = s2[0] + s2[1];
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
    if (m == 0u) sts32(xsums + (static_cast<uint32_t>(b) * 8u + j) * 4u, __float_as_uint(sum));
}

// IQ4_XS: the lanes holding the first half of a sub-block (lane & 3 < 2) lay out their two items
// with the x[k+16 ..] words taken from the lane two above.
__device__ __forceinline__ void m1_stage_iq4_chunk(const uint4 &v, int b, uint32_t xexp, int lane) {
    const uint4 w = make_uint4(__shfl_xor_sync(0xFFFFFFFFu, v.x, 2), __shfl_xor_sync(0xFFFFFFFFu, v.y, 2),
                               __shfl_xor_sync(0xFFFFFFFFu, v.z, 2), __shfl_xor_sync(0xFFFFFFFFu, v.w, 2));
    const uint32_t j = static_cast<uint32_t>(lane) >> 2, m = static_cast<uint32_t>(lane) & 3u;
    if (m >= 2u) return;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t uq = 2u * m + static_cast<uint32_t>(h);
        const uint32_t vx = h ? v.z : v.x, vy = h ? v.w : v.y, wx = h ? w.z : w.x, wy = h ? w.w : w.y;
        const uint32_t w4 = uq + 4u * (j & 1u), u = w4 ^ (2u * (j >> 1));
        const uint32_t e = xexp + static_cast<uint32_t>(b) * kM1Sb + (2u * u) * kM1Rec;
        sts64(e + 8u * j, prmt(vx, wx, 0x5410u), prmt(vx, wx, 0x7632u));            // h = 0
        sts64(e + kM1Rec + 8u * j, prmt(vy, wy, 0x5410u), prmt(vy, wy, 0x7632u));   // h = 1
        sts64(e + 8u * (j ^ 1u), 0u, 0u);
        sts64(e + kM1Rec + 8u * (j ^ 1u), 0u, 0u);
        if (j < 2u) {
            sts64(e + 64u, 0u, 0u);
            sts64(e + kM1Rec + 64u, 0u, 0u);
        }
    }
}

// Builds the staged B records and the fp32 sub-block sums straight from x in global memory:
// superblocks [kb0, kb0 + kw) of the warp's slice, those at or past nsb as zeros. Item q
// (sub-block j = q >> 3 & 7, word u = q & 7) of a superblock is x[4q .. 4q+3], so a warp's 32
// items are 256 contiguous bytes; eight items per lane are loaded before any is used. Reading x
// directly saves a tensor copy's round trip through a barrier and a shared-memory tile.
__device__ __forceinline__ void m1_stage_global(const __half *x, int kb0, int nsb, uint32_t xexp, uint32_t xsums,
                                                int kw, int lane, int qswap) {
    constexpr int kBatch = 8;
    const uint32_t nitems = 64u * static_cast<uint32_t>(kw);   // a multiple of 32
    for (uint32_t q0 = lane; q0 < nitems; q0 += 32u * kBatch) {
        uint2 vv[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const uint32_t q = q0 + 32u * i, b = q >> 6;
            vv[i] = make_uint2(0u, 0u);
            if (q < nitems && kb0 + static_cast<int>(b) < nsb)
                vv[i] = __ldg(reinterpret_cast<const uint2 *>(x + static_cast<int64_t>(kb0 + static_cast<int>(b)) * 256 +
                                                              4u * (q & 63u)));
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const uint32_t q = q0 + 32u * i;
            if (q >= nitems) break;   // warp-uniform: nitems is a multiple of 32
            const uint32_t u = q & 7u, j = (q >> 3) & 7u, b = q >> 6;
            const uint2 v = vv[i];
            const uint32_t p02 = prmt(v.x, v.y, 0x5410u), p13 = prmt(v.x, v.y, 0x7632u);   // (x0, x2), (x1, x3)
            const uint32_t us = u ^ ((qswap && ((j >> 1) & 1u)) ? 4u : 0u);
            const uint32_t e = xexp + b * kM1Sb + (2u * us) * kM1Rec + 8u * j;
            if (j & 1u) {
                sts64(e, 0u, p02);
                sts64(e + kM1Rec, 0u, p13);
            } else {
                sts64(e, p02, 0u);
                sts64(e + kM1Rec, p13, 0u);
            }
            if (j == 0u) {
                sts64(e + 64u, 0u, 0u);
                sts64(e + kM1Rec + 64u, 0u, 0u);
            }
            const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
            const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
            float sum = (f0.x + f0.y) + (f1.x + f1.y);
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 4);
            if (u == 0u) sts32(xsums + (b * 8u + j) * 4u, __float_as_uint(sum));
        }
    }
}

// One superblock of rows g, g+8 for the single-token path: acc[0] (row g) and acc[1] (row
// g+8) gain this lane's two sub-blocks. bx = the lane's slot in the superblock's first staged
// record, sums = the superblock's eight fp32 sub-block sums of x.
// swap16 = 16 for lanes that read their 32-byte quant group as (second, first) half: with a stage
// pitch of 32 or 96 (mod 128) bytes rows g and g+1 sit 2 or 6 bank groups apart and the lanes of
// odd c then fill the bank groups the even ones leave (4 wavefronts per 16-byte load instead of
// 8); the staged records of their columns are stored in the same order.
template <int TYPE>
__device__ __forceinline__ void superblock_kq_m1(uint32_t blk_a, uint32_t blk_b, uint32_t bx, uint32_t sums, int c,
                                                 uint32_t swap16, float (&acc)[2]) {
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
    float d1[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t rl = (4u - 2u * c) & 31u, rh = (7u - 2u * c) & 31u;   // Q5_K: bit 2c -> bit 4, 2c+1 -> bit 8
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint32_t wa = word_of(qa0, qa1, u), wb = word_of(qb0, qb1, u);
        const uint32_t wa3 = wa >> 8, wb3 = wb >> 8;
        uint32_t la02 = wa & 0x000F000Fu, la13 = wa3 & 0x000F000Fu;   // q         (bytes 0,2 / 1,3)
        uint32_t ha02 = wa & 0x00F000F0u, ha13 = wa3 & 0x00F000F0u;   // 16 q
        uint32_t lb02 = wb & 0x000F000Fu, lb13 = wb3 & 0x000F000Fu;
        uint32_t hb02 = wb & 0x00F000F0u, hb13 = wb3 & 0x00F000F0u;
        if constexpr (Q5) {
            const uint32_t qa = word_of(ha0, ha1, u), qb = word_of(hb0, hb1, u);
            const uint32_t qa3 = qa >> 8, qb3 = qb >> 8;
            la02 = or_and(la02, rotl(qa, rl), 0x00100010u);
            la13 = or_and(la13, rotl(qa3, rl), 0x00100010u);
            ha02 = or_and(ha02, rotl(qa, rh), 0x01000100u);
            ha13 = or_and(ha13, rotl(qa3, rh), 0x01000100u);
            lb02 = or_and(lb02, rotl(qb, rl), 0x00100010u);
            lb13 = or_and(lb13, rotl(qb3, rl), 0x00100010u);
            hb02 = or_and(hb02, rotl(qb, rh), 0x01000100u);
            hb13 = or_and(hb13, rotl(qb3, rh), 0x01000100u);
        }
        const uint2 B0 = lds64(bx + (2u * u) * kM1Rec), B1 = lds64(bx + (2u * u + 1u) * kM1Rec);
        mma16816(d1, la02, lb02, ha02, hb02, B0.x, B0.y);
        mma16816(e1, la13, lb13, ha13, hb13, B1.x, B1.y);
    }
    // scales and mins of sub-blocks 2c, 2c+1 (12-byte field, header words y, z, w)
    auto scm = [&](const uint4 &h, float &s0, float &s1, float &m0, float &m1) {
        const uint32_t A = h.y, B = h.z, C = h.w;
        const uint32_t sc_lo4 = A & 0x3F3F3F3Fu, m_lo4 = B & 0x3F3F3F3Fu;
        const uint32_t sc_hi4 = and_or(C, 0x0F0F0F0Fu, (A >> 2) & 0x30303030u);
        const uint32_t m_hi4 = and_or(C >> 4, 0x0F0F0F0Fu, (B >> 2) & 0x30303030u);
        const uint32_t sel = (2u * c) | ((2u * c + 1u) << 4);
        const uint32_t vs = prmt(sc_lo4, sc_hi4, sel), vm = prmt(m_lo4, m_hi4, sel);
        s0 = static_cast<float>(vs & 0xFFu);
        s1 = static_cast<float>((vs >> 8) & 0xFFu);
        m0 = static_cast<float>(vm & 0xFFu);
        m1 = static_cast<float>((vm >> 8) & 0xFFu);
    };
    float sa0, sa1, ma0, ma1, sb0, sb1, mb0, mb1;
    scm(ha, sa0, sa1, ma0, ma1);
    scm(hb, sb0, sb1, mb0, mb1);
    const uint2 xs2 = lds64(sums + 8u * c);   // sums of x over sub-blocks 2c, 2c+1
    const float xs0 = __uint_as_float(xs2.x), xs1 = __uint_as_float(xs2.y);
    const float da = half_lo_to_float(ha.x), dma = half_hi_to_float(ha.x);
    const float db = half_lo_to_float(hb.x), dmb = half_hi_to_float(hb.x);
    constexpr float k24 = 16777216.0f, k20 = 1048576.0f;   // 2^24, 2^20
    acc[0] += da * (sa0 * k24 * (d1[0] + e1[0]) + sa1 * k20 * (d1[1] + e1[1])) - dma * (ma0 * xs0 + ma1 * xs1);
    acc[1] += db * (sb0 * k24 * (d1[2] + e1[2]) + sb1 * k20 * (d1[3] + e1[3])) - dmb * (mb0 * xs0 + mb1 * xs1);
}

// ---------------------------------------------------------------- single-token IQ4_XS path
//
// IQ4_XS takes the same column scheme with the codebook lookup moved into shared memory: a table
// of the 256 quant bytes whose entry is the fp16 pair (kv[b & 15], kv[b >> 4]) (exact integers,
// so D[row][j] is the unscaled sum over sub-block j of kv * x and d (ls_j - 32) is applied once
// per sub-block in fp32). The table is replicated 32 times and lane l reads copy l (entry b of
// copy l at b * 128 + 4 l, always bank l): one conflict-free 32-bit load per quant byte replaces
// the byte-permute lookup, moving the decode's cost from the integer pipe to shared memory.
// Quant byte p of a sub-block holds weights p (low nibble) and p + 16 (high nibble), so a table
// entry is the A pair of one k-slot pair and the staged B holds (x_p, x_{p+16}).
//
// Lane (g, c) decodes qs bytes 32c .. 32c+31 of rows g, g+8 (words w = 0..3: sub-block 2c,
// 4..7: 2c+1), reading its four 8-byte chunks in the order i ^ c: at step u it holds word
// w = u ^ 2c, which spreads a warp's chunk loads over all banks (two wavefronts each) at every
// stage pitch but those of 64 mod 128 bytes. MMA (u, h) takes bytes 2h, 2h+1 of that word:
// a0 / a1 = the entries of byte 2h of rows g / g+8, a2 / a3 = byte 2h+1. Record (b, 2u + h)
// holds in slot j, for the four columns the lanes carry at step u, the pairs (x[p], x[p+16]),
// (x[p+1], x[p+17]) with p = 32j + 4(w & 3) + 2h and w = u ^ 2(j >> 1); its other four slots
// and slot 8 are zero.
constexpr uint32_t kIq4LutBytes = 256u * 128u;

// Codebook value kv[i] (the IQ4 tables hold kv + 128 bytes).
__device__ __forceinline__ int iq4_kv(uint32_t i) {
    const uint32_t t = (i < 4) ? kIq4T0 : (i < 8) ? kIq4T1 : (i < 12) ? kIq4T2 : kIq4T3;
    return static_cast<int>((t >> (8u * (i & 3u))) & 0xFFu) - 128;
}

// All threads of the CTA fill the table (run before the dependency wait: it is constant).
__device__ __forceinline__ void iq4_lut_fill(uint32_t lut) {
    for (uint32_t i = threadIdx.x; i < 256u * 32u; i += blockDim.x) {
        const uint32_t b = i >> 5, l = i & 31u;
        const uint32_t lo = __half_as_ushort(__int2half_rn(iq4_kv(b & 15u)));
        const uint32_t hi = __half_as_ushort(__int2half_rn(iq4_kv(b >> 4)));
        sts32(lut + b * 128u + 4u * l, lo | (hi << 16));
    }
}

// The staged B records of the IQ4_XS single-token path, read straight from x in global memory
// (superblocks at or past nsb as zeros; eight items per lane loaded before any is stored). Item
// (b, j, word w & 3) writes slot j of records 2u, 2u+1 (u = w ^ 2 (j >> 1), the step at which
// its carrier holds word w) and zeros slot j ^ 1 of them; the zero slot 8 is written by the
// items of sub-blocks 0 and 1.
__device__ __forceinline__ void m1_stage_iq4_global(const __half *x, int kb0, int nsb, uint32_t xexp, int kw, int lane) {
    constexpr int kBatch = 8;
    const uint32_t nitems = 32u * static_cast<uint32_t>(kw);   // a multiple of 32
    for (uint32_t q0 = lane; q0 < nitems; q0 += 32u * kBatch) {
        uint2 vv[kBatch], ww[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const uint32_t q = q0 + 32u * i, b = q >> 5;
            const uint32_t k = 32u * ((q >> 2) & 7u) + 4u * (q & 3u);
            vv[i] = ww[i] = make_uint2(0u, 0u);
            if (q < nitems && kb0 + static_cast<int>(b) < nsb) {
                const __half *xs = x + static_cast<int64_t>(kb0 + static_cast<int>(b)) * 256 + k;
                vv[i] = __ldg(reinterpret_cast<const uint2 *>(xs));        // x[k .. k+3]
                ww[i] = __ldg(reinterpret_cast<const uint2 *>(xs + 16));   // x[k+16 .. k+19]
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const uint32_t q = q0 + 32u * i;
            if (q >= nitems) break;   // warp-uniform: nitems is a multiple of 32
            const uint32_t uq = q & 3u, j = (q >> 2) & 7u, b = q >> 5;
            const uint32_t w4 = uq + 4u * (j & 1u), u = w4 ^ (2u * (j >> 1));
            const uint2 v = vv[i], w = ww[i];
            const uint32_t e = xexp + b * kM1Sb + (2u * u) * kM1Rec;
            sts64(e + 8u * j, prmt(v.x, w.x, 0x5410u), prmt(v.x, w.x, 0x7632u));            // h = 0
            sts64(e + kM1Rec + 8u * j, prmt(v.y, w.y, 0x5410u), prmt(v.y, w.y, 0x7632u));   // h = 1
            sts64(e + 8u * (j ^ 1u), 0u, 0u);
            sts64(e + kM1Rec + 8u * (j ^ 1u), 0u, 0u);
            if (j < 2u) {
                sts64(e + 64u, 0u, 0u);
                sts64(e + kM1Rec + 64u, 0u, 0u);
            }
        }
    }
}

// One IQ4_XS superblock of rows g, g+8 for the single-token path: acc[0] (row g) and acc[1]
// (row g+8) gain this lane's sub-blocks 2c, 2c+1. bx_lo / bx_hi = the lane's slot in the
// superblock's first record for steps 0-3 / 4-7 (the column it carries then, or the zero
// slot); lutl = this lane's copy of the byte table.
__device__ __forceinline__ void superblock_iq4_m1(uint32_t blk_a, uint32_t blk_b, uint32_t bx_lo, uint32_t bx_hi,
                                                  uint32_t lutl, int c, float (&acc)[2]) {
    const uint2 ha = lds64(blk_a), hb = lds64(blk_b);
    uint2 qa[4], qb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        qa[i] = lds64(blk_a + 8 + 32 * c + 8 * (i ^ c));
        qb[i] = lds64(blk_b + 8 + 32 * c + 8 * (i ^ c));
    }
    float d1[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
    auto entry = [&](uint32_t w, uint32_t k) { return lds32(lutl + 128u * prmt(w, 0u, 0x4440u | k)); };
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint32_t wa = (u & 1) ? qa[u >> 1].y : qa[u >> 1].x, wb = (u & 1) ? qb[u >> 1].y : qb[u >> 1].x;
        const uint32_t bx = u < 4 ? bx_lo : bx_hi;
        const uint2 B0 = lds64(bx + (2u * u) * kM1Rec), B1 = lds64(bx + (2u * u + 1u) * kM1Rec);
        mma16816(d1, entry(wa, 0), entry(wb, 0), entry(wa, 1), entry(wb, 1), B0.x, B0.y);
        mma16816(e1, entry(wa, 2), entry(wb, 2), entry(wa, 3), entry(wb, 3), B1.x, B1.y);
    }
    // ls of sub-blocks 2c, 2c+1: low nibble from scales_l (bytes 4..7 of the block), high two
    // bits from scales_h (bytes 2, 3)
    auto ls_pair = [&](const uint2 &h, float &l0, float &l1) {
        const uint32_t lo = (h.y >> (8 * c)) & 0xFFu, hi2 = (h.x >> (16 + 4 * c)) & 0xFu;
        l0 = static_cast<float>(static_cast<int>((lo & 15u) | ((hi2 & 3u) << 4)) - 32);
        l1 = static_cast<float>(static_cast<int>((lo >> 4) | ((hi2 >> 2) << 4)) - 32);
    };
    float la0, la1, lb0, lb1;
    ls_pair(ha, la0, la1);
    ls_pair(hb, lb0, lb1);
    const float da = half_lo_to_float(ha.x), db = half_lo_to_float(hb.x);
    acc[0] += da * (la0 * (d1[0] + e1[0]) + la1 * (d1[1] + e1[1]));
    acc[1] += db * (lb0 * (d1[2] + e1[2]) + lb1 * (d1[3] + e1[3]));
}

// ---------------------------------------------------------------- fused prologues

// Shared-memory scratch after the warps' ring barriers (the barrier region is padded to whole
// kilobytes and ends at red_offset): the RMSNorm prologue's per-warp partial sums of h^2 for
// each token, then the greedy-head epilogue's per-warp best keys of one token.
__host__ __device__ constexpr uint32_t scratch_offset(int warps, int stages) {
    return (8u * static_cast<uint32_t>(warps) * static_cast<uint32_t>(stages + 1) + 15u) & ~15u;
}
constexpr uint32_t kScratchBytes = 4u * 16u * kGemvMaxM + 8u * 16u;   // up to 16 warps

// Key whose unsigned order is (value, then the smaller row): the float's bits made monotonic
// (+0 and -0 made equal), then the row counted down from 2^32 - 1.
__device__ __forceinline__ unsigned long long argmax_key(float v, int row) {
    const uint32_t bits = (v == 0.f) ? 0u : __float_as_uint(v);
    const uint32_t ord = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
    return (static_cast<unsigned long long>(ord) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(row));
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// silu(g) * u in fp32: g / (1 + e^-g), with e^-g capped at e^80 (where silu rounds to 0 in
// fp16 anyway) so that the fast division stays in its exact range. __expf and __fdividef err
// by a few fp32 ulp, far below the fp16 rounding that follows.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f))) * u;
}

// Inputs of eight consecutive activations x[tok][k0 .. k0+7] of a fused prologue.
struct ChunkIn {
    uint4 gate;          // pro 1: 8 fp16
    float4 a0, a1;       // pro 1: up; pro 2: h
    float4 w0, w1;       // pro 2: norm weight
};

__device__ __forceinline__ ChunkIn chunk_load(const GemvArgs &p, int tok, int64_t k0) {
    ChunkIn c;
    const int64_t o = static_cast<int64_t>(tok) * p.K + k0;
    c.a0 = __ldg(reinterpret_cast<const float4 *>(p.up_or_h + o));
    c.a1 = __ldg(reinterpret_cast<const float4 *>(p.up_or_h + o) + 1);
    if (p.pro == 1) {
        c.gate = __ldg(reinterpret_cast<const uint4 *>(p.gate + o));
    } else {
        c.w0 = __ldg(reinterpret_cast<const float4 *>(p.norm_w + k0));
        c.w1 = __ldg(reinterpret_cast<const float4 *>(p.norm_w + k0) + 1);
    }
    return c;
}

// The eight activations as fp16 in k order, each rounded once from fp32.
__device__ __forceinline__ uint4 chunk_compute(const GemvArgs &p, const ChunkIn &c, float rstd) {
    float v[8];
    if (p.pro == 1) {
        const __half2 *g2 = reinterpret_cast<const __half2 *>(&c.gate);
        const float2 g0 = __half22float2(g2[0]), g1 = __half22float2(g2[1]);
        const float2 g2f = __half22float2(g2[2]), g3 = __half22float2(g2[3]);
        v[0] = silu_mul(g0.x, c.a0.x); v[1] = silu_mul(g0.y, c.a0.y);
        v[2] = silu_mul(g1.x, c.a0.z); v[3] = silu_mul(g1.y, c.a0.w);
        v[4] = silu_mul(g2f.x, c.a1.x); v[5] = silu_mul(g2f.y, c.a1.y);
        v[6] = silu_mul(g3.x, c.a1.z); v[7] = silu_mul(g3.y, c.a1.w);
    } else {
        v[0] = c.a0.x * rstd * c.w0.x; v[1] = c.a0.y * rstd * c.w0.y;
        v[2] = c.a0.z * rstd * c.w0.z; v[3] = c.a0.w * rstd * c.w0.w;
        v[4] = c.a1.x * rstd * c.w1.x; v[5] = c.a1.y * rstd * c.w1.y;
        v[6] = c.a1.z * rstd * c.w1.z; v[7] = c.a1.w * rstd * c.w1.w;
    }
    return make_uint4(pack_half2(v[0], v[1]), pack_half2(v[2], v[3]), pack_half2(v[4], v[5]), pack_half2(v[6], v[7]));
}

// Chunks a lane fills per group of a fused prologue: their global loads are all issued before
// any is used.
constexpr int kFillGroup = 4;

// ---------------------------------------------------------------- the kernel
//
// Persistent: CTA b owns a contiguous run of 16-row tiles (an equal share of the T tiles of all
// projections, G = grid size, one CTA per SM). Warp (kidx, tg) owns the fixed K slice of
// superblocks [kidx kw, (kidx+1) kw) of the CTA's tiles tg, tg + tgc, ..., so its slice of x
// is loaded once (xres) or, when that does not fit, with each stage. Each warp streams its
// units (tile, stage of S superblocks) through a ring of `stages` slots, issuing a slot's
// next unit as soon as it has consumed it, across tile boundaries. The warps' 16 x 8 partial
// tiles go to shared memory; after each round of tiles they are summed in fixed order.

template <int TYPE, bool TMA, bool XRES, bool MULTI, bool PRO, bool ARGMAX, bool M1>
__global__ void __launch_bounds__(32 * GemvFmt<TYPE>::MAXW, 1) gemv_kernel(const __grid_constant__ GemvMaps wmaps,
                                                      const __grid_constant__ CUtensorMap xmap,
                                                      const __grid_constant__ GemvArgs p) {
    constexpr int BB = GemvFmt<TYPE>::BB;
    constexpr bool PERM = XRES && TYPE != 23 && !M1;   // resident x is permuted once for the K-quant/Q6_K pairing
    constexpr bool XSUM = XRES && (TYPE == 12 || TYPE == 13) && !M1;   // staged sub-block sums of x (min term)
    static_assert(!M1 || (XRES && (TYPE == 12 || TYPE == 13 || TYPE == 23)),
                  "single-token path: K-quants and IQ4_XS, resident x");
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int D = p.stages, S = p.S;

    const uint32_t base = (smem_u32(smem) + 1023u) & ~1023u;   // the launch adds 1 KB of slack
    uint8_t *const gbase = smem + (base - smem_u32(smem));
    float *red = reinterpret_cast<float *>(gbase + p.red_offset);   // [round tile][K slice][token][16 rows]
    const uint32_t bar0 = base + 8u * warp * (D + 1);              // D ring barriers + 1 x barrier
    const uint32_t xbar = bar0 + 8u * D;
    const uint32_t xreg = base + p.x_offset + warp * p.x_warp_bytes;
    const uint32_t xsum_base = xreg + p.x_tx;   // XSUM: [token][superblock of the slice] x 32 bytes
    // M1: staged B records [superblock][16 MMAs][9 slots] x 8 bytes, then fp32 sums [superblock][8]
    const uint32_t xexp = xreg, xsums = xexp + kM1Sb * p.kw;   // (no x tile in the single-token kernels)
    const uint32_t ring = base + p.ring_offset + warp * D * p.slot_bytes;

    const uint32_t ring_end = base + p.ring_offset + (blockDim.x >> 5) * D * p.slot_bytes;
    if constexpr (kBoundsChecks) {   // the layout inside the launch's dynamic shared memory
        uint32_t dyn;
        asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
        const bool lay = ring_end - smem_u32(smem) <= dyn && p.red_offset >= scratch_offset(blockDim.x >> 5, D) &&
                         p.x_offset >= p.red_offset && p.ring_offset >= p.x_offset + (blockDim.x >> 5) * p.x_warp_bytes &&
                         (!XRES || (M1 ? kM1Sb * p.kw + (TYPE == 23 ? 0u : 32u * p.kw) <= p.x_warp_bytes
                                       : p.x_tx <= p.x_warp_bytes)) &&
                         p.w_bytes + (XRES ? 0u : p.x_bytes) <= p.slot_bytes &&
                         (!(M1 && TYPE == 23) || (p.lut_offset >= p.red_offset && p.lut_offset + kIq4LutBytes <= p.x_offset));
        if (!in_bounds(lay, p.status)) return;
    }
    const int G = gridDim.x, b = blockIdx.x;
    const int T = p.tile0[p.nproj];   // row tiles of all projections; CTA b owns [T b / G, T (b+1) / G)
    const int t_begin = static_cast<int>(static_cast<int64_t>(T) * b / G);
    const int t_end = static_cast<int>(static_cast<int64_t>(T) * (b + 1) / G);
    const int ntiles = t_end - t_begin;
    // CTA-local tile t -> its projection j and its first row within that projection
    auto tile_rows = [&](int t, int &j) {
        const int gt = t_begin + t;
        j = 0;
        if constexpr (!MULTI) {
            return 16 * gt;   // one projection: the lookup cost 3-4% on GB300
        } else {
            while (j + 1 < p.nproj && gt >= p.tile0[j + 1]) ++j;
            return 16 * (gt - p.tile0[j]);
        }
    };

    // warp = (tile group tg, K slice kidx): it owns superblocks [kb0, kb1) of the CTA's tiles
    // tg, tg + tgc, tg + 2 tgc, ...
    const int kidx = warp % p.ks, tg = warp / p.ks;
    const int kb0 = kidx * p.kw;
    const int kb1 = min(kb0 + p.kw, p.nsb);
    const int nmine = max(kb1 - kb0, 0);
    const int nst = (nmine + S - 1) / S;   // stages per tile for this warp (0 for idle warps)
    const int mytiles = ntiles > tg ? (ntiles - tg + p.tgc - 1) / p.tgc : 0;
    const int total = mytiles * nst;

    if (lane == 0) {
        for (int s = 0; s <= D; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
        if constexpr (!PRO) prefetch_tmap(&xmap);
        if constexpr (TMA)
            for (int j = 0; j < p.nproj; ++j) prefetch_tmap(&wmaps.m[j]);
    }
    __syncwarp();

    // x slot of a ring slot (per-stage x) sits in front of its weights
    auto wslot = [&](int s) { return ring + s * p.slot_bytes + (XRES ? 0u : p.x_bytes); };
    auto xslot = [&](int s) { return ring + s * p.slot_bytes; };

    auto issue = [&](int s, int t, int si) {
        const int sb = kb0 + si * S;
        int j;
        const int row0 = tile_rows(t, j);
        const uint32_t bar = bar0 + 8 * s;
        const uint32_t xtx = XRES ? 0u : p.x_tx;
        if constexpr (TMA) {
            if (lane == 0) {
                if (in_bounds(s < D && wslot(s) + p.w_bytes <= ring + (s + 1) * p.slot_bytes && sb < p.nsb &&
                                  (XRES || xslot(s) + xtx <= wslot(s)),
                              p.status)) {
                    mbar_arrive_expect_tx(bar, p.w_bytes + xtx);
                    tma_load_2d(wslot(s), &wmaps.m[j], sb * (BB / 8), row0, bar);
                    if (!XRES) tma_load_3d(xslot(s), &xmap, 0, sb * 4, 0, bar);
                } else {
                    mbar_arrive(bar);
                }
            }
        } else {
            const int ns = min(S, kb1 - sb);
            uint32_t nbytes = 0, dst = 0;
            const uint8_t *src = nullptr;
            int tail_len = 0;
            uint32_t tail_off = 0;
            int64_t t16 = 0;
            const uint8_t *const W = p.W[j];
            if (lane < 16 && row0 + lane < p.N[j]) {
                const int64_t o = (static_cast<int64_t>(row0 + lane) * p.nsb + sb) * BB;
                const int64_t lo = o & ~int64_t(15);
                int64_t hi = (o + static_cast<int64_t>(ns) * BB + 15) & ~int64_t(15);
                t16 = p.total_bytes[j] & ~int64_t(15);
                if (hi > t16) {   // the span ends in the last, partial 16 bytes of W
                    hi = t16;
                    tail_len = static_cast<int>(o + static_cast<int64_t>(ns) * BB - t16);
                    tail_off = static_cast<uint32_t>(t16 - lo);
                }
                const int64_t end = o + static_cast<int64_t>(ns) * BB;
                if (in_bounds(lo >= 0 && end <= p.total_bytes[j] && (end + 15 - lo) / 16 * 16 <= p.row_pitch &&
                                  wslot(s) + (lane + 1) * p.row_pitch <= ring + (s + 1) * p.slot_bytes,
                              p.status)) {
                    src = W + lo;
                    dst = wslot(s) + lane * p.row_pitch;
                    nbytes = static_cast<uint32_t>(hi - lo);
                } else {
                    tail_len = 0;
                }
            }
            if (tail_len > 0) {
                uint8_t *gd = smem + (dst + tail_off - smem_u32(smem));
                for (int i = 0; i < tail_len; ++i) gd[i] = __ldg(W + t16 + i);
            }
            const uint32_t sum = __reduce_add_sync(0xFFFFFFFFu, nbytes);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_expect_tx(bar, sum + xtx);
                if (!XRES) tma_load_3d(xslot(s), &xmap, 0, sb * 4, 0, bar);
            }
            __syncwarp();
            if (nbytes) bulk_g2s(dst, src, nbytes, bar);
        }
    };

    // Weights are constant inputs: their first stages stream while the preceding kernel in the
    // stream finishes. x (and, per stage, its x tiles) is read only after that kernel is done.
    pdl_launch_dependents();
    bool ok = true;
    int it = 0, isi = 0;   // next stage to issue: my tile it, stage isi (counters, no division)
    auto issue_next = [&](int s) {
        issue(s, tg + it * p.tgc, isi);
        if (++isi == nst) {
            isi = 0;
            ++it;
        }
    };
    if constexpr (XRES) {
        for (int s = 0; s < D && s < total; ++s) issue_next(s);
        if constexpr (M1 && TYPE == 23) {   // the codebook table: constant, built before the wait
            iq4_lut_fill(base + p.lut_offset);
            __syncthreads();
        }
        pdl_wait();
        float *const sq = reinterpret_cast<float *>(gbase + scratch_offset(blockDim.x >> 5, D));   // [warp][token]
        if (PRO && p.pro == 2) {
            // sum of h^2 per token: each warp a strided share of the row, fixed order
            const int kstep = static_cast<int>(blockDim.x) * 4;
            for (int m = 0; m < p.M; ++m) {
                const float *hrow = p.up_or_h + static_cast<int64_t>(m) * p.K;
                float acc2 = 0.f;
                for (int k0 = (warp * 32 + lane) * 4; k0 < p.K; k0 += 8 * kstep) {
                    float4 h[8];   // eight independent loads in flight, then summed in order
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        h[i] = k0 + i * kstep < p.K ? __ldg(reinterpret_cast<const float4 *>(hrow + k0 + i * kstep))
                                                    : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc2 += (h[i].x * h[i].x + h[i].y * h[i].y) + (h[i].z * h[i].z + h[i].w * h[i].w);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc2 += __shfl_xor_sync(0xFFFFFFFFu, acc2, o);
                if (lane == 0) sq[warp * kGemvMaxM + m] = acc2;
            }
            __syncthreads();   // every warp of the CTA runs this set-up
        }
        // The single-token records are built straight from x in global memory (no tensor copy and
        // barrier round trip; measured 1.8-3.6% faster per call for Q4_K). The general kernel's
        // permute pass reading x from global memory instead of the copied tile measured slower
        // (4096x4096: 4.78 -> 5.21 us), so it keeps the copy, as do the fused prologues.
        constexpr bool M1_DIRECT = M1 && !PRO;
        if constexpr (!PRO && !M1_DIRECT) {
            if (nmine > 0 && lane == 0) {   // this warp's x slice, all tokens, once
                mbar_arrive_expect_tx(xbar, p.x_tx);
                tma_load_3d(xreg, &xmap, 0, kb0 * 4, 0, xbar);
            }
            if (nmine > 0) ok = mbar_wait(xbar, 0);
        }
        if constexpr ((PERM || PRO) && !M1) {
            // One pass over the warp's x tile: fill it (fused prologue), permute it in place
            // [x0 x1 x2 x3] -> [x0 x2 x1 x3] inside every 16-byte chunk (K-quants, Q6_K) and,
            // for the K-quants, store the sums of x over each 32-wide sub-block. The tile is
            // 128-byte rows r = token * 4 kw + 4 * superblock + segment with chunk c of a row
            // stored at c ^ (r & 7); that swizzle keeps each aligned group of four chunks (one
            // sub-block) together, so four neighbouring lanes hold one sub-block and two shuffles
            // sum it. x_tx / 16 is a multiple of 32: every lane runs every pass.
            auto put = [&](uint32_t q, const uint4 &v) {   // store chunk q (k order) permuted, add its sums
                if constexpr (PERM)
                    sts128(xreg + 16u * q, make_uint4(prmt(v.x, v.y, 0x5410u), prmt(v.x, v.y, 0x7632u),
                                                      prmt(v.z, v.w, 0x5410u), prmt(v.z, v.w, 0x7632u)));
                else
                    sts128(xreg + 16u * q, v);
                if constexpr (XSUM) {
                    const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
                    const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
                    const float2 f2 = __half22float2(*reinterpret_cast<const __half2 *>(&v.z));
                    const float2 f3 = __half22float2(*reinterpret_cast<const __half2 *>(&v.w));
                    float sum = ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
                    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
                    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
                    if ((q & 3u) == 0u) {
                        const uint32_t r = q >> 3, half = ((q & 7u) ^ (r & 7u)) >> 2;   // sub-block 2 (r & 3) + half
                        const __half hi = __float2half_rn(sum);
                        const __half lo = __float2half_rn(sum - __half2float(hi));
                        __half *rec = reinterpret_cast<__half *>(gbase + (xsum_base - base) + (r >> 2) * 32u + 8u * (r & 3u));
                        rec[half] = hi;
                        rec[2 + half] = lo;
                    }
                }
            };
            const uint32_t nq = p.x_tx / 16u;
            if constexpr (!PRO) {
                for (uint32_t q = lane; q < nq; q += 32) put(q, lds128(xreg + 16u * q));
            } else {
                // chunk q holds columns k0 .. k0+7 of token tokq (the tile's swizzle undone)
                const uint32_t xrows_tok = 4u * static_cast<uint32_t>(p.kw);
                auto chunk_pos = [&](uint32_t q, uint32_t &tokq) {
                    const uint32_t r = q >> 3;
                    tokq = r / xrows_tok;
                    const uint32_t seg = r - tokq * xrows_tok;
                    return (static_cast<int64_t>(kb0) * 4 + seg) * 64 + 8 * ((q & 7u) ^ (r & 7u));
                };
                for (uint32_t q0 = lane; q0 < nq; q0 += 32u * kFillGroup) {   // nq is a multiple of 32: uniform
                    ChunkIn in[kFillGroup];
#pragma unroll
                    for (int i = 0; i < kFillGroup; ++i) {
                        uint32_t tokq;
                        const uint32_t q = q0 + 32u * i;
                        const int64_t k0 = chunk_pos(q, tokq);
                        if (q < nq && k0 < p.K) in[i] = chunk_load(p, static_cast<int>(tokq), k0);
                    }
#pragma unroll
                    for (int i = 0; i < kFillGroup; ++i) {
                        uint32_t tokq;
                        const uint32_t q = q0 + 32u * i;
                        if (q >= nq) break;
                        const int64_t k0 = chunk_pos(q, tokq);
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);   // columns beyond K (a partial last slice)
                        if (k0 < p.K) {
                            float rstd = 0.f;
                            if (p.pro == 2) {
                                float tot = 0.f;
                                for (int w2 = 0; w2 < static_cast<int>(blockDim.x >> 5); ++w2) tot += sq[w2 * kGemvMaxM + tokq];
                                rstd = rsqrtf(tot / static_cast<float>(p.K) + p.eps);
                            }
                            v = chunk_compute(p, in[i], rstd);
                            if (p.pro == 2 && p.xnorm && b == 0 && tg == 0)   // one writer per element
                                *reinterpret_cast<uint4 *>(p.xnorm + static_cast<int64_t>(tokq) * p.K + k0) = v;
                        }
                        put(q, v);
                    }
                }
            }
            __syncwarp();
        }
        if constexpr (M1) {   // the staged B records, built without an x tile
            if constexpr (M1_DIRECT) {
                if (nmine > 0) {
                    if constexpr (TYPE == 23) m1_stage_iq4_global(p.x, kb0, p.nsb, xexp, p.kw, lane);
                    else m1_stage_global(p.x, kb0, p.nsb, xexp, xsums, p.kw, lane, p.qswap);
                }
            } else if (nmine > 0) {
                // fused prologue: lane l computes the 8 activations of chunk l of each superblock
                // (loads of kFillGroup superblocks issued first) and lays them out as the plain
                // staging does, with the sub-block sums added in the same order
                float rstd = 0.f;
                if (p.pro == 2) {
                    float tot = 0.f;
                    for (int w2 = 0; w2 < static_cast<int>(blockDim.x >> 5); ++w2) tot += sq[w2 * kGemvMaxM];
                    rstd = rsqrtf(tot / static_cast<float>(p.K) + p.eps);
                }
                for (int b0 = 0; b0 < p.kw; b0 += kFillGroup) {
                    ChunkIn in[kFillGroup];
#pragma unroll
                    for (int i = 0; i < kFillGroup; ++i) {
                        const int64_t k0 = static_cast<int64_t>(kb0 + b0 + i) * 256 + 8 * lane;
                        if (b0 + i < p.kw && k0 < p.K) in[i] = chunk_load(p, 0, k0);
                    }
#pragma unroll
                    for (int i = 0; i < kFillGroup; ++i) {
                        if (b0 + i >= p.kw) break;   // warp-uniform
                        const int64_t k0 = static_cast<int64_t>(kb0 + b0 + i) * 256 + 8 * lane;
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);   // superblocks past nsb
                        if (k0 < p.K) {
                            v = chunk_compute(p, in[i], rstd);
                            if (p.pro == 2 && p.xnorm && b == 0 && tg == 0)   // one writer per element
                                *reinterpret_cast<uint4 *>(p.xnorm + k0) = v;
                        }
                        if constexpr (TYPE == 23) m1_stage_iq4_chunk(v, b0 + i, xexp, lane);
                        else m1_stage_chunk(v, b0 + i, xexp, xsums, lane, p.qswap);
                    }
                }
            }
            __syncwarp();
        }
    } else {
        pdl_wait();
        for (int s = 0; s < D && s < total; ++s) issue_next(s);
    }
    

    const uint32_t tok = static_cast<uint32_t>(min(g, p.M - 1));
    const uint32_t xrows = XRES ? 4u * p.kw : 4u * S;   // x rows per token in its tile
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float acc1[2] = {0.f, 0.f};   // M1: rows g, g+8 over this lane's sub-blocks
    int u = 0, s = 0, jt = 0;   // stage counter, ring slot, my tile counter
    uint32_t ph = 0;
    for (int round0 = 0; round0 < ntiles; round0 += p.round_tiles) {
      const int rend = min(round0 + p.round_tiles, ntiles);
      for (; tg + jt * p.tgc < rend; ++jt) {
        const int t = tg + jt * p.tgc;
        int jp;
        const int row0 = tile_rows(t, jp);
        const int ra = min(row0 + g, p.N[jp] - 1), rb = min(row0 + g + 8, p.N[jp] - 1);
        for (int si = 0; si < nst; ++si, ++u) {
            if (ok && !mbar_wait(bar0 + 8 * s, ph)) ok = false;
            if (ok) {
                const uint32_t wst = wslot(s);
                const uint32_t xst = XRES ? xreg : xslot(s);
                const int sb0 = kb0 + si * S;
                const int ns = min(S, kb1 - sb0);
                const uint32_t xsb0 = XRES ? static_cast<uint32_t>(si * S) : 0u;   // x superblock index base
                uint32_t base_a = wst + g * p.row_pitch, base_b = wst + (g + 8) * p.row_pitch;
                if constexpr (!TMA) {   // block data starts (o & 15) bytes into the row's window; unsigned
                    // arithmetic wraps modulo 2^32, which keeps the low four bits of the byte offset
                    const uint32_t nsb = static_cast<uint32_t>(p.nsb), sbu = static_cast<uint32_t>(sb0);
                    base_a += ((static_cast<uint32_t>(ra) * nsb + sbu) * static_cast<uint32_t>(BB)) & 15u;
                    base_b += ((static_cast<uint32_t>(rb) * nsb + sbu) * static_cast<uint32_t>(BB)) & 15u;
                }
                // the stage's blocks inside its slot; the x it pairs with inside this warp's x region
                const uint32_t span = static_cast<uint32_t>(ns) * BB, xsbe = xsb0 + static_cast<uint32_t>(ns);
                const uint32_t x_end = M1 ? xexp + xsbe * kM1Sb : xst + (tok * xrows + 4u * xsbe) * 128u;
                const uint32_t x_lim = XRES ? xreg + p.x_tx : xst + p.x_bytes;
                const bool stage_ok = in_bounds(ns >= 1 && base_b + span <= wst + p.w_bytes && base_a + span <= wst + p.w_bytes &&
                                                    (M1 ? x_end <= xsums && (TYPE == 23 || xsums + 32u * xsbe <= xreg + p.x_warp_bytes)
                                                        : x_end <= x_lim),
                                                p.status);
                if (!stage_ok) {
                } else if constexpr (M1 && TYPE == 23) {
                    // B of column g when this lane carries it at steps 0-3 (column 2c for c < 2, 2c+1
                    // for c >= 2: the chunk order i ^ c swaps the halves) or steps 4-7 (the other)
                    const int ja = 2 * c + (c >= 2 ? 1 : 0), jb = 2 * c + (c >= 2 ? 0 : 1);
                    const uint32_t slot_lo = (g == ja) ? 8u * g : 64u, slot_hi = (g == jb) ? 8u * g : 64u;
                    const uint32_t lutl = base + p.lut_offset + 4u * static_cast<uint32_t>(lane);
#pragma unroll 2
                    for (int j = 0; j < ns; ++j) {
                        const uint32_t rb = xexp + (xsb0 + j) * kM1Sb;
                        superblock_iq4_m1(base_a + j * BB, base_b + j * BB, rb + slot_lo, rb + slot_hi, lutl, c, acc1);
                    }
                } else if constexpr (M1) {
                    const uint32_t slot = ((g >> 1) == c) ? 8u * g : 64u;   // B of column g, or the zero slot
                    const uint32_t swap16 = (p.qswap && (c & 1)) ? 16u : 0u;
#pragma unroll 2
                    for (int j = 0; j < ns; ++j) {
                        const uint32_t b = xsb0 + j;
                        superblock_kq_m1<TYPE>(base_a + j * BB, base_b + j * BB, xexp + b * kM1Sb + slot,
                                               xsums + 32u * b, c, swap16, acc1);
                    }
                } else {
#pragma unroll 2   // two superblocks' independent decode chains can interleave
                    for (int j = 0; j < ns; ++j) {
                        const uint32_t blk_a = base_a + j * BB, blk_b = base_b + j * BB;
                        const uint32_t r0 = tok * xrows + 4u * (xsb0 + j);   // x row of segment 0
                        if constexpr (TYPE == 12 || TYPE == 13)
                            superblock_kq<TYPE, PERM, XSUM>(blk_a, blk_b, xrow(xst, r0 + c), c, acc,
                                                            xsum_base + (tok * p.kw + xsb0 + j) * 32u);
                        else if constexpr (TYPE == 14 || TYPE == kQ6KAligned)
                            superblock_q6<PERM, TYPE == kQ6KAligned>(blk_a, blk_b, xst, r0, c, acc);
                        else superblock_iq4(blk_a, blk_b, xrow(xst, r0 + c), c, acc);
                    }
                }
            }
            // Refill the slot. Its previous contents were read by this warp's ordinary loads,
            // all consumed above (and kept ahead of the copy issue by its memory clobber), so
            // the write-after-read needs no proxy fence.
            __syncwarp();
            if (ok && u + D < total) issue_next(s);
            if (++s == D) {
                s = 0;
                ph ^= 1u;
            }
        }
        // This warp's partial of tile t goes to its slot of the current round (tokens < M only);
        // warps run on without waiting for each other.
        float *pt = red + ((t - round0) * p.ks + kidx) * 16 * p.M;
        if (!in_bounds(t - round0 < p.round_tiles && kidx < p.ks &&
                           p.red_offset + 4u * static_cast<uint32_t>(((t - round0 + 1) * p.ks) * 16 * p.M) <= p.x_offset,
                       p.status))
            pt = nullptr;   // bounds check failed: the partial is not stored
        if (!pt) {
            acc1[0] = acc1[1] = 0.f;
        } else if constexpr (M1) {   // the four lanes of a row group hold its four sub-block pairs
            float a0 = acc1[0], a1 = acc1[1];
            a0 += __shfl_xor_sync(0xFFFFFFFFu, a0, 1);
            a1 += __shfl_xor_sync(0xFFFFFFFFu, a1, 1);
            a0 += __shfl_xor_sync(0xFFFFFFFFu, a0, 2);
            a1 += __shfl_xor_sync(0xFFFFFFFFu, a1, 2);
            if (c == 0) {
                pt[g] = a0;
                pt[g + 8] = a1;
            }
            acc1[0] = acc1[1] = 0.f;
        } else if (2 * c < p.M) {
            pt[2 * c * 16 + g] = acc[0];
            pt[2 * c * 16 + g + 8] = acc[2];
        }
        if (pt && 2 * c + 1 < p.M) {
            pt[(2 * c + 1) * 16 + g] = acc[1];
            pt[(2 * c + 1) * 16 + g + 8] = acc[3];
        }
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
      }
      // end of the round: each tile's partials summed over its K slices in fixed order
      __syncthreads();
      const int per_tile = 16 * p.M;
      if constexpr (ARGMAX) {
          // greedy head: per token, the CTA's best (value, row) key, then one atomic max;
          // each value is summed exactly as the y path sums it
          unsigned long long *wbest = reinterpret_cast<unsigned long long *>(
              gbase + scratch_offset(blockDim.x >> 5, D) + 4u * 16u * kGemvMaxM);
          for (int m = 0; m < p.M; ++m) {
              unsigned long long bk = 0ull;
              for (int q = threadIdx.x; q < (rend - round0) * 16; q += blockDim.x) {
                  const int tt = q >> 4;
                  const float *src = red + tt * p.ks * per_tile + m * 16 + (q & 15);
                  float sum = 0.f;
                  for (int kk = 0; kk < p.ks; ++kk) sum += src[kk * per_tile];
                  int jp;
                  const int row = tile_rows(round0 + tt, jp) + (q & 15);
                  if (row < p.N[0]) bk = max(bk, argmax_key(sum, row));
              }
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) bk = max(bk, __shfl_xor_sync(0xFFFFFFFFu, bk, o));
              if (lane == 0) wbest[warp] = bk;
              __syncthreads();
              if (threadIdx.x == 0) {
                  unsigned long long cb = 0ull;
                  for (int w2 = 0; w2 < static_cast<int>(blockDim.x >> 5); ++w2) cb = max(cb, wbest[w2]);
                  atomicMax(p.best + m, cb);
              }
              __syncthreads();
          }
      } else {
          for (int q = threadIdx.x; q < (rend - round0) * per_tile; q += blockDim.x) {
              const int tt = q / per_tile, rem = q - tt * per_tile;   // tile of the round, token * 16 + row
              const float *src = red + tt * p.ks * per_tile + rem;
              float sum = 0.f;
              for (int kk = 0; kk < p.ks; ++kk) sum += src[kk * per_tile];
              int jp;
              const int row = tile_rows(round0 + tt, jp) + (rem & 15);
              if (row < p.N[jp]) {
                  const int64_t o = static_cast<int64_t>(rem >> 4) * p.N[jp] + row;
                  if constexpr (PRO) p.y[jp][o] = p.residual ? sum + p.residual[o] : sum;   // y may be the residual
                  else p.y[jp][o] = sum;
              }
          }
      }
      if (rend < ntiles) __syncthreads();   // the next round reuses the slots
    }
    if (!ok) {
        if (lane == 0) atomicOr(p.status, kStatusTimeout);
        // let copies still in flight land before the shared memory is released
        for (int j = u; j < total && j < u + D; ++j) (void)mbar_wait(bar0 + 8 * (j % D), (j / D) & 1);
    }
}

// ---------------------------------------------------------------- host side

struct GemvPlan {
    GemvArgs a;
    bool tma;
    int warps, grid;
    size_t smem;
};

// T: 16-row tiles over all projections. need_xres: only plans with x resident per warp (the
// fused prologues fill that tile). m1: the single-token K-quant kernel, whose resident x region
// also holds the staged B records (1 KB per superblock), a zero block and the sub-block sums.
GemvPlan make_plan(int type, int64_t T, int64_t K, int M, int num_sms, bool need_xres, bool m1) {
    GemvPlan pl{};
    GemvArgs &a = pl.a;
    const int bb = block_bytes_of(type);
    const int nsb = static_cast<int>(K / 256);
    const int64_t row_bytes = static_cast<int64_t>(nsb) * bb;
    // 2-D tensor copies need 16-byte row strides and box widths; IQ4_XS stages hold an even
    // number of 136-byte blocks.
    const int s_mult = (type == 23) ? 2 : 1;
    pl.tma = (row_bytes % 16 == 0) && type != 14 && (type != 23 || nsb % 2 == 0);
    const int s_max = pl.tma ? std::max(s_mult, (2048 / bb) / s_mult * s_mult) : 8;   // <= 2 KB per row
    auto pitch_of = [&](int S) {
        if (pl.tma) return static_cast<uint32_t>(S * bb);   // dense rows as the tensor copy lands them
        uint32_t pitch = static_cast<uint32_t>((S * bb + 30) & ~15);   // window incl. misalignment
        if ((pitch / 16) % 2 == 0) pitch += 16;                         // odd multiple of 16
        return pitch;
    };
    const size_t limit = 227 * 1024;
    // grid: one CTA per SM (persistent), each owning up to tmax 16-row tiles
    pl.grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(num_sms, T)));
    const int tmax = static_cast<int>((T + pl.grid - 1) / pl.grid);
    // Up to maxw warps = ks K slices (of kw superblocks, a multiple of s_mult) x tgc tile groups.
    // Candidates are ranked by the busiest warp's work, kw * ceil(tmax / tgc) superblocks,
    // then by more warps, then by fewer tile groups (less duplicated x).
    struct Cand { int kw, ks, tgc, cost; };
    const int maxw = gemv_max_warps(type);
    Cand cands[32 * 32];
    int nc = 0;
    for (int want = 1; want <= maxw; ++want) {
        int kw_ = (nsb + want - 1) / want;
        kw_ = (kw_ + s_mult - 1) / s_mult * s_mult;
        const int ks_ = (nsb + kw_ - 1) / kw_;
        if (ks_ != want) continue;   // same split as a smaller count
        for (int tgc_ = 1; ks_ * tgc_ <= maxw && tgc_ <= tmax; ++tgc_)
            cands[nc++] = Cand{kw_, ks_, tgc_, kw_ * ((tmax + tgc_ - 1) / tgc_)};
    }
    std::sort(cands, cands + nc, [](const Cand &x, const Cand &y) {
        if (x.cost != y.cost) return x.cost < y.cost;
        if (x.ks * x.tgc != y.ks * y.tgc) return x.ks * x.tgc > y.ks * y.tgc;
        return x.tgc < y.tgc;
    });
    int kw = 0, ks = 0, tgc = 0, w = 0, round_tiles = 1;
    auto layout = [&](bool xres, int S, int D, GemvArgs &o) {
        o.S = S;
        o.stages = D;
        o.row_pitch = pitch_of(S);
        o.w_bytes = 16 * o.row_pitch;
        o.x_tx = static_cast<uint32_t>(M * (xres ? kw : S) * 512);
        o.x_bytes = xres ? 0u : o.x_tx;
        const uint32_t xsum_bytes = (type == 12 || type == 13) ? static_cast<uint32_t>(M * kw * 32) : 0u;
        const uint32_t m1_bytes = m1 ? static_cast<uint32_t>(kw * (16 * 72) + (type == 23 ? 0 : kw * 32)) : 0u;
        // the single-token kernels build their records without an x tile
        o.x_warp_bytes = xres ? (((m1 ? 0u : o.x_tx) + (m1 ? m1_bytes : xsum_bytes) + 1023u) & ~1023u) : 0u;
        // a slot that also holds a 128-byte-swizzled x tile starts on 1 KB, weights alone on 128 B
        o.slot_bytes = xres ? ((o.w_bytes + 127u) & ~127u) : ((o.x_bytes + o.w_bytes + 1023u) & ~1023u);
        o.xres = xres ? 1 : 0;
        const uint32_t bars = (scratch_offset(w, D) + kScratchBytes + 1023u) & ~1023u;
        o.red_offset = bars;
        o.round_tiles = round_tiles;
        o.lut_offset = (bars + static_cast<uint32_t>(round_tiles * ks * 16 * M * sizeof(float)) + 1023u) & ~1023u;
        const uint32_t lut_bytes = (m1 && type == 23) ? kIq4LutBytes : 0u;
        o.x_offset = o.lut_offset + lut_bytes;
        o.ring_offset = o.x_offset + w * o.x_warp_bytes;
        return static_cast<size_t>(1024) + o.ring_offset + static_cast<size_t>(w) * D * o.slot_bytes;
    };
    size_t smem = 0;
    bool found = false;
    for (int ci = 0; ci < nc && !found; ++ci) {
        kw = cands[ci].kw;
        ks = cands[ci].ks;
        tgc = cands[ci].tgc;
        w = ks * tgc;
        // partials of up to round_tiles tiles (16 KB of shared memory) are reduced per round
        round_tiles = std::max(1, std::min(tmax, (16 * 1024) / (ks * 16 * M * 4)));
        for (int xres = 1; xres >= (need_xres || m1 ? 1 : 0) && !found; --xres) {
            for (int S = std::min(kw, s_max); S >= s_mult && !found; S -= s_mult) {
                const int nst = (kw + S - 1) / S;
                for (int D = std::min(4, std::max(2, 2 * nst)); D >= 2 && !found; --D) {
                    smem = layout(xres == 1, S, D, a);
                    found = smem <= limit;
                }
            }
        }
    }
    if (!found) {
        pl.smem = SIZE_MAX;
        return pl;
    }
    a.K = static_cast<int>(K);
    a.m1 = m1 ? 1 : 0;
    {
        const uint32_t delta = (a.row_pitch % 128u) / 16u;   // bank-group shift from row g to row g + 1
        a.qswap = (m1 && (type == 12 || type == 13) && (delta == 2u || delta == 6u)) ? 1 : 0;
    }
    a.M = M;
    a.nsb = nsb;
    a.kw = kw;
    a.ks = ks;
    a.tgc = tgc;
    pl.warps = w;
    // Ask for more than half of an SM's shared memory even when the plan needs less: the
    // partition assumes one CTA per SM, and two CTAs doubled up on one SM (which the block
    // scheduler otherwise does when they fit) run at half speed and stretch the launch's tail
    // (measured: the 8B-layer decode sequence 32.5 -> 27.4 us per step).
    pl.smem = std::max<size_t>(smem, 116 * 1024);
    return pl;
}

template <int TYPE, bool TMA, bool XRES, bool MULTI, bool PRO = false, bool ARGMAX = false, bool M1 = false>
cudaError_t launch_t(const GemvMaps &wm, const CUtensorMap &xm, const GemvArgs &a, int grid, int threads,
                     size_t smem, bool pdl, cudaStream_t st) {
    auto kern = gemv_kernel<TYPE, TMA, XRES, MULTI, PRO, ARGMAX, M1>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    void *args[] = {const_cast<GemvMaps *>(&wm), const_cast<CUtensorMap *>(&xm), const_cast<GemvArgs *>(&a)};
    return launch_pdl(reinterpret_cast<const void *>(kern), dim3(grid), dim3(threads), smem, st, pdl, args);
}

template <int TYPE>
cudaError_t launch_type(bool tma, bool xres, const GemvMaps &wm, const CUtensorMap &xm, const GemvArgs &a,
                        int grid, int threads, size_t smem, bool pdl, cudaStream_t st) {
    if constexpr (TYPE == 12 || TYPE == 13 || TYPE == 23) {
        if (a.m1) {   // single token, x resident and rows copied by 2-D tensor copies
            if (!xres || !tma) return cudaErrorInvalidValue;
            if (a.best) return launch_t<TYPE, true, true, false, false, true, true>(wm, xm, a, grid, threads, smem, pdl, st);
            if (a.pro != 0) return launch_t<TYPE, true, true, false, true, false, true>(wm, xm, a, grid, threads, smem, pdl, st);
            if (a.nproj > 1) return launch_t<TYPE, true, true, true, false, false, true>(wm, xm, a, grid, threads, smem, pdl, st);
            return launch_t<TYPE, true, true, false, false, false, true>(wm, xm, a, grid, threads, smem, pdl, st);
        }
    }
    if (a.best) {   // greedy head: one projection, x resident (the plan guarantees it)
        if (a.nproj != 1 || !xres || a.pro != 0) return cudaErrorInvalidValue;
        return tma ? launch_t<TYPE, true, true, false, false, true>(wm, xm, a, grid, threads, smem, pdl, st)
                   : launch_t<TYPE, false, true, false, false, true>(wm, xm, a, grid, threads, smem, pdl, st);
    }
    if (a.pro != 0) {   // fused prologues: one projection, x resident (the plan guarantees it)
        if (a.nproj != 1 || !xres) return cudaErrorInvalidValue;
        return tma ? launch_t<TYPE, true, true, false, true>(wm, xm, a, grid, threads, smem, pdl, st)
                   : launch_t<TYPE, false, true, false, true>(wm, xm, a, grid, threads, smem, pdl, st);
    }
    if (a.nproj > 1) {
        if (tma) return xres ? launch_t<TYPE, true, true, true>(wm, xm, a, grid, threads, smem, pdl, st)
                             : launch_t<TYPE, true, false, true>(wm, xm, a, grid, threads, smem, pdl, st);
        return xres ? launch_t<TYPE, false, true, true>(wm, xm, a, grid, threads, smem, pdl, st)
                    : launch_t<TYPE, false, false, true>(wm, xm, a, grid, threads, smem, pdl, st);
    }
    if (tma) return xres ? launch_t<TYPE, true, true, false>(wm, xm, a, grid, threads, smem, pdl, st)
                         : launch_t<TYPE, true, false, false>(wm, xm, a, grid, threads, smem, pdl, st);
    return xres ? launch_t<TYPE, false, true, false>(wm, xm, a, grid, threads, smem, pdl, st)
                : launch_t<TYPE, false, false, false>(wm, xm, a, grid, threads, smem, pdl, st);
}

}  // namespace

namespace {

// QL_GEMV_M1_IQ4=0: IQ4_XS single tokens on the general kernel (A/B measurement).
bool iq4_single_token_off() {
    static const bool off = [] {
        const char *e = std::getenv("QL_GEMV_M1_IQ4");
        return e && e[0] == '0';
    }();
    return off;
}

// QL_GEMV_M1=0 selects the general kernel for single tokens as well (A/B measurement).
bool single_token_off() {
    static const bool off = [] {
        const char *e = std::getenv("QL_GEMV_M1");
        return e && e[0] == '0';
    }();
    return off;
}

cudaError_t launch_impl(int type, int nproj, const GemvProj *proj, const __half *x, int64_t K, int M,
                        const GemvFusion *fu, unsigned *status, int num_sms, bool pdl, cudaStream_t stream) {
    const int bb = block_bytes_of(type);
    if (bb < 0 || M < 1 || M > kGemvMaxM || nproj < 1 || nproj > kGemvMaxProj) return cudaErrorInvalidValue;
    const int pro = fu ? fu->pro : 0;
    const bool head = fu && fu->best;
    if (pro < 0 || pro > 2 || (fu && (fu->residual || fu->best) && nproj != 1) || (head && pro != 0))
        return cudaErrorInvalidValue;
    int tile0[kGemvMaxProj + 1];
    int64_t T = 0;
    for (int j = 0; j < nproj; ++j) {
        tile0[j] = static_cast<int>(T);
        T += (proj[j].N + 15) / 16;
        if (T > (int64_t(1) << 30)) return cudaErrorInvalidValue;
    }
    tile0[nproj] = static_cast<int>(T);
    // One token: the single-token kernel when its plan fits and each warp has at least 2
    // superblocks to decode. With its x staged straight from global memory it measured 1-2.5%
    // faster than the general kernel on K=4096 N=4096 and N=1024 and 2% slower on K=1024
    // N=1024 (one superblock per warp). The choice depends on the shape only, so a prologue or
    // the greedy head sums exactly as the plain call does.
    const int64_t grid = std::min<int64_t>(num_sms > 0 ? num_sms : 1, T);
    const int64_t per_warp = (T + grid - 1) / grid * ((K / 256 + 7) / 8);   // tiles per CTA x superblocks per slice of 8
    const bool m1_type = type == 12 || type == 13 || (type == 23 && (K / 256) % 2 == 0 && !iq4_single_token_off());
    bool m1 = M == 1 && m1_type && per_warp >= 2 && !single_token_off();
    GemvPlan pl = make_plan(type, T, K, M, num_sms, pro != 0 || head, m1);
    if (m1 && pl.smem > 227 * 1024) {
        m1 = false;
        pl = make_plan(type, T, K, M, num_sms, pro != 0 || head, false);
    }
    if (pl.smem > 227 * 1024) return cudaErrorNotSupported;
    const int64_t row_bytes = K / 256 * bb;
    for (int j = 0; j <= nproj; ++j) pl.a.tile0[j] = tile0[j];
    for (int j = 0; j < nproj; ++j) {
        pl.a.W[j] = proj[j].W;
        pl.a.y[j] = proj[j].y;
        pl.a.N[j] = static_cast<int>(proj[j].N);
        pl.a.total_bytes[j] = proj[j].N * row_bytes;
    }
    pl.a.nproj = nproj;
    pl.a.x = x;
    pl.a.status = status;
    if (fu) {
        pl.a.pro = pro;
        pl.a.gate = fu->gate;
        pl.a.up_or_h = fu->up_or_h;
        pl.a.norm_w = fu->norm_w;
        pl.a.eps = fu->eps;
        pl.a.xnorm = fu->xnorm;
        pl.a.residual = fu->residual;
        pl.a.best = fu->best;
    }
    GemvMaps wm{};
    CUtensorMap xm{};
    // x viewed as [M tokens][K/64 rows][64 halves]; one box = all tokens x (4 rows per
    // superblock of a warp slice or of a stage), 128-byte swizzled
    const uint32_t xbox_rows = static_cast<uint32_t>(4 * (pl.a.xres ? pl.a.kw : pl.a.S));
    if (pro == 0 && !encode_tmap_3d(&xm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, 64, static_cast<uint64_t>(K / 64),
                                    static_cast<uint64_t>(M), 128, static_cast<uint64_t>(K) * 2, 64, xbox_rows,
                                    static_cast<uint32_t>(M), true))
        return cudaErrorInvalidValue;
    if (pl.tma) {   // W[j] viewed as [N rows][row bytes / 8] of 8-byte elements
        const uint64_t row_elems = static_cast<uint64_t>(row_bytes) / 8;
        for (int j = 0; j < nproj; ++j)
            if (!encode_tmap_2d(&wm.m[j], CU_TENSOR_MAP_DATA_TYPE_UINT64, proj[j].W, row_elems,
                                static_cast<uint64_t>(proj[j].N), row_elems * 8, static_cast<uint32_t>(pl.a.S * bb / 8),
                                16, false))
                return cudaErrorInvalidValue;
    }
    const int threads = 32 * pl.warps;
    switch (type) {
    case 12: return launch_type<12>(pl.tma, pl.a.xres != 0, wm, xm, pl.a, pl.grid, threads, pl.smem, pdl, stream);
    case 13: return launch_type<13>(pl.tma, pl.a.xres != 0, wm, xm, pl.a, pl.grid, threads, pl.smem, pdl, stream);
    case 14: return launch_type<14>(pl.tma, pl.a.xres != 0, wm, xm, pl.a, pl.grid, threads, pl.smem, pdl, stream);
    case kQ6KAligned:
        return launch_type<kQ6KAligned>(pl.tma, pl.a.xres != 0, wm, xm, pl.a, pl.grid, threads, pl.smem, pdl, stream);
    case 23: return launch_type<23>(pl.tma, pl.a.xres != 0, wm, xm, pl.a, pl.grid, threads, pl.smem, pdl, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t gemv_launch_multi(int type, int nproj, const GemvProj *proj, const __half *x, int64_t K, int M,
                              unsigned *status, int num_sms, bool pdl, cudaStream_t stream) {
    return launch_impl(type, nproj, proj, x, K, M, nullptr, status, num_sms, pdl, stream);
}

namespace {
// QL_GEMV_STREAM=0 keeps single-matrix decode calls on the persistent kernel (A/B measurement).
// The streaming kernel (gemv_stream.cu) runs plain calls only when QL_GEMV_STREAM=1: measured on
// GB300 it is slower than this kernel on every decode shape so far.
bool stream_kernel_off() {
    static const bool off = [] {
        const char *e = std::getenv("QL_GEMV_STREAM");
        return !(e && e[0] == '1');
    }();
    return off;
}
}  // namespace

cudaError_t gemv_launch(int type, const uint8_t *W, const __half *x, float *y, int64_t N, int64_t K, int M,
                        unsigned *status, int num_sms, bool pdl, cudaStream_t stream) {
    if (!stream_kernel_off()) {
        const cudaError_t e = gemv_stream_launch(type, W, x, y, N, K, M, status, num_sms, pdl, stream);
        if (e != cudaErrorNotSupported) return e;
    }
    const GemvProj one{W, y, N};
    return launch_impl(type, 1, &one, x, K, M, nullptr, status, num_sms, pdl, stream);
}

cudaError_t gemv_launch_fused(int type, const uint8_t *W, float *y, int64_t N, int64_t K, int M, const GemvFusion &f,
                              unsigned *status, int num_sms, bool pdl, cudaStream_t stream) {
    const GemvProj one{W, y, N};
    return launch_impl(type, 1, &one, nullptr, K, M, &f, status, num_sms, pdl, stream);
}

namespace {

// Packed keys -> row (in place, as int64) and value.
__global__ void argmax_finalize_kernel(unsigned long long *keys, float *val, int M) {
    const int m = threadIdx.x;
    if (m < M) {
        const unsigned long long k = keys[m];
        const uint32_t ord = static_cast<uint32_t>(k >> 32);
        const uint32_t bits = (ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord;
        if (val) val[m] = __uint_as_float(bits);
        reinterpret_cast<long long *>(keys)[m] = static_cast<long long>(0xFFFFFFFFu - static_cast<uint32_t>(k));
    }
}

}  // namespace

cudaError_t gemv_launch_argmax(int type, const uint8_t *W, int64_t N, int64_t K, const __half *x, int M,
                               long long *index_out, float *value_out, unsigned *status, int num_sms, cudaStream_t stream) {
    if (M < 1 || M > kGemvMaxM) return cudaErrorInvalidValue;
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(index_out);
    cudaError_t e = cudaMemsetAsync(keys, 0, static_cast<size_t>(M) * sizeof(unsigned long long), stream);
    if (e != cudaSuccess) return e;
    GemvFusion f;
    f.best = keys;
    const GemvProj one{W, nullptr, N};
    // launched in full stream order (no early start): the keys must be zero before any atomic
    e = launch_impl(type, 1, &one, x, K, M, &f, status, num_sms, false, stream);
    if (e != cudaSuccess) return e;
    argmax_finalize_kernel<<<1, 32, 0, stream>>>(keys, value_out, M);
    return cudaGetLastError();
}

}  // namespace ql
