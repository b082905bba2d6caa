// gemv_stream.cu -- decode-path quantized linear y[M, N] = x[M, K] . dequant(W)[N, K]^T for one
// weight matrix, built around how HBM is kept busy across back-to-back launches.
//
// Work split (sm_103a, one CTA per SM):
//  * CTA b owns rows [N b / G, N (b+1) / G): every CTA moves the same number of weight bytes
//    (to within one row). The rows are cut into 16-row tiles (the MMA's m); the last tile of a
//    CTA may be partial.
//  * A work unit is (tile, K range); warp w takes units w, w + NW, ... . A unit is fetched in
//    chunks of C superblocks: one 2-D tensor copy of 16 rows x C superblocks per chunk,
//    completing on the chunk buffer's barrier; a partial tile, and formats whose rows are not
//    16-byte multiples, take one bulk copy per row (over the 16-byte aligned window of the span).
//    A warp's chunks are issued in order, so it decodes a chunk while its later chunks are still
//    in flight.
//  * Each warp owns a ring of D chunk buffers. When D covers all of its chunks (the CTA's whole
//    share fits in shared memory) every weight byte of the launch is requested before the
//    kernel waits for the preceding kernel; otherwise buffers are refilled as they are consumed.
//    Measured on GB300 with a copy-only skeleton of this scheme, back-to-back launches of the
//    K=4096 N=12288 Q4_K layer stream at 0.94 of the measured HBM copy bandwidth. (Many small
//    copies do not: the copy engine accepts about one copy every 18 SM cycles.)
//  * x is brought in once per CTA after the wait by one tensor copy (128-byte swizzled rows),
//    then permuted in place and summed over 32-wide sub-blocks by all warps.
//  * A unit's result goes straight to y when the tile has one K range; otherwise the ranges'
//    partial sums meet in shared memory and are added in fixed order (deterministic).
//  * Bank conflicts: lane (g, c) reads the two 16-byte halves of 32-byte quant group c of rows g
//    and g + 8, and a warp's quarter holds rows g, g + 1. With the K-quants' 2-superblock chunks
//    the row pitch is 32 or 96 (mod 128) bytes, so rows g and g + 1 sit 2 or 6 bank groups apart;
//    lanes with odd c then read their halves in the other order (and pair them with the matching
//    x chunks: the k-slots a lane owns are the same for every row, so this is the same
//    contraction), which makes the quant, header and single-token x reads conflict-free.
//
// Single token with Q4_K / Q5_K: the MMA's eight n columns carry the superblock's eight 32-wide
// sub-blocks (column j holds x only at the k-slots of sub-block j), the quants enter as exact
// fp16 subnormals (a masked nibble read as fp16 bits is q 2^-24, the high nibble 16 q 2^-24) and
// scales/mins are applied once per sub-block in fp32. Only 8 of the 32 lanes hold a non-zero B
// value per MMA (lane (g, c) with g = 2c in b0, g = 2c + 1 in b1): each lane reads the x pair of
// column g from the staged x (one conflict-free shared-memory wavefront for the warp) and masks
// it into b0 or b1.
#include <algorithm>
#include <cstdint>
#include <cuda.h>

#include "decode.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace ql {

namespace {

constexpr int kGsMaxWarps = 16;
constexpr int kGsMaxD = 16;

template <int TYPE>
struct GsFmt;
// BB: bytes per block; MAXW: most warps for the single-token kernel (K-quants) and for the
// tokens-on-n kernel (register budgets: 16 warps allow 128 registers, 12 allow 168).
template <>
struct GsFmt<12> { static constexpr int BB = 144, MAXW = 12, MAXW_GEN = 12; };
template <>
struct GsFmt<13> { static constexpr int BB = 176, MAXW = 12, MAXW_GEN = 12; };
template <>
struct GsFmt<14> { static constexpr int BB = 210, MAXW = 8, MAXW_GEN = 8; };
template <>
struct GsFmt<kQ6KAligned> { static constexpr int BB = 224, MAXW = 8, MAXW_GEN = 8; };
template <>
struct GsFmt<23> { static constexpr int BB = 136, MAXW = 12, MAXW_GEN = 12; };

struct GsArgs {
    const uint8_t *W;
    const __half *x;
    float *y;
    unsigned *status;
    int64_t total_bytes;   // N * nsb * BB
    int N, K, M, nsb;
    int C;                 // superblocks per chunk
    int nchunk;            // chunks per row
    int ks;                // K ranges per tile
    int cpr;               // chunks per K range (the last range may hold fewer)
    int D;                 // ring depth (chunk buffers per warp)
    int tma;               // 1: full tiles by 2-D tensor copies, rows at pitch C * BB
    int swap;              // 1: lanes with odd c read their 32-byte quant groups as (second, first) half
    int xboxes;            // x tensor copies (boxes of up to 256 rows of 64 halves)
    uint32_t xbox_bytes;   // bytes one x copy delivers
    uint32_t pitch;        // bytes between rows inside a chunk buffer
    uint32_t xb_off;       // staged x (1 KB aligned); single token: its records, then the zero block
    uint32_t xs_off;       // sums of x over 32-wide sub-blocks (K-quants)
    uint32_t red_off;      // per (tile, K range) partials when ks > 1
    uint32_t wbuf_off[kGsMaxWarps + 1];   // warp w's ring starts at wbuf_off[w]
    uint32_t wbuf_rows[kGsMaxWarps];      // rows per chunk buffer of warp w (16, or the last tile's)
    uint32_t wslot[kGsMaxWarps];          // bytes per chunk buffer of warp w (128-byte multiple)
};

struct GsMaps {
    CUtensorMap w;   // W as [N rows][row bytes / 8] of 8-byte elements, box C * BB / 8 x 16 rows
    CUtensorMap x;   // x as [M][K / 64][64 halves], 128-byte swizzle
};

// ---------------------------------------------------------------- single-token K-quant superblock

// Single-token x records: for superblock sb, sub-block (column) j and quant word u of a 32-byte
// group, 16 bytes [d.b0, d.b1, e.b0, e.b1] = the B fragments the lane that carries column j feeds
// the two MMAs of word u: X02(u) = (x[32j + 4u], x[32j + 4u + 2]) pairs with the nibbles of quant
// bytes 0 and 2 (MMA d), X13(u) = (x[32j + 4u + 1], x[32j + 4u + 3]) with bytes 1 and 3 (MMA e);
// an even j (low nibbles) holds them in b0 and zero in b1, an odd j the reverse. The lanes that
// carry no column read a block of zeros, so no lane masks its B operand (the integer pipe is the
// decode's busiest). Columns are kM1RecPitch = 144 bytes (nine bank groups) apart and a column
// whose carrier reads its quant halves swapped stores its records in that order (position u
// holds word u ^ 4): the eight carriers' reads of one position fall in eight different bank
// groups (two wavefronts per warp read with the zero block).
constexpr uint32_t kM1RecPitch = 144;               // 8 records + 16 bytes
constexpr uint32_t kM1RecSb = 8 * kM1RecPitch;      // one superblock
constexpr uint32_t kM1ZeroBytes = 128;              // after the last superblock

// One superblock of rows g, g+8 (blk_a, blk_b) for the single-token path: acc[0] (row g) and acc[1]
// (row g+8) gain this lane's two sub-blocks 2c, 2c+1. rec = this lane's x records of this
// superblock (column g's when the lane carries it, else the zero block); sums = the superblock's
// eight fp32 sub-block sums of x. swap16: see the bank-conflict note.
template <int TYPE>
__device__ __forceinline__ void m1_superblock(uint32_t blk_a, uint32_t blk_b, uint32_t rec, uint32_t sums, int c,
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
    // Two accumulator chains (bytes 0, 2 and bytes 1, 3): measured on GB300, four chains and
    // moving the shifts to the multiply pipe were both slower.
    float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t rl = (4u - 2u * c) & 31u, rh = (7u - 2u * c) & 31u;   // Q5_K: bit 2c -> bit 4, 2c+1 -> bit 8
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint4 r = lds128(rec + 16u * u);
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
        mma16816(d, la02, lb02, ha02, hb02, r.x, r.y);
        mma16816(e, la13, lb13, ha13, hb13, r.z, r.w);
    }
    float d1[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) d1[j] = d[j] + e[j];
    // Scales and mins of sub-blocks 2c, 2c+1 from the 12-byte field (header words y, z, w): for
    // j < 4, sc = y.byte[j] & 63 and m = z.byte[j] & 63; for j >= 4, the low four bits come from
    // w.byte[j-4] (low / high nibble) and the top two from y.byte[j-4] / z.byte[j-4] >> 6. Lane c
    // needs byte pair 2c & 3 of each word: bring it to bytes 0, 1, then one shift-mask-or each.
    // The bytes become floats through 2^23 + b (exact) minus 2^23.
    const uint32_t pair_sel = (c & 1) ? 0x4432u : 0x4410u;
    const bool hi = c >= 2;
    const uint32_t sa = hi ? 2u : 0u, mA = hi ? 0x3030u : 0x3F3Fu, mC = hi ? 0x0F0Fu : 0u;
    auto scm = [&](const uint4 &h, float &s0, float &s1, float &m0, float &m1) {
        const uint32_t A = prmt(h.y, 0u, pair_sel), B = prmt(h.z, 0u, pair_sel), Cw = prmt(h.w, 0u, pair_sel);
        const uint32_t sc = and_or(A >> sa, mA, Cw & mC);
        const uint32_t mn = and_or(B >> sa, mA, (Cw >> 4) & mC);
        constexpr float k23 = 8388608.0f;
        s0 = __uint_as_float(prmt(sc, 0x4B000000u, 0x7440u)) - k23;
        s1 = __uint_as_float(prmt(sc, 0x4B000000u, 0x7441u)) - k23;
        m0 = __uint_as_float(prmt(mn, 0x4B000000u, 0x7440u)) - k23;
        m1 = __uint_as_float(prmt(mn, 0x4B000000u, 0x7441u)) - k23;
    };
    float sa0, sa1, ma0, ma1, sb0, sb1, mb0, mb1;
    scm(ha, sa0, sa1, ma0, ma1);
    scm(hb, sb0, sb1, mb0, mb1);
    const uint2 xs2 = lds64(sums + 8u * c);   // sums of x over sub-blocks 2c, 2c+1
    const float xs0 = __uint_as_float(xs2.x), xs1 = __uint_as_float(xs2.y);
    const float da = half_lo_to_float(ha.x), dma = half_hi_to_float(ha.x);
    const float db = half_lo_to_float(hb.x), dmb = half_hi_to_float(hb.x);
    constexpr float k24 = 16777216.0f, k20 = 1048576.0f;   // 2^24, 2^20
    acc[0] += da * (sa0 * k24 * d1[0] + sa1 * k20 * d1[1]) - dma * (ma0 * xs0 + ma1 * xs1);
    acc[1] += db * (sb0 * k24 * d1[2] + sb1 * k20 * d1[3]) - dmb * (mb0 * xs0 + mb1 * xs1);
}

// Single-token staging straight from global x (written by the preceding kernel, read through L2):
// thread q builds record q = (sb, j, u) from x[4q .. 4q+3], and the eight lanes of one (sb, j) sum
// its 32 values (fp32, fixed order) into sums[sb][j]. A thread issues all of its x loads before
// its first store, so the L2 latency is paid about once. swap: the plan's half swap (columns 2,
// 3, 6, 7 store their records in swapped order). Threads 0..7 also clear the zero block.
constexpr int kM1StageBatch = 8;   // records per thread per pass
__device__ __forceinline__ void stage_m1(const __half *x, int nsb, uint32_t recs, uint32_t sums, int swap) {
    const uint32_t nrec = static_cast<uint32_t>(nsb) * 64u;   // a multiple of 64: whole warps iterate together
    const uint2 *x8 = reinterpret_cast<const uint2 *>(x);
    if (threadIdx.x < kM1ZeroBytes / 16)
        sts128(recs + static_cast<uint32_t>(nsb) * kM1RecSb + 16u * threadIdx.x, make_uint4(0, 0, 0, 0));
    for (uint32_t q0 = threadIdx.x; q0 < nrec; q0 += kM1StageBatch * blockDim.x) {
        uint2 v[kM1StageBatch];
#pragma unroll
        for (int i = 0; i < kM1StageBatch; ++i) {
            const uint32_t q = q0 + static_cast<uint32_t>(i) * blockDim.x;
            v[i] = q < nrec ? __ldcg(x8 + q) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < kM1StageBatch; ++i) {
            const uint32_t q = q0 + static_cast<uint32_t>(i) * blockDim.x;
            if (q >= nrec) break;   // uniform across the warp
            const uint32_t sb = q >> 6, j = (q >> 3) & 7u, u = q & 7u;
            const uint32_t pos = u ^ ((swap && ((j >> 1) & 1u)) ? 4u : 0u);
            const uint32_t x02 = prmt(v[i].x, v[i].y, 0x5410u), x13 = prmt(v[i].x, v[i].y, 0x7632u);
            const uint4 rec = (j & 1u) ? make_uint4(0u, x02, 0u, x13) : make_uint4(x02, 0u, x13, 0u);
            sts128(recs + sb * kM1RecSb + j * kM1RecPitch + 16u * pos, rec);
            const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&v[i].x));
            const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&v[i].y));
            float sum = (f0.x + f0.y) + (f1.x + f1.y);
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 4);
            if (u == 0) sts32(sums + (sb * 8u + j) * 4u, __float_as_uint(sum));
        }
    }
}

// ---------------------------------------------------------------- x staging

// After the x tensor copy has landed: x[tok] is 128-byte rows r = tok * K/64 + k/64 with 16-byte
// chunk p of row r stored at p ^ (r & 7). One pass over the stored chunks permutes each chunk in
// place, [x0 x1 x2 x3] -> [x0 x2 x1 x3] per group of four (PERM), and sums x over every 32-wide
// sub-block: M1 as fp32 [superblock][8]; XSUM as 32-byte records [tok][superblock] holding, at
// 8 c, the (hi, hi, lo, lo) fp16 halves of the sums of sub-blocks 2c, 2c+1. The swizzle keeps a
// sub-block's four chunks in one aligned group of four stored chunks, so four neighbouring lanes
// hold one sub-block and two shuffles sum it. nchunks = M K / 8 is a multiple of 32.
template <bool PERM, bool M1SUM, bool XSUM>
__device__ __forceinline__ void stage_x(uint32_t xb, uint32_t xs, int M, int K) {
    const uint32_t rows_tok = static_cast<uint32_t>(K) / 64u;
    const uint32_t nchunks = static_cast<uint32_t>(M) * rows_tok * 8u;
    const uint32_t nsb = rows_tok / 4u;
    for (uint32_t q = threadIdx.x; q < nchunks; q += blockDim.x) {
        const uint32_t a = xb + 16u * q;
        const uint4 v = lds128(a);
        if constexpr (PERM)
            sts128(a, make_uint4(prmt(v.x, v.y, 0x5410u), prmt(v.x, v.y, 0x7632u), prmt(v.z, v.w, 0x5410u),
                                 prmt(v.z, v.w, 0x7632u)));
        if constexpr (M1SUM || XSUM) {
            const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
            const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
            const float2 f2 = __half22float2(*reinterpret_cast<const __half2 *>(&v.z));
            const float2 f3 = __half22float2(*reinterpret_cast<const __half2 *>(&v.w));
            float sum = ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
            if ((q & 3u) == 0u) {
                const uint32_t r = q >> 3;                           // stored row
                const uint32_t half = ((q & 7u) ^ (r & 7u)) >> 2;     // which 32-wide half of the row
                const uint32_t tok = r / rows_tok, rr = r - tok * rows_tok;
                const uint32_t sb = rr >> 2, j = 2u * (rr & 3u) + half;   // superblock, sub-block 0..7
                if constexpr (M1SUM) {
                    sts32(xs + (sb * 8u + j) * 4u, __float_as_uint(sum));
                } else {
                    const __half hi = __float2half_rn(sum);
                    const __half lo = __float2half_rn(sum - __half2float(hi));
                    const uint32_t rec = xs + (tok * nsb + sb) * 32u + 8u * (j >> 1) + 2u * (j & 1u);
                    asm volatile("st.shared.b16 [%0], %1;" ::"r"(rec), "h"(__half_as_ushort(hi)) : "memory");
                    asm volatile("st.shared.b16 [%0], %1;" ::"r"(rec + 4u), "h"(__half_as_ushort(lo)) : "memory");
                }
            }
        }
    }
}

// ---------------------------------------------------------------- the kernel

// Chunk cursor over a warp's units: unit u = w, w + NW, ...; chunk c of unit u in [c0(u), c1(u)).
struct Cursor {
    int u, c, c1;
};

template <int TYPE, bool M1, int MAXW>
__global__ void __launch_bounds__(32 * MAXW, 1) gemv_stream_kernel(const __grid_constant__ GsMaps maps,
                                                                   const __grid_constant__ GsArgs p) {
    constexpr int BB = GsFmt<TYPE>::BB;
    constexpr bool ALIGNED = (TYPE == 12 || TYPE == 13 || TYPE == kQ6KAligned);
    constexpr bool PERM = TYPE != 23;
    constexpr bool KQ = (TYPE == 12 || TYPE == 13);
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, NW = blockDim.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const uint32_t base = (smem_u32(smem) + 1023u) & ~1023u;   // the launch adds 1 KB of slack
    uint8_t *const gbase = smem + (base - smem_u32(smem));
    const uint32_t bar0 = base + 8u * kGsMaxD * warp;
    const uint32_t xbar = base + 8u * kGsMaxD * kGsMaxWarps;
    const uint32_t xb = base + p.xb_off, xs = base + p.xs_off;
    float *const red = reinterpret_cast<float *>(gbase + p.red_off);
    const uint32_t ring = base + p.wbuf_off[warp];
    const int brows = static_cast<int>(p.wbuf_rows[warp]);
    const uint32_t cbuf = p.wslot[warp];
    const int D = p.D;
    if constexpr (kBoundsChecks) {   // the whole layout inside the launch's dynamic shared memory
        uint32_t dyn;
        asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
        const uint32_t nsbu = static_cast<uint32_t>(p.nsb), mu = static_cast<uint32_t>(p.M);
        const uint32_t x_need = M1 ? nsbu * kM1RecSb + kM1ZeroBytes : static_cast<uint32_t>(p.xboxes) * p.xbox_bytes;
        const uint32_t s_need = M1 ? nsbu * 32u : (KQ ? mu * nsbu * 32u : 0u);
        const int ntile_cta = (static_cast<int>(static_cast<int64_t>(p.N) * (blockIdx.x + 1) / gridDim.x) -
                               static_cast<int>(static_cast<int64_t>(p.N) * blockIdx.x / gridDim.x) + 15) / 16;
        const uint32_t r_need = p.ks > 1 ? static_cast<uint32_t>(ntile_cta * p.ks) * mu * 64u : 0u;
        bool lay = base - smem_u32(smem) + p.wbuf_off[NW] <= dyn && NW <= kGsMaxWarps && D <= kGsMaxD && D >= 1 &&
                   x_need <= p.xs_off - p.xb_off && p.xs_off >= p.xb_off && x_need >= mu * static_cast<uint32_t>(p.K) * 2u &&
                   s_need <= p.red_off - p.xs_off && p.red_off >= p.xs_off && r_need <= p.wbuf_off[0] - p.red_off &&
                   p.wbuf_off[0] >= p.red_off && p.xb_off >= 8u * kGsMaxD * kGsMaxWarps + 8u;
        for (int w = 0; w < NW; ++w) lay = lay && p.wbuf_off[w + 1] >= p.wbuf_off[w] + static_cast<uint32_t>(D) * p.wslot[w];
        if (!in_bounds(lay, p.status)) return;
    }

    const int G = gridDim.x, b = blockIdx.x;
    const int r0 = static_cast<int>(static_cast<int64_t>(p.N) * b / G);
    const int r1 = static_cast<int>(static_cast<int64_t>(p.N) * (b + 1) / G);
    const int ntile = (r1 - r0 + 15) / 16;
    const int units = ntile * p.ks;

    if (lane == 0) {
        for (int s = 0; s < D; ++s) mbar_init(bar0 + 8 * s, 1);
        if (threadIdx.x == 0) mbar_init(xbar, 1);
        fence_mbar_init();
        if (!M1 && threadIdx.x == 0) prefetch_tmap(&maps.x);
        if (p.tma) prefetch_tmap(&maps.w);
    }
    // every warp waits on the x barrier that thread 0 initialised
    __syncthreads();

    auto unit_c0 = [&](int u) { return (u % p.ks) * p.cpr; };
    auto unit_c1 = [&](int u) { return min((u % p.ks + 1) * p.cpr, p.nchunk); };
    auto start = [&](Cursor &k) {
        k.u = warp;
        if (k.u < units) {
            k.c = unit_c0(k.u);
            k.c1 = unit_c1(k.u);
        }
    };
    auto advance = [&](Cursor &k) {
        if (++k.c == k.c1) {
            k.u += NW;
            if (k.u < units) {
                k.c = unit_c0(k.u);
                k.c1 = unit_c1(k.u);
            }
        }
    };

    const int64_t t16 = p.total_bytes & ~int64_t(15);
    // Fetch chunk (u, c) into ring slot s.
    auto issue = [&](int s, const Cursor &k) {
        const int t = k.u / p.ks;
        const int row0 = r0 + 16 * t, nrows = min(16, r1 - row0);
        const int sb0 = k.c * p.C;
        const uint32_t bar = bar0 + 8 * s, dst0 = ring + s * cbuf;
        if (p.tma && nrows == 16) {   // one tensor copy of the 16 rows
            if (lane == 0) {
                if (in_bounds(16u * p.pitch <= cbuf && row0 + 16 <= p.N && (sb0 + p.C) * BB <= p.nsb * BB &&
                                  dst0 + 16u * p.pitch <= ring + static_cast<uint32_t>(D) * cbuf,
                              p.status)) {
                    mbar_arrive_expect_tx(bar, 16u * p.pitch);
                    tma_load_2d(dst0, &maps.w, sb0 * (BB / 8), row0, bar);
                } else {
                    mbar_arrive(bar);
                }
            }
            return;
        }
        // one bulk copy per row over the 16-byte aligned window of the row's C superblocks;
        // bytes beyond the last 16-byte boundary of W, if any, are copied with plain loads
        const int ns = min(p.C, p.nsb - sb0);
        uint32_t nbytes = 0, dst = 0;
        const uint8_t *src = nullptr;
        if (lane < nrows) {
            const int64_t o = (static_cast<int64_t>(row0 + lane) * p.nsb + sb0) * BB;
            int64_t lo = o & ~int64_t(15), hi = (o + static_cast<int64_t>(ns) * BB + 15) & ~int64_t(15);
            const int64_t end = o + static_cast<int64_t>(ns) * BB;
            if (in_bounds(lo >= 0 && end <= p.total_bytes && lane < brows &&
                              (lane + 1) * p.pitch <= cbuf && static_cast<uint64_t>(hi - lo) <= p.pitch,
                          p.status)) {
                if (hi > t16) {   // the span ends in the last, partial 16 bytes of W
                    uint8_t *gd = gbase + (dst0 - base) + lane * p.pitch + (t16 - lo);
                    for (int64_t i = t16; i < end; ++i) gd[i - t16] = __ldg(p.W + i);
                    hi = t16;
                }
                src = p.W + lo;
                dst = dst0 + lane * p.pitch;
                nbytes = static_cast<uint32_t>(hi - lo);
            }
        }
        const uint32_t sum = __reduce_add_sync(0xFFFFFFFFu, nbytes);
        if (lane == 0) mbar_arrive_expect_tx(bar, sum);
        __syncwarp();
        if (nbytes) bulk_g2s(dst, src, nbytes, bar);
    };

    // Weights are constant inputs: every chunk the ring holds is requested before waiting for
    // the preceding kernel in the stream; x is read only after that kernel has completed.
    pdl_launch_dependents();
    Cursor ki, kc;
    start(ki);
    start(kc);
    int nissued = 0, nwaited = 0;   // chunk copies issued / completions seen
    for (; nissued < D && ki.u < units; ++nissued) {
        issue(nissued, ki);
        advance(ki);
    }
    pdl_wait();
    bool ok = true;
    if constexpr (M1) {
        stage_m1(p.x, p.nsb, xb, xs, p.swap);
    } else {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(p.xboxes) * p.xbox_bytes);
            for (int i = 0; i < p.xboxes; ++i) tma_load_3d(xb + i * p.xbox_bytes, &maps.x, 0, i * 256, 0, xbar);
        }
        if (!mbar_wait(xbar, 0)) ok = false;
        stage_x<PERM, false, KQ>(xb, xs, p.M, p.K);
    }
    __syncthreads();

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float acc1[2] = {0.f, 0.f};
    const uint32_t swap16 = (p.swap && (c & 1)) ? 16u : 0u;
    // single token: lane (g, c) carries column g when g / 2 == c; the others read the zero block
    const bool carrier = (g >> 1) == c;
    const uint32_t rec_step = carrier ? kM1RecSb : 0u;
    const uint32_t rec0 = carrier ? xb + static_cast<uint32_t>(g) * kM1RecPitch : xb + static_cast<uint32_t>(p.nsb) * kM1RecSb;
    const uint32_t tok = static_cast<uint32_t>(min(g, p.M - 1));
    const uint32_t xrows = static_cast<uint32_t>(p.K) / 64u;   // x rows per token
    int s = 0;
    uint32_t ph = 0;
    while (kc.u < units) {
        if (ok && !mbar_wait(bar0 + 8 * s, ph)) ok = false;
        if (ok) ++nwaited;
        const int t = kc.u / p.ks;
        const int row0 = r0 + 16 * t;
        const int sb0 = kc.c * p.C, ns = min(p.C, p.nsb - sb0);
        if (ok) {
            const uint32_t slot = ring + s * cbuf;
            uint32_t base_a = slot + g * p.pitch, base_b = slot + (g + 8) * p.pitch;
            if constexpr (!ALIGNED) {   // block data starts (o & 15) bytes into the row's window
                const uint32_t nsbu = static_cast<uint32_t>(p.nsb), sbu = static_cast<uint32_t>(sb0);
                const uint32_t ra = static_cast<uint32_t>(min(row0 + g, p.N - 1));
                const uint32_t rb = static_cast<uint32_t>(min(row0 + g + 8, p.N - 1));
                base_a += ((ra * nsbu + sbu) * static_cast<uint32_t>(BB)) & 15u;
                base_b += ((rb * nsbu + sbu) * static_cast<uint32_t>(BB)) & 15u;
            }
            // A buffer shorter than 16 rows (the CTA's last, partial tile) holds rows 0 .. brows-1:
            // lanes of rows beyond it decode row 0 instead (their results are never stored).
            if (g >= brows) base_a = slot;
            if (g + 8 >= brows) base_b = base_a;
            // the chunk's blocks inside this slot; its x (records or staged rows) and sums inside theirs
            const uint32_t span = static_cast<uint32_t>(ns) * BB, sbl = static_cast<uint32_t>(sb0 + ns - 1);
            const uint32_t x_end = M1 ? rec0 + sbl * rec_step + 128u
                                      : xb + (tok * xrows + 4u * sbl + 4u) * 128u;
            const uint32_t s_end = M1 ? xs + (sbl + 1u) * 32u : xs + (tok * static_cast<uint32_t>(p.nsb) + sbl + 1u) * 32u;
            const bool chunk_ok = in_bounds(ns >= 1 && sb0 + ns <= p.nsb && base_a + span <= slot + cbuf &&
                                                base_b + span <= slot + cbuf && x_end <= xs &&
                                                (!(M1 || KQ) || s_end <= base + p.red_off) &&
                                                (!M1 || rec0 >= xb),
                                            p.status);
            if (!chunk_ok) {
            } else if constexpr (M1) {
                // chunks of two superblocks (all but possibly a row's last) take a straight-line
                // body, so the compiler can interleave the two superblocks' loads and MMAs
                const uint32_t sb = static_cast<uint32_t>(sb0), rec = rec0 + sb * rec_step;
                if (ns == 2) {
                    m1_superblock<TYPE>(base_a, base_b, rec, xs + sb * 32u, c, swap16, acc1);
                    m1_superblock<TYPE>(base_a + BB, base_b + BB, rec + rec_step, xs + sb * 32u + 32u, c, swap16, acc1);
                } else {
                    for (int j = 0; j < ns; ++j)
                        m1_superblock<TYPE>(base_a + j * BB, base_b + j * BB, rec + j * rec_step, xs + (sb + j) * 32u, c,
                                            swap16, acc1);
                }
            } else {
#pragma unroll 2
                for (int j = 0; j < ns; ++j) {
                    const uint32_t sb = static_cast<uint32_t>(sb0 + j);
                    const uint32_t blk_a = base_a + j * BB, blk_b = base_b + j * BB;
                    const uint32_t rx = tok * xrows + 4u * sb;   // x row of segment 0 of this superblock
                    if constexpr (KQ) {
                        XRow xr = xrow(xb, rx + c);
                        xr.key ^= swap16 << 1;   // swapped halves pair with x chunks p ^ 2
                        superblock_kq<TYPE, PERM, true>(blk_a, blk_b, xr, c, acc,
                                                        xs + (tok * static_cast<uint32_t>(p.nsb) + sb) * 32u, swap16);
                    } else if constexpr (TYPE == 14 || TYPE == kQ6KAligned) {
                        superblock_q6<PERM, TYPE == kQ6KAligned>(blk_a, blk_b, xb, rx, c, acc);
                    } else {
                        superblock_iq4(blk_a, blk_b, xrow(xb, rx + c), c, acc);
                    }
                }
            }
        }
        // The slot's contents were read by this warp's ordinary loads, all consumed above (and
        // kept ahead of the copy issue by its memory clobber): no proxy fence for the refill.
        __syncwarp();
        const bool last_of_unit = (kc.c + 1 == kc.c1);
        const int u_done = kc.u;
        advance(kc);
        if (ok && ki.u < units) {
            issue(s, ki);
            advance(ki);
            ++nissued;
        }
        if (++s == D) {
            s = 0;
            ph ^= 1u;
        }
        if (last_of_unit) {
            const int tt = u_done / p.ks, jr = u_done % p.ks;
            const int rowt = r0 + 16 * tt;
            float out[4];
            int rows_of[4], toks_of[4];
            if constexpr (M1) {   // the four lanes of a row group hold its four sub-block pairs
                float a0 = acc1[0], a1 = acc1[1];
                a0 += __shfl_xor_sync(0xFFFFFFFFu, a0, 1);
                a1 += __shfl_xor_sync(0xFFFFFFFFu, a1, 1);
                a0 += __shfl_xor_sync(0xFFFFFFFFu, a0, 2);
                a1 += __shfl_xor_sync(0xFFFFFFFFu, a1, 2);
                acc1[0] = acc1[1] = 0.f;
                out[0] = a0; rows_of[0] = g; toks_of[0] = (c == 0) ? 0 : kGemvMaxM;
                out[1] = a1; rows_of[1] = g + 8; toks_of[1] = (c == 0) ? 0 : kGemvMaxM;
                out[2] = out[3] = 0.f; rows_of[2] = rows_of[3] = 0; toks_of[2] = toks_of[3] = kGemvMaxM;
            } else {
                out[0] = acc[0]; rows_of[0] = g; toks_of[0] = 2 * c;
                out[1] = acc[1]; rows_of[1] = g; toks_of[1] = 2 * c + 1;
                out[2] = acc[2]; rows_of[2] = g + 8; toks_of[2] = 2 * c;
                out[3] = acc[3]; rows_of[3] = g + 8; toks_of[3] = 2 * c + 1;
                acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = rowt + rows_of[i], m = toks_of[i];
                if (m < p.M && row < r1) {
                    const int ri = ((tt * p.ks + jr) * p.M + m) * 16 + rows_of[i];
                    if (p.ks == 1) {
                        if (in_bounds(row < p.N, p.status)) p.y[static_cast<int64_t>(m) * p.N + row] = out[i];
                    } else if (in_bounds(base + p.red_off + 4u * static_cast<uint32_t>(ri) + 4u <= base + p.wbuf_off[0],
                                         p.status)) {
                        red[ri] = out[i];
                    }
                }
            }
        }
    }
    if (p.ks > 1) {   // every unit of the CTA is done: sum each tile's K ranges in fixed order
        __syncthreads();
        const int per_tile = 16 * p.M;
        for (int q = threadIdx.x; q < ntile * per_tile; q += blockDim.x) {
            const int tt = q / per_tile, rem = q - tt * per_tile;   // tile, token * 16 + row
            const int row = r0 + 16 * tt + (rem & 15);
            if (row < r1) {
                float sum = 0.f;
                for (int jr = 0; jr < p.ks; ++jr) sum += red[(tt * p.ks + jr) * per_tile + rem];
                if (in_bounds(row < p.N && (rem >> 4) < p.M, p.status)) p.y[static_cast<int64_t>(rem >> 4) * p.N + row] = sum;
            }
        }
    }
    if (!ok) {
        if (lane == 0) atomicOr(p.status, kStatusTimeout);
        // let copies still in flight land before the shared memory is released
        for (int q = nwaited; q < nissued; ++q) (void)mbar_wait(bar0 + 8 * (q % D), (q / D) & 1);
        if (!M1) (void)mbar_wait(xbar, 0);
    }
}

// ---------------------------------------------------------------- host side

struct GsPlan {
    GsArgs a;
    int warps = 0, grid = 0;
    size_t smem = 0;
    bool ok = false;
};

int gs_max_warps(int type, bool m1) {
    switch (type) {
    case 12: return m1 ? GsFmt<12>::MAXW : GsFmt<12>::MAXW_GEN;
    case 13: return m1 ? GsFmt<13>::MAXW : GsFmt<13>::MAXW_GEN;
    case 14: return GsFmt<14>::MAXW_GEN;
    case kQ6KAligned: return GsFmt<kQ6KAligned>::MAXW_GEN;
    default: return GsFmt<23>::MAXW_GEN;
    }
}

// Superblocks per chunk (at most 2 KB per row: 256 box elements). K-quants: 2 (288 / 352 bytes,
// a row pitch of 32 or 96 mod 128 bytes: see the bank-conflict note above). Per-row bulk copies
// (Q6_K's 210-byte blocks): 3, about 0.6 KB per copy.
int gs_chunk(int type, bool tma) {
    if (!tma) return 3;
    switch (type) {
    case 12: return 2;            // 288 B
    case 13: return 2;            // 352 B
    case kQ6KAligned: return 4;   // 896 B
    default: return 4;            // IQ4_XS: 544 B
    }
}

GsPlan gs_plan_ranges(int type, int64_t N64, int64_t K64, int M, bool m1, int G, int ntile, int last_rows, int maxw,
                      bool tma, int C, int nchunk, int ks, int cpr, int xboxes, int xbox_rows);

GsPlan gs_make_plan(int type, int64_t N64, int64_t K64, int M, int num_sms, bool m1) {
    GsPlan pl;
    const int bb = block_bytes_of(type);
    const int nsb = static_cast<int>(K64 / 256);
    const int N = static_cast<int>(N64);
    const int64_t row_bytes = static_cast<int64_t>(nsb) * bb;
    // x: one box of up to 256 rows of 64 halves per copy; several tokens need a single box
    const int xrows = static_cast<int>(K64 / 64);
    const int xbox_rows = std::min(256, xrows);
    const int xboxes = (xrows + xbox_rows - 1) / xbox_rows;
    if (xboxes > 1 && M > 1) return pl;
    if (m1 && (K64 / 256) * kM1RecSb > 160 * 1024) return pl;   // records of very long rows: not planned
    // grid: at least 8 rows per CTA, at most one CTA per SM
    const int G = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(num_sms, (N64 + 7) / 8)));
    const int rows_max = (N + G - 1) / G;
    const int ntile = (rows_max + 15) / 16;
    const int last_rows = rows_max - 16 * (ntile - 1);
    const int maxw = gs_max_warps(type, m1);
    const bool tma = (row_bytes % 16 == 0) && type != 14 && (type != 23 || nsb % 2 == 0);
    // K ranges per tile: enough units for about twelve (single token) or eight warps
    const int target = m1 ? 12 : 8;
    const int ks_want = ntile >= target ? 1 : (target + ntile - 1) / ntile;
    int C = gs_chunk(type, tma);
    if (!tma && nsb / C < ks_want) C = std::max(1, nsb / ks_want);
    const int nchunk = (nsb + C - 1) / C;
    // K ranges per tile: at least ks_want (enough units for the warps), then the count whose
    // round-robin deal of units to warps gives the busiest warp the fewest chunks (fewer ranges
    // on a tie: less to reduce)
    auto busiest = [&](int ks_, int cpr_, int nw) {
        int most_ = 0;
        for (int w = 0; w < nw; ++w) {
            int n = 0;
            for (int u = w; u < ntile * ks_; u += nw) n += std::min((u % ks_ + 1) * cpr_, nchunk) - (u % ks_) * cpr_;
            most_ = std::max(most_, n);
        }
        return most_;
    };
    // candidates (busiest warp's chunks, ranges, chunks per range), tried best first until one fits
    struct Cand { int busy, ks, cpr; } cand[16];
    int ncand = 0;
    for (int k = std::min(ks_want, nchunk); k <= std::min(nchunk, 16); ++k) {
        const int cp = (nchunk + k - 1) / k, kk = (nchunk + cp - 1) / cp;
        if (kk != k) continue;
        cand[ncand++] = Cand{busiest(kk, cp, std::max(1, std::min(maxw, ntile * kk))), kk, cp};
    }
    std::sort(cand, cand + ncand, [](const Cand &x, const Cand &y) { return x.busy != y.busy ? x.busy < y.busy : x.ks < y.ks; });
    for (int i = 0; i < ncand; ++i) {
        GsPlan q = gs_plan_ranges(type, N64, K64, M, m1, G, ntile, last_rows, maxw, tma, C, nchunk, cand[i].ks, cand[i].cpr,
                                  xboxes, xbox_rows);
        if (q.ok) return q;
    }
    return pl;
}

// The rest of the plan for ks K ranges of cpr chunks each: the shared-memory layout and ring depth.
GsPlan gs_plan_ranges(int type, int64_t N64, int64_t K64, int M, bool m1, int G, int ntile, int last_rows, int maxw,
                      bool tma, int C, int nchunk, int ks, int cpr, int xboxes, int xbox_rows) {
    GsPlan pl;
    GsArgs &a = pl.a;
    const int bb = block_bytes_of(type);
    const int nsb = static_cast<int>(K64 / 256);
    const int N = static_cast<int>(N64);
    const int64_t row_bytes = static_cast<int64_t>(nsb) * bb;
    const int units = ntile * ks;
    const int NW = std::max(1, std::min(maxw, units));
    uint32_t pitch;
    int swap = 0;
    if (tma) {
        pitch = static_cast<uint32_t>(C * bb);   // rows land densely (a partial tile's rows too)
        const uint32_t delta = (pitch % 128u) / 16u;   // bank-group shift from row g to row g + 1
        swap = ((type == 12 || type == 13) && (delta == 2u || delta == 6u)) ? 1 : 0;
    } else {
        // the widest window of C blocks, an odd multiple of 16 bytes
        pitch = (static_cast<uint32_t>(C * bb) + 30u + 15u) & ~15u;
        if ((pitch / 16u) % 2u == 0u) pitch += 16u;
    }
    // staged x and its sums
    const uint32_t xbox_bytes = static_cast<uint32_t>(xbox_rows) * 128u * static_cast<uint32_t>(M);
    const uint32_t xbytes = m1 ? static_cast<uint32_t>(nsb) * kM1RecSb + kM1ZeroBytes
                               : static_cast<uint32_t>(xboxes) * xbox_bytes;
    uint32_t xsbytes = 0;
    if (m1) xsbytes = static_cast<uint32_t>(nsb) * 32u;
    else if (type == 12 || type == 13) xsbytes = static_cast<uint32_t>(M) * static_cast<uint32_t>(nsb) * 32u;
    const uint32_t barbytes = 8u * kGsMaxD * kGsMaxWarps + 128u;   // warps' rings, then x
    const uint32_t redbytes = ks > 1 ? static_cast<uint32_t>(ntile * ks * M * 16 * 4) : 0u;
    uint32_t off = (barbytes + 1023u) & ~1023u;
    a.xb_off = off;
    off = (off + xbytes + 127u) & ~127u;
    a.xs_off = off;
    off = (off + xsbytes + 127u) & ~127u;
    a.red_off = off;
    off = (off + redbytes + 127u) & ~127u;
    // ring: warp w's buffers hold 16 rows, or the last tile's rows when all its units are there
    size_t per_d = 0;
    for (int w = 0; w < NW; ++w) {
        bool only_last = true;
        for (int u = w; u < units; u += NW)
            if (u / ks != ntile - 1) only_last = false;
        a.wbuf_rows[w] = only_last ? static_cast<uint32_t>(last_rows) : 16u;
        a.wslot[w] = (a.wbuf_rows[w] * pitch + 127u) & ~127u;
        per_d += a.wslot[w];
    }
    // chunks of the busiest warp
    int most = 0;
    for (int w = 0; w < NW; ++w) {
        int n = 0;
        for (int u = w; u < units; u += NW) n += std::min((u % ks + 1) * cpr, nchunk) - (u % ks) * cpr;
        most = std::max(most, n);
    }
    const size_t limit = 227 * 1024 - 1024;   // 1 KB of alignment slack
    if (off + per_d > limit) return pl;
    const int D = static_cast<int>(std::min<size_t>({static_cast<size_t>(most), static_cast<size_t>(kGsMaxD),
                                                     (limit - off) / per_d}));
    if (D < std::min(2, most)) return pl;
    for (int w = 0; w < NW; ++w) {
        a.wbuf_off[w] = off;
        off += static_cast<uint32_t>(D) * a.wslot[w];
    }
    a.wbuf_off[NW] = off;
    for (int w = NW; w < kGsMaxWarps; ++w) a.wbuf_rows[w] = a.wslot[w] = 0;
    a.N = N;
    a.K = static_cast<int>(K64);
    a.M = M;
    a.nsb = nsb;
    a.C = C;
    a.nchunk = nchunk;
    a.ks = ks;
    a.cpr = cpr;
    a.D = D;
    a.tma = tma ? 1 : 0;
    a.swap = swap;
    a.xboxes = xboxes;
    a.xbox_bytes = xbox_bytes;
    a.pitch = pitch;
    a.total_bytes = N64 * row_bytes;
    pl.warps = NW;
    pl.grid = G;
    pl.smem = static_cast<size_t>(off) + 1024;
    pl.ok = true;
    return pl;
}

template <int TYPE, bool M1>
cudaError_t gs_launch_t(const GsMaps &m, const GsArgs &a, int grid, int warps, size_t smem, bool pdl, cudaStream_t st) {
    constexpr int MAXW = M1 ? GsFmt<TYPE>::MAXW : GsFmt<TYPE>::MAXW_GEN;
    auto kern = gemv_stream_kernel<TYPE, M1, MAXW>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    void *args[] = {const_cast<GsMaps *>(&m), const_cast<GsArgs *>(&a)};
    return launch_pdl(reinterpret_cast<const void *>(kern), dim3(grid), dim3(32 * warps), smem, st, pdl, args);
}

}  // namespace

bool gemv_stream_supported(int type, int64_t N, int64_t K, int M, int num_sms) {
    if (block_bytes_of(type) < 0 || M < 1 || M > kGemvMaxM) return false;
    const bool m1 = M == 1 && (type == 12 || type == 13);
    return gs_make_plan(type, N, K, M, num_sms, m1).ok;
}

cudaError_t gemv_stream_launch(int type, const uint8_t *W, const __half *x, float *y, int64_t N, int64_t K, int M,
                               unsigned *status, int num_sms, bool pdl, cudaStream_t stream) {
    if (M < 1 || M > kGemvMaxM || block_bytes_of(type) < 0) return cudaErrorInvalidValue;
    const bool m1 = M == 1 && (type == 12 || type == 13);
    GsPlan pl = gs_make_plan(type, N, K, M, num_sms, m1);
    if (!pl.ok) return cudaErrorNotSupported;
    pl.a.W = W;
    pl.a.x = x;
    pl.a.y = y;
    pl.a.status = status;
    GsMaps maps{};
    const uint64_t row_elems = static_cast<uint64_t>(pl.a.nsb) * block_bytes_of(type) / 8;
    if (pl.a.tma &&   // W as [N rows][row bytes / 8] of 8-byte elements, boxes of 16 rows x C superblocks
        !encode_tmap_2d(&maps.w, CU_TENSOR_MAP_DATA_TYPE_UINT64, W, row_elems, static_cast<uint64_t>(N), row_elems * 8,
                        static_cast<uint32_t>(pl.a.C * block_bytes_of(type) / 8), 16, false))
        return cudaErrorInvalidValue;
    // x as [M tokens][K/64 rows][64 halves]; one box = up to 256 rows of every token, 128-byte swizzled
    const uint32_t xbox_rows = pl.a.xbox_bytes / (128u * static_cast<uint32_t>(M));
    if (!encode_tmap_3d(&maps.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, 64, static_cast<uint64_t>(K / 64),
                        static_cast<uint64_t>(M), 128, static_cast<uint64_t>(K) * 2, 64, xbox_rows,
                        static_cast<uint32_t>(M), true))
        return cudaErrorInvalidValue;
    switch (type) {
    case 12: return m1 ? gs_launch_t<12, true>(maps, pl.a, pl.grid, pl.warps, pl.smem, pdl, stream)
                       : gs_launch_t<12, false>(maps, pl.a, pl.grid, pl.warps, pl.smem, pdl, stream);
    case 13: return m1 ? gs_launch_t<13, true>(maps, pl.a, pl.grid, pl.warps, pl.smem, pdl, stream)
                       : gs_launch_t<13, false>(maps, pl.a, pl.grid, pl.warps, pl.smem, pdl, stream);
    case 14: return gs_launch_t<14, false>(maps, pl.a, pl.grid, pl.warps, pl.smem, pdl, stream);
    case kQ6KAligned: return gs_launch_t<kQ6KAligned, false>(maps, pl.a, pl.grid, pl.warps, pl.smem, pdl, stream);
    case 23: return gs_launch_t<23, false>(maps, pl.a, pl.grid, pl.warps, pl.smem, pdl, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ql
