// gemm_tc.cu -- prefill-path quantized linear y[M, N] = x[M, K] . dequant(W)[N, K]^T on the
// 5th-generation tensor cores (tcgen05, sm_103a).
//
// Tiling ("swap AB"): a CTA owns 128 weight rows (the MMA's M side, one TMEM lane per row)
// and a tile of n_tile tokens (the MMA's N side, 32..256). The fp32 accumulator lives in
// TMEM columns [0, n_tile). K is walked superblock by superblock (256 k = 16 MMAs of K = 16);
// every hand-off between roles is per superblock, because a wait/fence/commit round costs
// several hundred cycles, far above one MMA issue (about 30 cycles at small N), and finer
// hand-offs would starve the tensor pipe at small N.
//
// Warp roles (352 threads):
//   warps 0-7  dequantisers: warp w serves TMEM lane quarter w % 4 (rows 32(w%4)..+31, one
//              thread per row) and the superblocks of parity w / 4. Each thread decodes its
//              row's 256 weights of a superblock from the staged block into fp16 and writes
//              them with tcgen05.st into a TMEM A-operand ring (2 or 3 superblock slots of 128
//              columns); the MMA reads A straight from TMEM, so dequantised weights never touch
//              shared memory. After the K loop the same warps drain the accumulator to y, warp
//              w taking the column half w / 4.
//   warp 8     weight producer: one 2-D TMA tensor copy per stage (S superblocks of the 128
//              rows) into a shared-memory ring when rows are 16-byte multiples, else one bulk
//              copy per row over the aligned window around the row's span.
//   warp 9     activation producer: 2-D TMA of the x tile [n_tile tokens x 64 k], 128-byte
//              swizzled, the MMA's B operand.
//   warp 10    TMEM allocator and MMA issue (the warp runs the loop, one elected lane issues).
// All hand-offs are mbarriers; every wait is bounded and an expired wait aborts the CTA
// (status word set, TMEM freed).
//
// Few row tiles (at most half the SM count) and M <= 256 take gemm_split_kernel instead: all M
// tokens in one tile and each row tile's superblocks shared by a pair of CTAs in a thread-block
// cluster, the second adding its partial sums into the first's through one bulk copy between
// their shared memories. Several token tiles would each decode every weight again.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <cuda.h>
#include <mutex>
#include <type_traits>
#include <vector>

#include "kernels.h"
#include "ptx.cuh"

namespace ql {

namespace {

constexpr int kRows = 128;          // weight rows per CTA (MMA M)
constexpr int kChunkK = 64;         // k per pipeline chunk
constexpr int kMaxASlots = 3;       // TMEM A ring: superblock slots of 128 columns
constexpr uint32_t kASlotCols = 128;
constexpr int kDequantWarps = 8;
constexpr int kThreads = 32 * 11;
constexpr uint32_t kTmemCols = 512;
constexpr int kAccBars = 2;         // accumulator final; (head) the tail's partial sums handed over
// Heads per tail in the split kernel. Measured on GB300 at M=32, K=4096: two heads per tail
// (where pairs do not fit) gave N=10240 14.8 -> 13.9 us; three gave N=12288 15.0 -> 16.4 us for
// Q4_K (Q6_K 38.9 -> 37.6, IQ4_XS 21.8 -> 21.3), the tail's serial drain of three tiles costing
// more than the superblocks saved. Pairs gain 1.75-2.3x wherever they fit.
constexpr int kMaxSplitK = 2;

struct GemmArgs {
    const uint8_t *W;
    float *y;
    unsigned *status;
    int N, K, M, nsb;
    int n_tile;
    int S;                     // superblocks per weight stage
    uint32_t row_pitch;        // bytes per weight row in a weight stage
    int qstages, bstages;
    int xk;                    // 64-wide chunks per activation stage (1, 2 or 4)
    int a_slots;               // TMEM A ring depth in superblocks (2 or 3)
    uint32_t a_col;            // first TMEM column of the A ring (256 or 128)
    uint32_t q_stage_bytes, b_stage_bytes;   // b stage = xk boxes of n_tile x 128 bytes
    uint32_t q_off, bar_off;   // offsets from the 1024-aligned shared base
    int64_t total_bytes;
    int bb;                    // bytes per superblock
    int type;
    // Work split (the SPLIT kernel, one token tile): clusters of k + 1 CTAs. Rank r < k is the head of
    // row tile cid k + r and takes superblocks [0, L); rank k takes the tails [L, nsb) of the
    // cluster's tiles back to back, tile i's sums in TMEM columns [i n_tile, (i+1) n_tile). The
    // tail stages tile i's sums at the base of its shared memory (rows of part_stride floats)
    // and copies them into head i's receive area at recv_off.
    // Unsplit: one CTA per (row tile, token tile), all superblocks.
    int k, L, tail, row_tiles, part_stride;
    uint32_t recv_off;
};

// ------------------------------------------------------------ per-row dequantisers
// Each produces the 32 fp16 weights k = 32h .. 32h+31 of 64-wide chunk gg of one row as 16
// packed pairs (k, k+1), i.e. the 16 TMEM columns [16h, 16h+16) of that chunk. K-quant weights
// d * (sc q) - dmin m are formed by one mixed-precision FMA (sc q an exact fp16 integer) and
// rounded once to fp32 and once to fp16, so the MMA operand is the weight to within one fp16
// rounding also where d sc q and dmin m nearly cancel. Q6_K and IQ4_XS weights are the integer
// code times the fp32 scale (d sc exact), whose product may round in fp32 (at most 2^-24
// relative) before the fp16 rounding.

// (q0, q1) exact integers in fp16 -> fp16x2(q0 * s + o, q1 * s + o), each rounded once
__device__ __forceinline__ uint32_t scale_pair(uint32_t q2, float s, float o) {
    const float2 q = __half22float2(*reinterpret_cast<const __half2 *>(&q2));
    const __half2 r = __floats2half2_rn(fmaf(q.x, s, o), fmaf(q.y, s, o));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// (q0, q1) fp16 pair of exact integers -> fp16x2(d * q0 + c, d * q1 + c): each product and sum
// formed exactly by a mixed-precision FMA (f16 inputs, f32 addend and result) and rounded once
// to fp32, then to fp16.
__device__ __forceinline__ uint32_t affine_pair(uint32_t q2, uint32_t d2, float c) {
    float r0, r1;
    asm("{\n\t.reg .b16 q0, q1, d0, d1;\n\tmov.b32 {q0, q1}, %2;\n\tmov.b32 {d0, d1}, %3;\n\t"
        "fma.rn.f32.f16 %0, d0, q0, %4;\n\tfma.rn.f32.f16 %1, d0, q1, %4;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "r"(q2), "r"(d2), "f"(c));
    const __half2 r = __floats2half2_rn(r0, r1);
    return *reinterpret_cast<const uint32_t *>(&r);
}

struct KqRow {
    // Sub-blocks 2gg + h, gg = 0..3. The decoded pair v is (1024 + q) (h = 0) or (1024 + 16q)
    // (h = 1); hfma2(v, sc2, nsc2) with sc2 = sc (sc/16) and nsc2 = -1024 sc (-64 sc) is sc*q,
    // exact: the fused product is exact and sc*q <= 63*31 fits fp16's 11 bits.
    uint32_t sc2[4], nsc2[4];
    float ndm[4];   // -dmin*m (exact in fp32)
    uint32_t d2;    // (d, d)
};

__device__ __forceinline__ KqRow kq_row(uint32_t blk, int h) {
    const uint4 hd = lds128(blk);
    const uint32_t A = hd.y, B = hd.z, C = hd.w;
    const uint32_t sc_lo4 = A & 0x3F3F3F3Fu, m_lo4 = B & 0x3F3F3F3Fu;
    const uint32_t sc_hi4 = and_or(C, 0x0F0F0F0Fu, (A >> 2) & 0x30303030u);
    const uint32_t m_hi4 = and_or(C >> 4, 0x0F0F0F0Fu, (B >> 2) & 0x30303030u);
    // pool byte j = value of sub-block j; pick j = h, 2+h, 4+h, 6+h
    const uint32_t sel = static_cast<uint32_t>(h) | ((2u + h) << 4) | ((4u + h) << 8) | ((6u + h) << 12);
    const uint32_t sc4 = prmt(sc_lo4, sc_hi4, sel), m4 = prmt(m_lo4, m_hi4, sel);
    const float dmin = half_hi_to_float(hd.x);
    KqRow r;
    r.d2 = prmt(hd.x, 0u, 0x1010u);
    // scales as exact fp16 pairs (1024 + sc) - 1024, times 1 or 1/16 (exact), and the offsets
    const uint32_t scale = h ? kH2_1_16 : 0x3C003C00u, off = h ? kH2_m64 : kH2_m1024;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t s = (sc4 >> (8 * i)) & 0xFFu;
        const uint32_t sc = hsub2((s | (s << 16)) | kH2_1024, kH2_1024);
        r.sc2[i] = hmul2(sc, scale);
        r.nsc2[i] = hmul2(sc, off);
        r.ndm[i] = -dmin * static_cast<float>((m4 >> (8 * i)) & 0xFFu);
    }
    return r;
}

template <bool Q5, int h>
__device__ __forceinline__ void kq_chunk(uint32_t blk, int gg, const KqRow &r, uint32_t (&out)[16]) {
    constexpr uint32_t QS = Q5 ? 48 : 16;
    const uint4 q0 = lds128(blk + QS + 32 * gg), q1 = lds128(blk + QS + 32 * gg + 16);
    uint4 h0 = make_uint4(0, 0, 0, 0), h1 = h0;
    if constexpr (Q5) {
        h0 = lds128(blk + 16);
        h1 = lds128(blk + 32);
    }
    const uint32_t sc2 = r.sc2[gg], nsc2 = r.nsc2[gg], d2 = r.d2;
    const float ndm = r.ndm[gg];
    const uint32_t j = 2u * gg + h;   // sub-block (and qh bit) of these weights
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint32_t w = u < 4 ? (u == 0 ? q0.x : u == 1 ? q0.y : u == 2 ? q0.z : q0.w)
                                 : (u == 4 ? q1.x : u == 5 ? q1.y : u == 6 ? q1.z : q1.w);
        const uint32_t w2 = prmt(w, 0u, 0x3120u), w3 = w2 >> 8;
        uint32_t v01, v23, q01, q23;
        if (h == 0) {
            v01 = and_or(w2, 0x000F000Fu, kH2_1024);
            v23 = and_or(w3, 0x000F000Fu, kH2_1024);
        } else {
            v01 = and_or(w2, 0x00F000F0u, kH2_1024);
            v23 = and_or(w3, 0x00F000F0u, kH2_1024);
        }
        if constexpr (Q5) {
            const uint32_t hw = u < 4 ? (u == 0 ? h0.x : u == 1 ? h0.y : u == 2 ? h0.z : h0.w)
                                      : (u == 4 ? h1.x : u == 5 ? h1.y : u == 6 ? h1.z : h1.w);
            const uint32_t hq2 = prmt(hw, 0u, 0x3120u), hq3 = hq2 >> 8;
            // bit j of each qh byte -> bit 4 (low nibble path) or bit 8 (high nibble path, x16)
            const uint32_t rot = ((h == 0 ? 4u : 8u) - j) & 31u;
            const uint32_t mask = h == 0 ? 0x00100010u : 0x01000100u;
            v01 = or_and(v01, rotl(hq2, rot), mask);
            v23 = or_and(v23, rotl(hq3, rot), mask);
        }
        q01 = hfma2(v01, sc2, nsc2);   // sc*q, exact
        q23 = hfma2(v23, sc2, nsc2);
        out[2 * u] = affine_pair(q01, d2, ndm);
        out[2 * u + 1] = affine_pair(q23, d2, ndm);
    }
}

__device__ __forceinline__ uint4 lds128_a2(uint32_t addr) {
    const uint32_t a = addr & ~3u;
    const uint32_t sel = (addr & 2u) ? 0x5432u : 0x3210u;
    const uint32_t w0 = lds32(a), w1 = lds32(a + 4), w2 = lds32(a + 8), w3 = lds32(a + 12), w4 = lds32(a + 16);
    return make_uint4(prmt(w0, w1, sel), prmt(w1, w2, sel), prmt(w2, w3, sel), prmt(w3, w4, sel));
}

// Q6_K chunk gg: half hf = gg / 2 of the block, quarter t = 2 (gg % 2) + h, l = 0..31.
// ALIGNED: blocks start on 16-byte boundaries (the 224-byte layout).
template <int h, bool ALIGNED = false>
__device__ __forceinline__ void q6_chunk(uint32_t blk, int gg, uint32_t (&out)[16]) {
    const int hf = gg >> 1, t = 2 * (gg & 1) + h;
    const float d = half_lo_to_float(lds16(blk + 208));
    const uint32_t scb = lds16(blk + 192 + 8 * hf + 2 * t);   // sc[8hf+2t], sc[8hf+2t+1] (int8)
    const float ds0 = d * static_cast<float>(static_cast<int8_t>(scb & 0xFFu));          // l < 16
    const float ds1 = d * static_cast<float>(static_cast<int8_t>((scb >> 8) & 0xFFu));   // l >= 16
    const uint32_t qlo = 64 * hf + 32 * h, qho = 128 + 32 * hf;
    auto ld16 = [](uint32_t a) { return ALIGNED ? lds128(a) : lds128_a2(a); };
    const uint4 l0 = ld16(blk + qlo), l1 = ld16(blk + qlo + 16);
    const uint4 g0 = ld16(blk + qho), g1 = ld16(blk + qho + 16);
    const int sh = 4 - 2 * t;   // qh bits 2t, 2t+1 -> bits 4, 5
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint32_t lw = u < 4 ? (u == 0 ? l0.x : u == 1 ? l0.y : u == 2 ? l0.z : l0.w)
                                  : (u == 4 ? l1.x : u == 5 ? l1.y : u == 6 ? l1.z : l1.w);
        const uint32_t hw = u < 4 ? (u == 0 ? g0.x : u == 1 ? g0.y : u == 2 ? g0.z : g0.w)
                                  : (u == 4 ? g1.x : u == 5 ? g1.y : u == 6 ? g1.z : g1.w);
        uint32_t l2 = prmt(lw, 0u, 0x3120u);
        if (t >= 2) l2 >>= 4;
        const uint32_t l3 = l2 >> 8;
        const uint32_t h2 = prmt(hw, 0u, 0x3120u), h3 = h2 >> 8;
        uint32_t v01 = and_or(l2, 0x000F000Fu, kH2_1024);
        uint32_t v23 = and_or(l3, 0x000F000Fu, kH2_1024);
        v01 = or_and(v01, sh >= 0 ? (h2 << sh) : (h2 >> -sh), 0x00300030u);
        v23 = or_and(v23, sh >= 0 ? (h3 << sh) : (h3 >> -sh), 0x00300030u);
        const float ds = u < 4 ? ds0 : ds1;
        out[2 * u] = scale_pair(hsub2(v01, kH2_1056), ds, 0.f);
        out[2 * u + 1] = scale_pair(hsub2(v23, kH2_1056), ds, 0.f);
    }
}

constexpr uint32_t kIq4T0 = 0x3F2D1801u, kIq4T1 = 0x766A5D4Fu, kIq4T2 = 0xA6998D81u, kIq4T3 = 0xF1D9C5B5u;

__device__ __forceinline__ uint32_t iq4_lookup(uint32_t s) {
    const uint32_t s7 = s & 0x7777u;
    const uint32_t lo = prmt(kIq4T0, kIq4T1, s7), hi = prmt(kIq4T2, kIq4T3, s7);
    return prmt(lo, hi, ((s >> 1) & 0x4444u) | 0x3210u);
}

// IQ4_XS chunk gg, half h: sub-block j = 2gg + h, 16 qs bytes -> [low nibbles, high nibbles].
template <int h>
__device__ __forceinline__ void iq4_chunk(uint32_t blk, int gg, uint32_t (&out)[16]) {
    const int j = 2 * gg + h;
    const uint2 hd = lds64(blk);
    const uint32_t ls = ((hd.y >> (4 * j)) & 15u) | (((hd.x >> (16 + 2 * j)) & 3u) << 4);
    const float dl = half_lo_to_float(hd.x) * static_cast<float>(static_cast<int>(ls) - 32);   // d * (ls - 32)
    const uint2 a = lds64(blk + 8 + 16 * j), b = lds64(blk + 16 + 16 * j);
    const uint32_t kH2_1152 = 0x64806480u;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint32_t w = u == 0 ? a.x : u == 1 ? a.y : u == 2 ? b.x : b.y;   // bytes p = 4u .. 4u+3
        const uint32_t r01 = iq4_lookup(w), r23 = iq4_lookup(w >> 16);
        out[2 * u] = scale_pair(hsub2(prmt(r01, 0x64646464u, 0x4240u), kH2_1152), dl, 0.f);       // r = p, p+1
        out[2 * u + 1] = scale_pair(hsub2(prmt(r23, 0x64646464u, 0x4240u), kH2_1152), dl, 0.f);   // p+2, p+3
        out[8 + 2 * u] = scale_pair(hsub2(prmt(r01, 0x64646464u, 0x4341u), kH2_1152), dl, 0.f);   // p+16, p+17
        out[9 + 2 * u] = scale_pair(hsub2(prmt(r23, 0x64646464u, 0x4341u), kH2_1152), dl, 0.f);   // p+18, p+19
    }
}

// The four chunks of one superblock, half h, into TMEM columns acol + 32 gg + [0, 16).
template <int TYPE, int h>
__device__ __forceinline__ void dequant_superblock(uint32_t blk, const KqRow &kr, uint32_t acol) {
#pragma unroll
    for (int gg = 0; gg < 4; ++gg) {
        uint32_t out[16];
        if constexpr (TYPE == 12) kq_chunk<false, h>(blk, gg, kr, out);
        else if constexpr (TYPE == 13) kq_chunk<true, h>(blk, gg, kr, out);
        else if constexpr (TYPE == 14) q6_chunk<h>(blk, gg, out);
        else if constexpr (TYPE == kQ6KAligned) q6_chunk<h, true>(blk, gg, out);
        else iq4_chunk<h>(blk, gg, out);
        tmem_st16(acol + 32 * gg, out);
    }
}

// ------------------------------------------------------------ clusters (split kernel)

// Barrier `id` (1..15) over `count` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// ---- thread-block clusters and distributed shared memory
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of `addr` (a shared::cta address) in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from this CTA's shared
// memory to another CTA's of the cluster (`dst`, `bar`: shared::cluster addresses); completes
// as transaction bytes on the destination CTA's mbarrier. The source must have been written
// before a fence.proxy.async.
__device__ __forceinline__ void bulk_s2s_cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "r"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// Every thread of every CTA of the cluster: no CTA leaves before all have arrived, so no
// shared memory another CTA may still read is released early.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------ bounded waits with abort

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                              unsigned *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait_for(bar, parity, 100000u)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort_flag = 1u;
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
    return true;
}

}  // namespace

// The 16 MMAs of one superblock (A in TMEM at a0, accumulator d, overwritten by the first MMA
// when `overwrite`), over the superblock's 4 / XK x stages of the ring (stage sbb, phase bph,
// advanced here): for each stage the warp waits for it, then one elected lane issues the
// stage's MMAs and the commits that release it (after the last stage also the A slot). One
// elected block per stage rather than per 64-wide chunk: measured on GB300 at n_tile 32, Q4_K
// K=4096 N=12288 M=32 went 18.9 -> 15.2 us. False when a wait expired.
template <int XK>
__device__ __forceinline__ bool mma_superblock(uint32_t d, uint32_t a0, bool overwrite, uint32_t idesc, uint32_t b_ring,
                                               uint32_t b_stage_bytes, uint32_t box_bytes, uint32_t bfull0,
                                               uint32_t bempty0, uint32_t aempty_bar, int BS, int &sbb, uint32_t &bph,
                                               volatile uint32_t *abort_flag, unsigned *status) {
#pragma unroll
    for (int g0 = 0; g0 < 4; g0 += XK) {
        if (!__all_sync(0xFFFFFFFFu, wait_or_abort(bfull0 + 8u * sbb, bph, abort_flag, status))) return false;
        tc_fence_after();
        const uint64_t bd = smem_desc_sw128(b_ring + sbb * b_stage_bytes);
        if (elect_one()) {
#pragma unroll
            for (int i = 0; i < XK; ++i)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_ts(d, a0 + 32 * (g0 + i) + 8 * kk, bd + ((i * box_bytes) >> 4) + 2 * kk, idesc,
                              !(overwrite && g0 + i == 0 && kk == 0));
            tc_commit(bempty0 + 8u * sbb);
            if (g0 + XK >= 4) tc_commit(aempty_bar);
        }
        __syncwarp();
        if (++sbb == BS) {
            sbb = 0;
            bph ^= 1u;
        }
    }
    return true;
}

template <int TYPE, bool TMA>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap, const GemmArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t b_ring = base;
    const uint32_t q_ring = base + p.q_off;
    const uint32_t bars = base + p.bar_off;
    const int QS = p.qstages, BS = p.bstages;
    auto qfull = [&](int s) { return bars + 8u * s; };
    auto qempty = [&](int s) { return bars + 8u * (QS + s); };
    auto bfull = [&](int s) { return bars + 8u * (2 * QS + s); };
    auto bempty = [&](int s) { return bars + 8u * (2 * QS + BS + s); };
    auto afull = [&](int s) { return bars + 8u * (2 * QS + 2 * BS + s); };
    auto aempty = [&](int s) { return bars + 8u * (2 * QS + 2 * BS + kMaxASlots + s); };
    const uint32_t accfull = bars + 8u * (2 * QS + 2 * BS + 2 * kMaxASlots);
    const uint32_t misc_off = p.bar_off + 8u * (2 * QS + 2 * BS + 2 * kMaxASlots + 1);
    const int AS = p.a_slots;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + misc_off);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + misc_off + 4);

    const int n0 = blockIdx.x * kRows;
    const int t0 = blockIdx.y * p.n_tile;
    const int nchunks = p.nsb * 4;
    if constexpr (kBoundsChecks) {   // rings, barriers and TMEM columns inside their budgets
        uint32_t dyn;
        asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
        const bool lay = misc_off + 8u + (base - raw) <= dyn && static_cast<uint32_t>(BS) * p.b_stage_bytes <= p.q_off &&
                         p.q_off + static_cast<uint32_t>(QS) * p.q_stage_bytes <= p.bar_off &&
                         p.q_stage_bytes >= kRows * p.row_pitch && p.row_pitch >= static_cast<uint32_t>(p.S * p.bb) &&
                         static_cast<uint32_t>(p.n_tile) <= p.a_col && AS <= kMaxASlots &&
                         p.a_col + static_cast<uint32_t>(AS) * kASlotCols <= kTmemCols &&
                         p.b_stage_bytes >= static_cast<uint32_t>(p.xk * p.n_tile) * 128u;
        if (!in_bounds(lay, p.status)) return;
    }

    if (threadIdx.x == 0) {
        // a stage of one superblock is read by the 4 warps of its parity, a wider one by all 8
        for (int s = 0; s < QS; ++s) {
            mbar_init(qfull(s), 1);
            mbar_init(qempty(s), p.S == 1 ? kDequantWarps / 2 : kDequantWarps);
        }
        for (int s = 0; s < BS; ++s) {
            mbar_init(bfull(s), 1);
            mbar_init(bempty(s), 1);
        }
        for (int s = 0; s < kMaxASlots; ++s) {
            mbar_init(afull(s), kDequantWarps / 2);   // the 4 warps of one superblock parity
            mbar_init(aempty(s), 1);
        }
        mbar_init(accfull, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 10) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 9 && lane == 0) prefetch_tmap(&xmap);
    if (TMA && warp == 8 && lane == 0) prefetch_tmap(&wmap);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The weights stream while the preceding kernel in the stream finishes; x is loaded (and
    // y written, downstream of x) only after it has completed.
    pdl_launch_dependents();

    if (warp < kDequantWarps) {
        // ---------------------------------------------------- dequantisers
        // The two warps of a TMEM lane quarter (one per scheduler pair) take alternate
        // superblocks and decode both chunk halves of theirs: one warp's hand-off and header
        // decode then overlap the other's decode, instead of both stalling at the same time.
        const int q = warp & 3, par = warp >> 2, h = warp >> 2;   // h: epilogue column half
        const int r = 32 * q + lane;
        const int row = min(n0 + r, p.N - 1);
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const int lg_s = __ffs(p.S) - 1;   // S is 1, 2 or 4
        bool ok = true;
        for (int sb = par; sb < p.nsb && ok; sb += 2) {
            // weight stage sb >> lg_s at ring slot qs with phase qph; its copy may already have
            // been waited for by this warp (the wait then returns at once: the slot cannot be
            // refilled before this warp's release of it below)
            const int si = sb >> lg_s, j = sb & (p.S - 1);
            const int qs = si % QS;
            const uint32_t qph = static_cast<uint32_t>(si / QS) & 1u;
            ok = wait_or_abort(qfull(qs), qph, abort_flag, p.status);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            const uint32_t stage = q_ring + qs * p.q_stage_bytes;
            uint32_t blk = stage + r * p.row_pitch + j * p.bb;
            if constexpr (!TMA)   // block data starts (o & 15) bytes into the row's window (unsigned
                                  // arithmetic wraps modulo 2^32 and keeps the low four bits)
                blk += ((static_cast<uint32_t>(row) * static_cast<uint32_t>(p.nsb) + static_cast<uint32_t>(sb - j)) *
                        static_cast<uint32_t>(p.bb)) & 15u;
            if (!in_bounds(blk + static_cast<uint32_t>(p.bb) <= stage + (r + 1) * p.row_pitch, p.status))
                blk = stage + r * p.row_pitch;   // bounds check failed: decode the row's first block instead
            KqRow kr0{}, kr1{};
            if constexpr (TYPE == 12 || TYPE == 13) {
                kr0 = kq_row(blk, 0);
                kr1 = kq_row(blk, 1);
            }
            const int sa = sb % AS;
            const uint32_t aph = static_cast<uint32_t>(sb / AS) & 1u;
            ok = wait_or_abort(aempty(sa), aph ^ 1u, abort_flag, p.status);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t acol = tmem + lane_base + p.a_col + sa * kASlotCols;
            dequant_superblock<TYPE, 0>(blk, kr0, acol);
            dequant_superblock<TYPE, 1>(blk, kr1, acol + 16);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(afull(sa));
                // release the stage after this warp's last superblock in it
                if ((sb + 2) >> lg_s != si || sb + 2 >= p.nsb) mbar_arrive(qempty(qs));
            }
        }
        // ---------------------------------------------------- epilogue: TMEM -> y
        if (ok) ok = wait_or_abort(accfull, 0, abort_flag, p.status);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (ok) {
            tc_fence_after();
            // 16-column groups of the accumulator: the first half of them to h = 0, the rest to h = 1
            const int ng = p.n_tile / 16, g_mid = ng / 2;
            for (int c0 = 16 * (h ? g_mid : 0); c0 < 16 * (h ? ng : g_mid); c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem + lane_base + c0, v);
                tmem_wait_ld();
                if (n0 + r < p.N) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int t = t0 + c0 + i;
                        if (t < p.M) p.y[static_cast<int64_t>(t) * p.N + n0 + r] = __uint_as_float(v[i]);
                    }
                }
            }
        }
    } else if (warp == 8) {
        // ---------------------------------------------------- weight producer
        const int nstages = (p.nsb + p.S - 1) / p.S;
        int issued = 0, s = 0;
        uint32_t ph = 0;
        for (int si = 0; si < nstages; ++si) {
            if (!wait_or_abort(qempty(s), ph ^ 1u, abort_flag, p.status)) break;
            fence_proxy_async_smem();
            const uint32_t st = q_ring + s * p.q_stage_bytes;
            if constexpr (TMA) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(qfull(s), p.q_stage_bytes);
                    tma_load_2d(st, &wmap, si * p.S * (p.bb / 4), n0, qfull(s));
                }
            } else {
                const int sb = si * p.S, ns = min(p.S, p.nsb - sb);
                uint32_t my = 0;
                const uint8_t *src[4];
                uint32_t dst[4], nb[4];
                int tail_len = 0;
                uint32_t tail_dst = 0;
                const uint8_t *tail_src = nullptr;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int rr = lane + 32 * i, rowi = n0 + rr;
                    nb[i] = 0;
                    src[i] = nullptr;
                    dst[i] = 0;
                    if (rowi < p.N) {
                        const int64_t o = (static_cast<int64_t>(rowi) * p.nsb + sb) * p.bb;
                        const int64_t lo = o & ~int64_t(15);
                        int64_t hi = (o + static_cast<int64_t>(ns) * p.bb + 15) & ~int64_t(15);
                        const int64_t t16 = p.total_bytes & ~int64_t(15);
                        if (hi > t16) {
                            hi = t16;
                            tail_len = static_cast<int>(o + static_cast<int64_t>(ns) * p.bb - t16);
                            tail_src = p.W + t16;
                            tail_dst = st + rr * p.row_pitch + static_cast<uint32_t>(t16 - lo);
                        }
                        const int64_t end = o + static_cast<int64_t>(ns) * p.bb;
                        if (in_bounds(lo >= 0 && end <= p.total_bytes && (end + 15 - lo) / 16 * 16 <= p.row_pitch,
                                      p.status)) {
                            src[i] = p.W + lo;
                            dst[i] = st + rr * p.row_pitch;
                            nb[i] = static_cast<uint32_t>(hi - lo);
                        } else {
                            tail_len = 0;
                        }
                    }
                    my += nb[i];
                }
                if (tail_len > 0) {
                    uint8_t *gd = gbase + (tail_dst - base);
                    for (int i = 0; i < tail_len; ++i) gd[i] = __ldg(tail_src + i);
                }
                const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, my);
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(qfull(s), total);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (nb[i]) bulk_g2s(dst[i], src[i], nb[i], qfull(s));
            }
            issued = si + 1;
            if (++s == QS) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (*abort_flag) {   // let issued copies land before the CTA's shared memory is released
            for (int si = max(0, issued - QS); si < issued; ++si) (void)mbar_wait(qfull(si % QS), (si / QS) & 1);
        }
    } else if (warp == 9) {
        // ---------------------------------------------------- activation producer
        if (lane == 0) {
            pdl_wait();
            int issued = 0;
            const int nx = (nchunks + p.xk - 1) / p.xk;
            const uint32_t box_bytes = static_cast<uint32_t>(p.n_tile) * 128u;
            int s = 0;
            uint32_t ph = 0;
            for (int xs = 0; xs < nx; ++xs) {
                if (!wait_or_abort(bempty(s), ph ^ 1u, abort_flag, p.status)) break;
                const int nb = min(p.xk, nchunks - xs * p.xk);
                mbar_arrive_expect_tx(bfull(s), nb * box_bytes);
                for (int i = 0; i < nb; ++i)
                    tma_load_2d(b_ring + s * p.b_stage_bytes + i * box_bytes, &xmap, (xs * p.xk + i) * kChunkK, t0,
                                bfull(s));
                issued = xs + 1;
                if (++s == BS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (*abort_flag) {
                for (int c = max(0, issued - BS); c < issued; ++c) (void)mbar_wait(bfull(c % BS), (c / BS) & 1);
            }
        }
    } else {
        // ---------------------------------------------------- MMA issuer (warp 10)
        // The whole warp runs the loop on warp-uniform values and one elected lane (always
        // lane 0 of the converged warp, so the commits track its MMAs) issues. Measured on
        // GB300 beside eight ALU-bound warps: an n = 32 MMA issues every ~35 cycles this way
        // against ~85 from a branch that only lane 0 enters.
        const uint32_t idesc = idesc_f16_f32(kRows, p.n_tile);
        bool ok = true;
        const uint32_t box_bytes = static_cast<uint32_t>(p.n_tile) * 128u;
        int sa = 0, sbb = 0;   // A slot, x stage
        uint32_t aph = 0, bph = 0;
        for (int sb = 0; sb < p.nsb && ok; ++sb) {
            ok = __all_sync(0xFFFFFFFFu, wait_or_abort(afull(sa), aph, abort_flag, p.status));
            if (!ok) break;
            tc_fence_after();
            const uint32_t a0 = tmem + p.a_col + sa * kASlotCols;
            const auto issue = [&](auto xk) {
                return mma_superblock<decltype(xk)::value>(tmem, a0, sb == 0, idesc, b_ring, p.b_stage_bytes, box_bytes,
                                                           bfull(0), bempty(0), aempty(sa), BS, sbb, bph, abort_flag,
                                                           p.status);
            };
            ok = p.xk == 4 ? issue(std::integral_constant<int, 4>{})
                 : p.xk == 2 ? issue(std::integral_constant<int, 2>{}) : issue(std::integral_constant<int, 1>{});
            if (++sa == AS) {
                sa = 0;
                aph ^= 1u;
            }
        }
        if (elect_one()) tc_commit(accfull);   // also drains in-flight MMAs on the abort path
        __syncwarp();
        if (!ok) (void)mbar_wait(accfull, 0);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 10) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Split form for one token tile over few row tiles: clusters of k + 1 CTAs, where rank r < k
// (a head) takes superblocks [0, L) of row tile cid k + r and rank k (the tail) the remaining
// [L, nsb) of all k tiles, tile after tile, with tile i's sums in TMEM columns [i n_tile,
// (i+1) n_tile). The roles and hand-offs inside a CTA are those of gemm_kernel; the superblock
// position v of a CTA maps to (row tile, superblock) through counters stepped with v. At the end
// the tail stages each tile's sums in its idle rings and copies them with one bulk
// shared-to-shared copy into that head's receive area, completing on the head's barrier pfull;
// the head adds them after its own (a fixed order, so results are reproducible) and stores y.
// A separate kernel rather than a branch of gemm_kernel: folded into it, the unsplit path ran
// 2% slower (Q4_K M=512, GB300).
template <int TYPE, bool TMA>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_split_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap, const GemmArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t b_ring = base;
    const uint32_t q_ring = base + p.q_off;
    const uint32_t bars = base + p.bar_off;
    const int QS = p.qstages, BS = p.bstages;
    auto qfull = [&](int s) { return bars + 8u * s; };
    auto qempty = [&](int s) { return bars + 8u * (QS + s); };
    auto bfull = [&](int s) { return bars + 8u * (2 * QS + s); };
    auto bempty = [&](int s) { return bars + 8u * (2 * QS + BS + s); };
    auto afull = [&](int s) { return bars + 8u * (2 * QS + 2 * BS + s); };
    auto aempty = [&](int s) { return bars + 8u * (2 * QS + 2 * BS + kMaxASlots + s); };
    const uint32_t accfull = bars + 8u * (2 * QS + 2 * BS + 2 * kMaxASlots);
    const uint32_t pfull = accfull + 8u;   // head: the tail's partial sums have landed in the receive area
    const uint32_t misc_off = p.bar_off + 8u * (2 * QS + 2 * BS + 2 * kMaxASlots + kAccBars);
    const int AS = p.a_slots;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + misc_off);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + misc_off + 4);

    const int crank = static_cast<int>(cluster_rank());
    const bool is_tail = crank == p.k;
    const int tile_c = static_cast<int>(blockIdx.x) / (p.k + 1) * p.k;   // the cluster's first row tile
    const int kk = min(p.k, p.row_tiles - tile_c);                        // row tiles of this cluster
    const int nv = is_tail ? kk * p.tail : (crank < kk ? p.L : 0);        // superblock positions of this CTA
    const int own_tile = tile_c + crank;
    const uint32_t part_bytes = static_cast<uint32_t>(kRows * p.part_stride) * 4u;   // one tile's sums
    // (row tile, superblock) of position v: the superblock advances by one and, in the tail,
    // wraps from nsb to L with the next tile (counters: a division per superblock would cost the
    // issuing warps more than its MMAs)
    const int tile0 = is_tail ? tile_c : own_tile, sb0 = is_tail ? p.L : 0;
    auto step = [&](int &tile, int &sb, int by) {
        sb += by;
        while (is_tail && sb >= p.nsb) {
            sb -= p.tail;
            ++tile;
        }
    };
    const int nchunks = nv * 4;
    if constexpr (kBoundsChecks) {   // rings, barriers, hand-off areas and TMEM columns inside their budgets
        uint32_t dyn;
        asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
        const uint32_t q_end = p.q_off + static_cast<uint32_t>(QS) * p.q_stage_bytes;
        const bool lay = misc_off + 8u + (base - raw) <= dyn && static_cast<uint32_t>(BS) * p.b_stage_bytes <= p.q_off &&
                         q_end <= p.recv_off && p.recv_off + part_bytes <= p.bar_off &&
                         static_cast<uint32_t>(p.k) * part_bytes <= q_end &&
                         p.q_stage_bytes >= kRows * p.row_pitch && p.row_pitch >= static_cast<uint32_t>(p.S * p.bb) &&
                         static_cast<uint32_t>(p.n_tile * p.k) <= p.a_col && AS <= kMaxASlots &&
                         p.a_col + static_cast<uint32_t>(AS) * kASlotCols <= kTmemCols &&
                         p.b_stage_bytes >= static_cast<uint32_t>(p.xk * p.n_tile) * 128u && p.M <= p.n_tile;
        if (!in_bounds(lay, p.status)) return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < QS; ++s) {
            mbar_init(qfull(s), 1);
            mbar_init(qempty(s), p.S == 1 ? kDequantWarps / 2 : kDequantWarps);
        }
        for (int s = 0; s < BS; ++s) {
            mbar_init(bfull(s), 1);
            mbar_init(bempty(s), 1);
        }
        for (int s = 0; s < kMaxASlots; ++s) {
            mbar_init(afull(s), kDequantWarps / 2);
            mbar_init(aempty(s), 1);
        }
        mbar_init(accfull, 1);
        mbar_init(pfull, 1);
        *abort_flag = 0u;
        fence_mbar_init();
        if (!is_tail && crank < kk) mbar_arrive_expect_tx(pfull, part_bytes);   // the one arrival; the copy brings the bytes
    }
    if (warp == 10) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 9 && lane == 0) prefetch_tmap(&xmap);
    if (TMA && warp == 8 && lane == 0) prefetch_tmap(&wmap);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // every barrier of the cluster is initialised before any copy reaches it
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();

    if (warp < kDequantWarps) {
        // ---------------------------------------------------- dequantisers (as in gemm_kernel)
        const int q = warp & 3, par = warp >> 2, h = warp >> 2;
        const int r = 32 * q + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const int lg_s = __ffs(p.S) - 1;
        bool ok = true;
        for (int v = par; v < nv && ok; v += 2) {
            // (row tile, superblock) of position v: one division per superblock of decode work
            const int sb = is_tail ? p.L + v % p.tail : v;
            const int row = min((is_tail ? tile_c + v / p.tail : own_tile) * kRows + r, p.N - 1);
            // a stage never spans two row tiles (L and tail are multiples of S)
            const int si = v >> lg_s, j = v & (p.S - 1);
            const int qs = si % QS;
            const uint32_t qph = static_cast<uint32_t>(si / QS) & 1u;
            ok = __all_sync(0xFFFFFFFFu, wait_or_abort(qfull(qs), qph, abort_flag, p.status));
            if (!ok) break;
            const uint32_t stage = q_ring + qs * p.q_stage_bytes;
            uint32_t blk = stage + r * p.row_pitch + j * p.bb;
            if constexpr (!TMA)
                blk += ((static_cast<uint32_t>(row) * static_cast<uint32_t>(p.nsb) + static_cast<uint32_t>(sb - j)) *
                        static_cast<uint32_t>(p.bb)) & 15u;
            if (!in_bounds(blk + static_cast<uint32_t>(p.bb) <= stage + (r + 1) * p.row_pitch, p.status))
                blk = stage + r * p.row_pitch;
            KqRow kr0{}, kr1{};
            if constexpr (TYPE == 12 || TYPE == 13) {
                kr0 = kq_row(blk, 0);
                kr1 = kq_row(blk, 1);
            }
            const int sa = v % AS;
            const uint32_t aph = static_cast<uint32_t>(v / AS) & 1u;
            ok = __all_sync(0xFFFFFFFFu, wait_or_abort(aempty(sa), aph ^ 1u, abort_flag, p.status));
            if (!ok) break;
            tc_fence_after();
            const uint32_t acol = tmem + lane_base + p.a_col + sa * kASlotCols;
            dequant_superblock<TYPE, 0>(blk, kr0, acol);
            dequant_superblock<TYPE, 1>(blk, kr1, acol + 16);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(afull(sa));
                if ((v + 2) >> lg_s != si || v + 2 >= nv) mbar_arrive(qempty(qs));
            }
        }
        // ---------------------------------------------------- epilogue
        if (ok) ok = wait_or_abort(accfull, 0, abort_flag, p.status);
        ok = __all_sync(0xFFFFFFFFu, ok);
        const int ng = p.n_tile / 16, g_mid = ng / 2;
        const int c_lo = 16 * (h ? g_mid : 0), c_hi = 16 * (h ? ng : g_mid);
        if (is_tail) {
            // tile i's sums to rows [i 128, (i+1) 128) of the staging area at the base of shared
            // memory (the rings are idle once the accumulators are final), then one bulk copy per
            // head; sent even after an abort (the heads then see the status word)
            if (ok) {
                tc_fence_after();
                for (int i = 0; i < kk; ++i) {
                    float *part = reinterpret_cast<float *>(gbase) + (i * kRows + r) * p.part_stride;
                    for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
                        uint32_t v[16];
                        tmem_ld16(tmem + lane_base + i * p.n_tile + c0, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; e += 4)
                            *reinterpret_cast<float4 *>(part + c0 + e) =
                                make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                                            __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
                    }
                }
            }
            fence_proxy_async_smem();   // the staged sums, visible to the bulk copies
            named_bar_sync(1, 32 * kDequantWarps);
            if (threadIdx.x == 0) {
                for (int i = 0; i < kk; ++i)
                    bulk_s2s_cluster(mapa_shared(base + p.recv_off, static_cast<uint32_t>(i)), base + i * part_bytes,
                                     part_bytes, mapa_shared(pfull, static_cast<uint32_t>(i)));
            }
        } else if (crank < kk) {
            // head: its own sums (superblocks [0, L)) plus the tail's ([L, nsb)), in that order.
            // The tail's copy is waited for even after an abort (the tail sends it regardless), so
            // that it has landed before this CTA's shared memory is released; the wait is bounded.
            const int n0 = own_tile * kRows;
            const bool landed = mbar_wait(pfull, 0);
            if (!landed && lane == 0) atomicOr(p.status, kStatusTimeout);
            ok = __all_sync(0xFFFFFFFFu, ok && landed);
            const float *part = reinterpret_cast<const float *>(gbase + p.recv_off) + r * p.part_stride;
            if (ok) {
                tc_fence_after();
                for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tmem + lane_base + c0, v);
                    tmem_wait_ld();
                    float acc[16];
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        const float4 t4 = *reinterpret_cast<const float4 *>(part + c0 + e);
                        acc[e] = __uint_as_float(v[e]) + t4.x;
                        acc[e + 1] = __uint_as_float(v[e + 1]) + t4.y;
                        acc[e + 2] = __uint_as_float(v[e + 2]) + t4.z;
                        acc[e + 3] = __uint_as_float(v[e + 3]) + t4.w;
                    }
                    if (n0 + r < p.N) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (c0 + i < p.M) p.y[static_cast<int64_t>(c0 + i) * p.N + n0 + r] = acc[i];
                    }
                }
            }
        }
    } else if (warp == 8) {
        // ---------------------------------------------------- weight producer
        const int nstages = (nv + p.S - 1) / p.S;
        int issued = 0, s = 0;
        int tile = tile0, sb = sb0;   // of the stage's first superblock
        uint32_t ph = 0;
        for (int si = 0; si < nstages; ++si) {
            if (!wait_or_abort(qempty(s), ph ^ 1u, abort_flag, p.status)) break;
            fence_proxy_async_smem();
            const uint32_t st = q_ring + s * p.q_stage_bytes;
            const int n0 = tile * kRows;
            if constexpr (TMA) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(qfull(s), p.q_stage_bytes);
                    tma_load_2d(st, &wmap, sb * (p.bb / 4), n0, qfull(s));
                }
            } else {
                uint32_t my = 0;
                const uint8_t *src[4];
                uint32_t dst[4], nb[4];
                int tail_len = 0;
                uint32_t tail_dst = 0;
                const uint8_t *tail_src = nullptr;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int rr = lane + 32 * i, rowi = n0 + rr;
                    nb[i] = 0;
                    src[i] = nullptr;
                    dst[i] = 0;
                    if (rowi < p.N) {
                        const int64_t o = (static_cast<int64_t>(rowi) * p.nsb + sb) * p.bb;
                        const int64_t lo = o & ~int64_t(15);
                        int64_t hi = (o + static_cast<int64_t>(p.S) * p.bb + 15) & ~int64_t(15);
                        const int64_t t16 = p.total_bytes & ~int64_t(15);
                        if (hi > t16) {
                            hi = t16;
                            tail_len = static_cast<int>(o + static_cast<int64_t>(p.S) * p.bb - t16);
                            tail_src = p.W + t16;
                            tail_dst = st + rr * p.row_pitch + static_cast<uint32_t>(t16 - lo);
                        }
                        const int64_t end = o + static_cast<int64_t>(p.S) * p.bb;
                        if (in_bounds(lo >= 0 && end <= p.total_bytes && (end + 15 - lo) / 16 * 16 <= p.row_pitch,
                                      p.status)) {
                            src[i] = p.W + lo;
                            dst[i] = st + rr * p.row_pitch;
                            nb[i] = static_cast<uint32_t>(hi - lo);
                        } else {
                            tail_len = 0;
                        }
                    }
                    my += nb[i];
                }
                if (tail_len > 0) {
                    uint8_t *gd = gbase + (tail_dst - base);
                    for (int i = 0; i < tail_len; ++i) gd[i] = __ldg(tail_src + i);
                }
                const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, my);
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(qfull(s), total);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (nb[i]) bulk_g2s(dst[i], src[i], nb[i], qfull(s));
            }
            issued = si + 1;
            step(tile, sb, p.S);
            if (++s == QS) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (*abort_flag) {
            for (int si = max(0, issued - QS); si < issued; ++si) (void)mbar_wait(qfull(si % QS), (si / QS) & 1);
        }
    } else if (warp == 9) {
        // ---------------------------------------------------- activation producer
        if (lane == 0) {
            pdl_wait();
            int issued = 0;
            const int nx = (nchunks + p.xk - 1) / p.xk;
            const uint32_t box_bytes = static_cast<uint32_t>(p.n_tile) * 128u;
            int s = 0;
            uint32_t ph = 0;
            int ct = tile0, csb = sb0, cq = 0;   // position and k chunk of the next chunk
            for (int xs = 0; xs < nx; ++xs) {
                if (!wait_or_abort(bempty(s), ph ^ 1u, abort_flag, p.status)) break;
                const int nb = min(p.xk, nchunks - xs * p.xk);
                mbar_arrive_expect_tx(bfull(s), nb * box_bytes);
                for (int i = 0; i < nb; ++i) {
                    tma_load_2d(b_ring + s * p.b_stage_bytes + i * box_bytes, &xmap, (4 * csb + cq) * kChunkK, 0, bfull(s));
                    if (++cq == 4) {
                        cq = 0;
                        step(ct, csb, 1);
                    }
                }
                issued = xs + 1;
                if (++s == BS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (*abort_flag) {
                for (int c = max(0, issued - BS); c < issued; ++c) (void)mbar_wait(bfull(c % BS), (c / BS) & 1);
            }
        }
    } else {
        // ---------------------------------------------------- MMA issuer (warp 10)
        const uint32_t idesc = idesc_f16_f32(kRows, p.n_tile);
        bool ok = true;
        const uint32_t box_bytes = static_cast<uint32_t>(p.n_tile) * 128u;
        int sa = 0, sbb = 0;
        uint32_t aph = 0, bph = 0;
        int vt = 0, first = 0;   // tile of position v among the cluster's tiles (tail), v's index in that tile
        for (int v = 0; v < nv && ok; ++v) {
            ok = __all_sync(0xFFFFFFFFu, wait_or_abort(afull(sa), aph, abort_flag, p.status));
            if (!ok) break;
            tc_fence_after();
            const uint32_t a0 = tmem + p.a_col + sa * kASlotCols;
            const uint32_t d = tmem + static_cast<uint32_t>(vt * p.n_tile);   // the first superblock of a tile overwrites
            const auto issue = [&](auto xk) {
                return mma_superblock<decltype(xk)::value>(d, a0, first == 0, idesc, b_ring, p.b_stage_bytes, box_bytes,
                                                           bfull(0), bempty(0), aempty(sa), BS, sbb, bph, abort_flag,
                                                           p.status);
            };
            ok = p.xk == 4 ? issue(std::integral_constant<int, 4>{})
                 : p.xk == 2 ? issue(std::integral_constant<int, 2>{}) : issue(std::integral_constant<int, 1>{});
            if (++sa == AS) {
                sa = 0;
                aph ^= 1u;
            }
            if (++first == p.tail && is_tail) {
                first = 0;
                ++vt;
            }
        }
        if (elect_one()) tc_commit(accfull);
        __syncwarp();
        if (!ok) (void)mbar_wait(accfull, 0);
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // the tail's staging area stays until every head has its copy
    if (warp == 10) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------------ host side

namespace {

// Token tile: a multiple of 16 in [32, 256] minimising the estimated makespan, i.e. waves of
// CTAs (row tiles x token tiles over the SMs) times the per-superblock time of one CTA, which
// is the larger of its MMA time (8 n cycles: 16 MMAs of 128 x n x 16) and the time of its
// dequantisers (about 1200 cycles, independent of n).
int pick_n_tile(int64_t M, int64_t N, int num_sms) {
    const int64_t row_tiles = (N + kRows - 1) / kRows;
    int best = 32;
    int64_t best_cost = INT64_MAX;
    for (int n = 32; n <= 256; n += 16) {
        const int64_t ntok = (M + n - 1) / n;
        if (n > 32 && (ntok - 1) * n >= M) continue;   // a smaller tile covers M as well
        const int64_t waves = (row_tiles * ntok + num_sms - 1) / num_sms;
        const int64_t cost = waves * std::max<int64_t>(8 * n, 1200);
        if (cost < best_cost) {   // ties keep the smaller tile (less padding)
            best = n;
            best_cost = cost;
        }
    }
    return best;
}

// Superblocks per weight stage for the tensor-copy path, and whether the weights take it: whole
// rows and stages must be 16-byte multiples (Q6_K's 210-byte blocks take per-row bulk copies).
int tma_stage(int bb, int64_t K) {
    const int64_t nsb = K / 256;
    return (bb % 16 == 0) ? 1 : ((2 * bb) % 16 == 0 && nsb % 2 == 0) ? 2 : 1;
}
bool block_tma(int type, int bb, int64_t K) {
    const int64_t nsb = K / 256;
    return ((nsb * bb) % 16 == 0) && ((tma_stage(bb, K) * bb) % 16 == 0) && type != 14;
}

struct GemmPlan {
    int n_tile, qstages, bstages, S, xk, a_slots;
    uint32_t a_col;
    bool tma;
    uint32_t row_pitch, q_stage_bytes, b_stage_bytes, q_off, recv_off, bar_off;
    size_t smem;
    int k, L, tail;   // work split (k > 0): clusters of k heads and one tail CTA
};

// `reserve`: bytes of shared memory kept between the weight ring and the barriers (a split
// plan's receive area, at recv_off); `n_tile` > 0 fixes the token tile.
GemmPlan gemm_plan(int type, int bb, int64_t N, int64_t K, int64_t M, int num_sms, uint32_t reserve = 0, int n_tile = 0) {
    GemmPlan pl{};
    pl.n_tile = n_tile > 0 ? n_tile : pick_n_tile(M, N, num_sms);
    const int s_tma = tma_stage(bb, K);
    pl.tma = block_tma(type, bb, K);
    // activation stages of about 32 KB: 1, 2 or 4 chunks of 64 columns
    pl.xk = pl.n_tile >= 256 ? 1 : pl.n_tile >= 128 ? 2 : 4;
    pl.b_stage_bytes = static_cast<uint32_t>(pl.n_tile) * 128u * pl.xk;
    // TMEM: accumulator columns [0, n_tile), A ring after it in 128-column superblock slots
    pl.a_col = pl.n_tile > 128 ? 256u : 128u;
    pl.a_slots = static_cast<int>((kTmemCols - pl.a_col) / kASlotCols);
    const size_t limit = 227 * 1024 - 1024;
    // Superblocks per weight stage: fixed by the tensor copy's box for TMA types; for rows
    // copied one bulk copy each, as many as fit (up to 4), since the copy engine's cost is
    // per copy and a stage of S superblocks needs 128 copies.
    const int s_cands[3] = {4, 2, 1};
    for (int ci = 0; ci < 3; ++ci) {
        const int S = pl.tma ? s_tma : s_cands[ci];
        if (pl.tma && ci > 0) break;
        uint32_t pitch;
        if (pl.tma) {
            pitch = static_cast<uint32_t>(S * bb);   // dense rows as the tensor copy lands them
        } else {   // window of the span incl. misalignment, an odd multiple of 16 bytes
            pitch = static_cast<uint32_t>((S * bb + 30) & ~15);
            if ((pitch / 16) % 2 == 0) pitch += 16;
        }
        const uint32_t q_stage_bytes = kRows * pitch;
        for (int bs = 4; bs >= 2; --bs) {
            for (int qs = 8; qs >= 2; --qs) {
                const size_t q_off = static_cast<size_t>(bs) * pl.b_stage_bytes;
                const size_t recv_off = (q_off + static_cast<size_t>(qs) * q_stage_bytes + 15) & ~size_t(15);
                const size_t bar_off = recv_off + reserve;
                const size_t total = bar_off + 8 * (2 * qs + 2 * bs + 2 * kMaxASlots + kAccBars) + 16;
                if (total <= limit) {
                    pl.S = S;
                    pl.row_pitch = pitch;
                    pl.q_stage_bytes = q_stage_bytes;
                    pl.bstages = bs;
                    pl.qstages = qs;
                    pl.q_off = static_cast<uint32_t>(q_off);
                    pl.recv_off = static_cast<uint32_t>(recv_off);
                    pl.bar_off = static_cast<uint32_t>(bar_off);
                    pl.smem = total + 1024;   // slack for 1024-byte alignment of the base
                    return pl;
                }
            }
        }
    }
    pl.n_tile = 0;
    return pl;
}

// The kernel for (type, tma), its shared-memory limit raised once per device.
template <int TYPE, bool TMA, bool SPLIT>
const void *kernel_t() {
    const void *f = SPLIT ? reinterpret_cast<const void *>(gemm_split_kernel<TYPE, TMA>)
                          : reinterpret_cast<const void *>(gemm_kernel<TYPE, TMA>);
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
            return nullptr;
        attr_set[dev] = true;
    }
    return f;
}

template <int TYPE>
const void *kernel_type(bool tma, bool split) {
    return tma ? (split ? kernel_t<TYPE, true, true>() : kernel_t<TYPE, true, false>())
               : (split ? kernel_t<TYPE, false, true>() : kernel_t<TYPE, false, false>());
}

const void *kernel_of(int type, bool tma, bool split) {
    switch (type) {
    case 12: return kernel_type<12>(tma, split);
    case 13: return kernel_type<13>(tma, split);
    case 14: return kernel_type<14>(tma, split);
    case kQ6KAligned: return kernel_type<kQ6KAligned>(tma, split);
    case 23: return kernel_type<23>(tma, split);
    default: return nullptr;
    }
}

// How many clusters of `csize` CTAs of this kernel can be resident at once (clusters are
// placed within one GPC, so this can be below SMs / csize); cached per device and size.
int cluster_capacity(const void *f, int csize, size_t smem) {
    struct Entry {
        int dev;
        const void *f;
        int csize;
        size_t smem;
        int n;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> g(mu);
        for (const Entry &e : cache)
            if (e.dev == dev && e.f == f && e.csize == csize && e.smem == smem) return e.n;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(csize));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(csize);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, f, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;   // no split
    }
    std::lock_guard<std::mutex> g(mu);
    cache.push_back({dev, f, csize, smem, n});
    return n;
}

// Work split for one token tile whose T row tiles leave SMs idle: clusters of k heads and one
// tail; a head takes superblocks [0, L) of its row tile and the tail the remaining
// tail = nsb - L of all k tiles (k divides T), so a CTA's share is max(L, k tail) superblocks against nsb
// unsplit. Both L and tail are multiples of the weight stage S (no stage spans two tiles); the
// tail's k accumulators fit below the A ring and its hand-off area below the barriers. Taken
// when it saves more than one superblock per CTA (the hand-off costs about that).
template <class Cap>
void pick_split(GemmPlan &pl, int64_t M, int64_t N, int64_t nsb, int num_sms, Cap cap) {
    pl.k = 0;
    const int64_t T = (N + kRows - 1) / kRows;
    if (M > pl.n_tile || T >= num_sms) return;
    int64_t best = nsb - 1;
    for (int k = 1; k <= kMaxSplitK; ++k) {
        const uint32_t acc_cols = static_cast<uint32_t>(k * pl.n_tile);
        const uint32_t a_col = std::max<uint32_t>(pl.a_col, (acc_cols + kASlotCols - 1) / kASlotCols * kASlotCols);
        if (a_col + 2 * kASlotCols > kTmemCols) break;
        if (static_cast<size_t>(k) * kRows * (pl.n_tile + 4) * 4 > pl.recv_off) break;   // the tail's staging area
        const int64_t clusters = T / k;   // whole clusters only (every head has a tile)
        if (T % k != 0 || clusters * (k + 1) > num_sms) continue;
        for (int64_t tail = pl.S; tail < nsb; tail += pl.S) {
            const int64_t L = nsb - tail, cost = std::max<int64_t>(L, k * tail);
            if (cost < best && clusters <= cap(k + 1)) {
                best = cost;
                pl.k = k;
                pl.L = static_cast<int>(L);
                pl.tail = static_cast<int>(tail);
            }
        }
    }
    if (pl.k > 0) {
        pl.a_col = std::max<uint32_t>(pl.a_col, (static_cast<uint32_t>(pl.k * pl.n_tile) + kASlotCols - 1) / kASlotCols *
                                                    kASlotCols);
        pl.a_slots = static_cast<int>(std::min<uint32_t>((kTmemCols - pl.a_col) / kASlotCols, kMaxASlots));
    }
}

// The launch plan: the unsplit plan, or, for M <= 256, the split form with all M tokens in one
// tile (a multiple of 16, at least 32) and a row tile's superblocks shared by a cluster, where
// every CTA keeps a receive area for one tile's partial sums. The split form is taken when its
// estimate beats the unsplit one, whose token tiles each decode every weight again (costs as in
// pick_n_tile, plus one superblock for the hand-off). `cap(csize, smem)`: resident clusters.
template <class Cap>
GemmPlan choose_plan(int type, int bb, int64_t N, int64_t K, int64_t M, int sms, Cap cap) {
    GemmPlan pl = gemm_plan(type, bb, N, K, M, sms);
    if (pl.n_tile == 0 || M > 256) return pl;
    const int n1 = static_cast<int>(std::max<int64_t>(32, (M + 15) / 16 * 16));
    GemmPlan ps = gemm_plan(type, bb, N, K, M, sms, static_cast<uint32_t>(kRows * (n1 + 4) * 4), n1);
    if (ps.n_tile != n1) return pl;
    pick_split(ps, M, N, K / 256, sms, [&](int csize) { return cap(csize, ps.smem); });
    const int64_t T = (N + kRows - 1) / kRows, ntok = (M + pl.n_tile - 1) / pl.n_tile;
    const int64_t cost_plain = (T * ntok + sms - 1) / sms * (K / 256) * std::max<int64_t>(8 * pl.n_tile, 1200);
    const int64_t cost_split = (std::max<int64_t>(ps.L, static_cast<int64_t>(ps.k) * ps.tail) + 1) *
                               std::max<int64_t>(8 * n1, 1200);
    return ps.k > 0 && cost_split < cost_plain ? ps : pl;
}

}  // namespace

int gemm_launch_count(int, int64_t, int64_t, int64_t) { return 1; }

// The plan gemm_launch makes, without a device: num_sms SMs and caps[i] resident clusters of
// i + 2 CTAs (i = 0..6; null: none). out[14] = {n_tile, k, L, tail, S, xk, a_col, a_slots,
// recv_off, bar_off, grid_x, grid_y, cluster size, dynamic shared memory bytes}; k = 0 is the
// unsplit kernel (one CTA per row tile and token tile). 0, or -1 for an unknown type, -7 when
// no plan fits.
int gemm_plan_info(int type, int64_t N, int64_t K, int64_t M, int num_sms, const int *caps, int64_t *out) {
    const int bb = block_bytes_of(type);
    if (bb < 0) return -1;
    const GemmPlan pl = choose_plan(type, bb, N, K, M, num_sms, [&](int csize, size_t) {
        return caps != nullptr && csize >= 2 && csize <= 8 ? caps[csize - 2] : 0;
    });
    if (pl.n_tile == 0) return -7;
    const int64_t T = (N + kRows - 1) / kRows;
    const int64_t v[14] = {pl.n_tile,
                           pl.k,
                           pl.L,
                           pl.tail,
                           pl.S,
                           pl.xk,
                           pl.a_col,
                           pl.a_slots,
                           pl.recv_off,
                           pl.bar_off,
                           pl.k > 0 ? (T + pl.k - 1) / pl.k * (pl.k + 1) : T,
                           pl.k > 0 ? 1 : (M + pl.n_tile - 1) / pl.n_tile,
                           pl.k > 0 ? pl.k + 1 : 1,
                           static_cast<int64_t>(pl.smem)};
    for (int i = 0; i < 14; ++i) out[i] = v[i];
    return 0;
}

cudaError_t gemm_launch(int type, const uint8_t *W, const __half *x, float *y, int64_t N, int64_t K, int64_t M,
                        unsigned *status, int num_sms, bool pdl, cudaStream_t stream) {
    const int bb = block_bytes_of(type);
    if (bb < 0) return cudaErrorInvalidValue;
    const int sms = num_sms > 0 ? num_sms : 148;
    const void *kern_split = kernel_of(type, block_tma(type, bb, K), true);
    if (kern_split == nullptr) return cudaErrorInvalidValue;
    const GemmPlan pl = choose_plan(type, bb, N, K, M, sms, [&](int csize, size_t smem) {
        return cluster_capacity(kern_split, csize, smem);
    });
    if (pl.n_tile == 0) return cudaErrorNotSupported;
    const void *kern = pl.k > 0 ? kern_split : kernel_of(type, pl.tma, false);
    if (kern == nullptr) return cudaErrorInvalidValue;
    CUtensorMap xmap{}, wmap{};
    if (!encode_tmap_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                        static_cast<uint64_t>(K) * 2, kChunkK, static_cast<uint32_t>(pl.n_tile), true))
        return cudaErrorNotSupported;
    if (pl.tma) {
        const uint64_t row_words = static_cast<uint64_t>(K / 256) * bb / 4;
        if (!encode_tmap_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, W, row_words, static_cast<uint64_t>(N), row_words * 4,
                            static_cast<uint32_t>(pl.S * bb / 4), kRows, false))
            return cudaErrorNotSupported;
    }

    GemmArgs a{};
    a.W = W;
    a.y = y;
    a.status = status;
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.M = static_cast<int>(M);
    a.nsb = static_cast<int>(K / 256);
    a.n_tile = pl.n_tile;
    a.S = pl.S;
    a.row_pitch = pl.row_pitch;
    a.qstages = pl.qstages;
    a.bstages = pl.bstages;
    a.xk = pl.xk;
    a.a_slots = pl.a_slots;
    a.a_col = pl.a_col;
    a.q_stage_bytes = pl.q_stage_bytes;
    a.b_stage_bytes = pl.b_stage_bytes;
    a.q_off = pl.q_off;
    a.bar_off = pl.bar_off;
    a.total_bytes = N * (K / 256) * bb;
    a.bb = bb;
    a.type = type;
    a.row_tiles = static_cast<int>((N + kRows - 1) / kRows);
    a.k = pl.k;
    a.L = pl.L;
    a.tail = pl.tail;
    a.part_stride = pl.n_tile + 4;
    a.recv_off = pl.recv_off;
    const dim3 grid = pl.k > 0 ? dim3(static_cast<unsigned>((a.row_tiles + pl.k - 1) / pl.k * (pl.k + 1)))
                               : dim3(static_cast<unsigned>(a.row_tiles), static_cast<unsigned>((M + pl.n_tile - 1) / pl.n_tile));
    void *args[] = {&xmap, &wmap, &a};
    if (pl.k == 0) return launch_pdl(kern, grid, dim3(kThreads), pl.smem, stream, pdl, args);
    cudaLaunchConfig_t cfg{};   // clusters of k + 1 CTAs along x
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(pl.k + 1);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace ql
