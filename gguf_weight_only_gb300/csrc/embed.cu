// embed.cu -- embedding gather from a GGUF-quantized table: out[m, :] = dequant(W)[ids[m], :].
//
// One CTA of 256 threads per (token, group of superblocks); thread i decodes weight i of each
// superblock of the group straight from global memory (the block's bytes are shared by the
// CTA's threads through L1). Every weight is formed exactly in fp64 (an fp16 scale times small
// integers) and rounded once to the output type, fp32 or fp16 (the pages' embedding returns
// fp16: test/unit/test_llm_quant_cpu.py, test_q4_embedding_matches_reference).
//
// Block formats (ggml), weight i of a 256-weight superblock, j = i / 32:
//   Q4_K / Q5_K: w = d * sc_j * q - dmin * m_j; (sc, m) from the 12-byte packed 6-bit field;
//                q = nibble of qs[32 (i / 64) + i % 32] (low for i % 64 < 32), plus for Q5_K
//                16 * bit j of qh[i % 32].
//   Q6_K:        w = d * sc[i / 16] * (q - 32); low 4 bits from ql[64 h + l + 32 (t % 2)]
//                (low nibble for t < 2), high 2 bits = bits 2t, 2t+1 of qh[32 h + l], with
//                h = i / 128, t = (i % 128) / 32, l = i % 32.
//   IQ4_XS:      w = d * (ls_j - 32) * kv[nibble], ls_j 6-bit from scales_l / scales_h, nibble
//                of qs[16 j + i % 16] (low for i % 32 < 16), kv the 16-entry codebook.
#include <cstdint>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace ql {

namespace {

constexpr int kEmbedSbPerCta = 4;   // superblocks of one row per CTA

// IQ4_XS codebook (test/unit/test_llm_quant_cpu.py, test_unpack_lut_dot_uop)
__constant__ int8_t kIq4Kv[16] = {-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113};

__device__ __forceinline__ double half_at(const uint8_t *p) {
    return static_cast<double>(__half2float(__ushort_as_half(static_cast<unsigned short>(p[0] | (p[1] << 8)))));
}

// The exact weight i of the superblock at blk (every product below is exact in fp64).
template <int TYPE>
__device__ __forceinline__ double weight_at(const uint8_t *blk, int i) {
    if constexpr (TYPE == 12 || TYPE == 13) {
        const uint8_t *S = blk + 4;
        const int j = i >> 5;
        int sc, m;
        if (j < 4) {
            sc = S[j] & 63;
            m = S[j + 4] & 63;
        } else {
            sc = (S[j + 4] & 15) | ((S[j - 4] >> 6) << 4);
            m = (S[j + 4] >> 4) | ((S[j] >> 6) << 4);
        }
        const int qoff = (TYPE == 13) ? 48 : 16;
        const int byte = blk[qoff + 32 * (i >> 6) + (i & 31)];
        int q = ((i & 63) < 32) ? (byte & 15) : (byte >> 4);
        if constexpr (TYPE == 13) q += 16 * ((blk[16 + (i & 31)] >> j) & 1);
        return half_at(blk) * static_cast<double>(sc * q) - half_at(blk + 2) * static_cast<double>(m);
    } else if constexpr (TYPE == 14) {
        const int h = i >> 7, r = i & 127, t = r >> 5, l = r & 31;
        const int lb = blk[64 * h + l + 32 * (t & 1)];
        const int lo = (t < 2) ? (lb & 15) : (lb >> 4);
        const int hi = (blk[128 + 32 * h + l] >> (2 * t)) & 3;
        const int sc = static_cast<int8_t>(blk[192 + (i >> 4)]);
        return half_at(blk + 208) * static_cast<double>(sc * ((lo | (hi << 4)) - 32));
    } else {
        const int j = i >> 5, r = i & 31;
        const int scales_h = blk[2] | (blk[3] << 8);
        const int ls = ((blk[4 + (j >> 1)] >> (4 * (j & 1))) & 15) | (((scales_h >> (2 * j)) & 3) << 4);
        const int byte = blk[8 + 16 * j + (r & 15)];
        const int nib = (r < 16) ? (byte & 15) : (byte >> 4);
        return half_at(blk) * static_cast<double>((ls - 32) * kIq4Kv[nib]);
    }
}

__device__ __forceinline__ void put(float *o, double w) { *o = __double2float_rn(w); }
__device__ __forceinline__ void put(__half *o, double w) { *o = __double2half(w); }   // round to nearest even

template <int TYPE, int BB, typename T>
__global__ void __launch_bounds__(256) embed_kernel(const uint8_t *__restrict__ W, const int32_t *__restrict__ ids,
                                                    int64_t N, int nsb, T *__restrict__ out, unsigned *status) {
    const int m = blockIdx.y;
    const int id = ids[m];
    const int i = threadIdx.x;
    const int64_t K = static_cast<int64_t>(nsb) * 256;
    T *row = out + m * K;
    const int sb0 = blockIdx.x * kEmbedSbPerCta, sb1 = min(sb0 + kEmbedSbPerCta, nsb);
    if (id < 0 || id >= N) {   // bad index: zeros, and the status word records it
        for (int sb = sb0; sb < sb1; ++sb) put(row + sb * 256 + i, 0.0);
        if (i == 0 && blockIdx.x == 0) atomicOr(status, kStatusBadIndex);
        return;
    }
    const uint8_t *rowW = W + static_cast<int64_t>(id) * nsb * BB;
    for (int sb = sb0; sb < sb1; ++sb) put(row + sb * 256 + i, weight_at<TYPE>(rowW + static_cast<int64_t>(sb) * BB, i));
}

template <int TYPE, int BB>
cudaError_t launch(const uint8_t *W, const int32_t *ids, int64_t N, int64_t K, int64_t M, void *out, bool half_out,
                   unsigned *status, cudaStream_t st) {
    const int nsb = static_cast<int>(K / 256);
    const dim3 grid((nsb + kEmbedSbPerCta - 1) / kEmbedSbPerCta, static_cast<unsigned>(M));
    if (half_out)
        embed_kernel<TYPE, BB, __half><<<grid, 256, 0, st>>>(W, ids, N, nsb, static_cast<__half *>(out), status);
    else
        embed_kernel<TYPE, BB, float><<<grid, 256, 0, st>>>(W, ids, N, nsb, static_cast<float *>(out), status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t embed_launch(int type, const uint8_t *W, const int32_t *ids, int64_t N, int64_t K, int64_t M, void *out,
                         bool half_out, unsigned *status, cudaStream_t stream) {
    if (M < 1) return cudaErrorInvalidValue;
    const int64_t esz = half_out ? 2 : 4;
    for (int64_t m0 = 0; m0 < M; m0 += 65535) {   // the grid's y extent is at most 65535 tokens
        const int64_t mc = M - m0 < 65535 ? M - m0 : 65535;
        void *o = static_cast<char *>(out) + m0 * K * esz;
        cudaError_t e;
        switch (type) {
        case 12: e = launch<12, 144>(W, ids + m0, N, K, mc, o, half_out, status, stream); break;
        case 13: e = launch<13, 176>(W, ids + m0, N, K, mc, o, half_out, status, stream); break;
        case 14: e = launch<14, 210>(W, ids + m0, N, K, mc, o, half_out, status, stream); break;
        case kQ6KAligned: e = launch<14, 224>(W, ids + m0, N, K, mc, o, half_out, status, stream); break;
        case 23: e = launch<23, 136>(W, ids + m0, N, K, mc, o, half_out, status, stream); break;
        default: return cudaErrorInvalidValue;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int embed_launch_count(int64_t M) { return static_cast<int>((M + 65534) / 65535); }

namespace {

// One thread per 2-byte word of the aligned layout: words 0..104 of each 224-byte block come
// from the 210-byte source block, words 105..111 are zero.
__global__ void repack_q6k_kernel(const uint16_t *__restrict__ src, uint16_t *__restrict__ dst, int64_t nblocks) {
    const int64_t total = nblocks * 112;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = i / 112;
        const int w = static_cast<int>(i - b * 112);
        dst[i] = w < 105 ? src[b * 105 + w] : static_cast<uint16_t>(0);
    }
}

}  // namespace

cudaError_t repack_q6k_aligned(const uint8_t *W_src, int64_t N, int64_t K, uint8_t *W_dst, cudaStream_t stream) {
    const int64_t nblocks = N * (K / 256);
    const int64_t total = nblocks * 112;
    const int threads = 256;
    const int64_t want = (total + threads - 1) / threads;
    const unsigned grid = static_cast<unsigned>(want < 152 * 32 ? want : 152 * 32);
    repack_q6k_kernel<<<grid, threads, 0, stream>>>(reinterpret_cast<const uint16_t *>(W_src),
                                                    reinterpret_cast<uint16_t *>(W_dst), nblocks);
    return cudaGetLastError();
}

}  // namespace ql
