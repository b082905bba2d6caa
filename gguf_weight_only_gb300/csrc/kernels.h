// kernels.h -- internal interface between the C ABI (qlinear_api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace ql {

// Bytes per 256-weight superblock of a ggml type id (Q4_K 144, Q5_K 176, Q6_K 210,
// IQ4_XS 136; the aligned Q6_K layout 270: 224), or -1.
int block_bytes_of(int type);

// Q6_K repacked into 224-byte blocks: each 210-byte block followed by 14 zero bytes, so every
// block and row starts on a 16-byte boundary. Decoded exactly as Q6_K.
constexpr int kQ6KAligned = 270;

// Rewrites N x K/256 Q6_K blocks (W_src, 210 bytes each) into the aligned layout (W_dst,
// 224 bytes each) on `stream`.
cudaError_t repack_q6k_aligned(const uint8_t *W_src, int64_t N, int64_t K, uint8_t *W_dst, cudaStream_t stream);

// ---------------------------------------------------------------- decode GEMV (gemv.cu)

constexpr int kGemvMaxM = 8;
constexpr int kGemvMaxProj = 4;

// One projection of a multi-projection GEMV: W holds N rows of K/256 superblocks, y is [M, N].
struct GemvProj {
    const uint8_t *W;
    float *y;
    int64_t N;
};

// y[M <= 8, N] = x . dequant(W)^T, one launch. With `pdl` the kernel may start (and stream
// its constant weights) while the preceding kernel in the stream finishes; it reads x and
// writes y only after that kernel has completed.
cudaError_t gemv_launch(int type, const uint8_t *W, const __half *x, float *y, int64_t N, int64_t K, int M,
                        unsigned *status, int num_sms, bool pdl, cudaStream_t stream);

// The streaming decode kernel (gemv_stream.cu): one weight matrix, M <= kGemvMaxM. Every CTA
// owns an equal share of rows, fetched as (16-row tile, K range) units by its warps; the whole
// share is requested before the wait for the preceding kernel when it fits in shared memory.
// Returns cudaErrorNotSupported when x and the weight ring do not fit (gemv_launch then takes
// the persistent kernel below).
cudaError_t gemv_stream_launch(int type, const uint8_t *W, const __half *x, float *y, int64_t N, int64_t K, int M,
                               unsigned *status, int num_sms, bool pdl, cudaStream_t stream);
bool gemv_stream_supported(int type, int64_t N, int64_t K, int M, int num_sms);

// y_j = x . dequant(W_j)^T for nproj <= kGemvMaxProj projections sharing x and K, in one launch:
// the row tiles of all projections form one work list split over the persistent CTAs, and
// each CTA's warps load their slice of x once for all of them.
cudaError_t gemv_launch_multi(int type, int nproj, const GemvProj *proj, const __half *x, int64_t K, int M,
                              unsigned *status, int num_sms, bool pdl, cudaStream_t stream);

// Fused producer of x and consumer of y for one decode launch (M <= kGemvMaxM).
struct GemvFusion {
    int pro = 0;                     // 1: x = fp16(silu(gate) * up); 2: x = fp16(rmsnorm(h) * norm_w)
    const __half *gate = nullptr;    // pro 1: [M, K] fp16
    const float *up_or_h = nullptr;  // pro 1: up [M, K]; pro 2: h [M, K]
    const float *norm_w = nullptr;   // pro 2: [K]
    float eps = 0.f;                 // pro 2
    __half *xnorm = nullptr;         // pro 2: optional [M, K] copy of the fp16 normalised x
    const float *residual = nullptr; // optional [M, N], added to y (may be y)
    unsigned long long *best = nullptr;  // greedy head: per-token packed keys (zeroed), y not written
};
cudaError_t gemv_launch_fused(int type, const uint8_t *W, float *y, int64_t N, int64_t K, int M, const GemvFusion &f,
                              unsigned *status, int num_sms, bool pdl, cudaStream_t stream);

// Greedy output head: index_out[m] = the first n with the largest y[m, n] (int64), value_out[m]
// (optional) = that y, without writing y. index_out serves as the packed-key scratch: it is
// zeroed, reduced into by atomic max from every CTA, then rewritten by a one-warp kernel.
cudaError_t gemv_launch_argmax(int type, const uint8_t *W, int64_t N, int64_t K, const __half *x, int M,
                               long long *index_out, float *value_out, unsigned *status, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- prefill GEMM (gemm_tc.cu)

// Launches the tcgen05 kernel for any M >= 1. Returns cudaErrorNotSupported when the shape
// cannot be handled (the caller maps it to QL_ERR_UNSUPPORTED).
cudaError_t gemm_launch(int type, const uint8_t *W, const __half *x, float *y, int64_t N, int64_t K, int64_t M,
                        unsigned *status, int num_sms, bool pdl, cudaStream_t stream);
int gemm_launch_count(int type, int64_t N, int64_t K, int64_t M);

// ---------------------------------------------------------------- embedding gather (embed.cu)

// out[m, :] = dequant(W)[ids[m], :], the exact weights rounded once to fp32 (or fp16 with
// half_out); an id outside [0, N) gives a zero row and sets kStatusBadIndex in *status.
cudaError_t embed_launch(int type, const uint8_t *W, const int32_t *ids, int64_t N, int64_t K, int64_t M, void *out,
                         bool half_out, unsigned *status, cudaStream_t stream);
int embed_launch_count(int64_t M);

// ---------------------------------------------------------------- tensor maps (tmap.cu)

// Encode a 2-D tiled tensor map (no swizzle unless `swizzle128`); false if the driver
// entry point is unavailable or the encoding is rejected.
bool encode_tmap_2d(void *tmap_out, int dtype /* CUtensorMapDataType */, const void *base, uint64_t dim0,
                    uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1, bool swizzle128);
bool encode_tmap_3d(void *tmap_out, int dtype, const void *base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                    uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1, uint32_t box2,
                    bool swizzle128);

// Launch `func` with its argument pointers, optionally as a programmatic dependent launch.
cudaError_t launch_pdl(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl, void **args);

}  // namespace ql
