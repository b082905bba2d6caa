// kernels.h -- internal interface between the C ABI (qlinear_api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace ql {

// ---------------------------------------------------------------- decode GEMV (gemv.cu)

struct GemvArgs {
    const uint8_t *W;
    const __half *x;
    float *y;
    unsigned *status;
    int N, K, M;          // M <= 8
    int nsb;              // K / 256
    int sb_per_warp;      // contiguous superblocks per warp
    int stages;           // ring depth per warp
    uint32_t row_pitch;   // bytes per weight row in a stage (multiple of 16)
    uint32_t stage_bytes; // 16 * row_pitch + M * 576
    uint32_t warp_bytes;  // stages * stage_bytes
    uint32_t red_offset;  // byte offset of the reduction area in dynamic shared memory
    uint32_t region_offset;
    int64_t total_bytes;  // size of W in bytes
};

struct GemvPlan {
    int warps, stages, sb_per_warp, grid;
    uint32_t row_pitch, stage_bytes, warp_bytes, red_offset, region_offset;
    size_t smem;
};

constexpr int kGemvMaxM = 8;

int gemv_block_bytes(int type);
GemvPlan gemv_plan(int type, int64_t N, int64_t K, int M, int num_sms);
cudaError_t gemv_launch(int type, const uint8_t *W, const __half *x, float *y, int64_t N, int64_t K, int M,
                        unsigned *status, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- prefill GEMM (gemm_tc.cu)

// Launches the tcgen05 kernel for any M >= 1. Returns cudaErrorNotSupported when the shape
// cannot be handled (the caller maps it to QL_ERR_UNSUPPORTED).
cudaError_t gemm_launch(int type, const uint8_t *W, const __half *x, float *y, int64_t N, int64_t K, int64_t M,
                        unsigned *status, int num_sms, cudaStream_t stream);
int gemm_launch_count(int type, int64_t N, int64_t K, int64_t M);

}  // namespace ql
