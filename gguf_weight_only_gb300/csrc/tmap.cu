// tmap.cu -- host-side helpers: encoding of TMA tensor maps through the driver entry point
// (no link-time dependency on libcuda) and kernel launches with programmatic dependent launch.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.h"

namespace ql {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}
}  // namespace

bool encode_tmap_2d(void *tmap_out, int dtype, const void *base, uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes,
                    uint32_t box0, uint32_t box1, bool swizzle128) {
    auto enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t gdim[2] = {dim0, dim1};
    const cuuint64_t gstride[1] = {stride1_bytes};
    const cuuint32_t box[2] = {box0, box1};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(static_cast<CUtensorMap *>(tmap_out), static_cast<CUtensorMapDataType>(dtype), 2,
                           const_cast<void *>(base), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int block_bytes_of(int type) {
    switch (type) {
    case 12: return 144;
    case 13: return 176;
    case 14: return 210;
    case 270: return 224;   // Q6_K in 16-byte aligned blocks (qlinear_repack)
    case 23: return 136;
    default: return -1;
    }
}

}  // namespace ql

namespace ql {

bool encode_tmap_3d(void *tmap_out, int dtype, const void *base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                    uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1, uint32_t box2,
                    bool swizzle128) {
    auto enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t gdim[3] = {dim0, dim1, dim2};
    const cuuint64_t gstride[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {box0, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(static_cast<CUtensorMap *>(tmap_out), static_cast<CUtensorMapDataType>(dtype), 3,
                           const_cast<void *>(base), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace ql

namespace ql {

cudaError_t launch_pdl(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl, void **args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, func, args);
}

}  // namespace ql
