// qlinear_api.cu -- the C ABI declared in include/qlinear.h: argument validation, per-device
// state, and dispatch on M between the decode GEMV and the tcgen05 prefill GEMM.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "qlinear.h"

namespace ql {
// gemm_tc.cu: the prefill plan without a device (see qlinear_gemm_plan)
int gemm_plan_info(int type, int64_t N, int64_t K, int64_t M, int num_sms, const int *caps, int64_t *out);
}  // namespace ql

namespace {

// Device status word: kernels OR error bits into it (a bounded wait that ran out, an embedding
// id out of range, a failed bounds check of a QL_DEBUG build). qlinear_device_status takes it
// with an atomic exchange into g_status_taken.
__device__ unsigned g_status_word;
__device__ unsigned g_status_taken;

struct DeviceState {
    bool ready = false;
    int status = QL_OK;       // QL_OK or the error of the failed initialisation
    int dev = 0;
    int num_sms = 0;
    bool pdl = true;          // programmatic dependent launch (QL_PDL=0 disables)
    bool fail_launch = false; // QL_TEST_FAIL=launch: every launch reports a launch error instead
    unsigned *status_word = nullptr;
    unsigned *status_taken = nullptr;
    std::mutex status_mutex;  // one qlinear_device_status at a time per device
};

constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mutex;
thread_local int t_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return QL_ERR_CUDA;
}

// Per-device one-time set-up (SM count, sm_103 check, status-word address), done with
// the device current. Returns QL_OK or an error.
int device_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return QL_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceState &s = g_dev[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        if (major != 10 || minor != 3) {
            s.status = QL_ERR_DEVICE;
        } else {
            void *p = nullptr, *q = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_status_word)) != cudaSuccess) return cuda_fail(e);
            if ((e = cudaGetSymbolAddress(&q, g_status_taken)) != cudaSuccess) return cuda_fail(e);
            s.status_word = static_cast<unsigned *>(p);
            s.status_taken = static_cast<unsigned *>(q);
            s.dev = dev;
            s.num_sms = sms;
            const char *env = std::getenv("QL_PDL");
            s.pdl = !(env && env[0] == '0');
            const char *fail = std::getenv("QL_TEST_FAIL");
            s.fail_launch = fail && std::strcmp(fail, "launch") == 0;
            s.status = QL_OK;
        }
        s.ready = true;
    }
    *out = &s;
    return s.status;
}

// Every pointer a call hands to the kernels must be device (or managed) memory of the current
// device: a pointer of another GPU, or plain host memory, gives QL_ERR_DEVICE before any launch.
int check_on_device(const DeviceState &s, std::initializer_list<const void *> ptrs) {
    for (const void *ptr : ptrs) {
        if (!ptr) continue;
        cudaPointerAttributes at{};
        const cudaError_t e = cudaPointerGetAttributes(&at, ptr);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();   // an unknown pointer: not an error of the context
            return QL_ERR_DEVICE;
        }
        if ((at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) || at.device != s.dev)
            return QL_ERR_DEVICE;
    }
    return QL_OK;
}

// The launch-failure hook of the failure-path tests: with QL_TEST_FAIL=launch in the environment
// (read once per device) a call that would launch returns QL_ERR_CUDA with
// cudaErrorLaunchOutOfResources recorded, and launches nothing.
bool launch_refused(const DeviceState &s) {
    if (!s.fail_launch) return false;
    t_last_cuda_error = static_cast<int>(cudaErrorLaunchOutOfResources);
    return true;
}

// Prefill token tiles go on grid.y (at most 65535) and are at least 32 tokens: larger M is refused.
constexpr int64_t kMaxTokens = int64_t(65535) * 32;

int validate(int type, const void *W, int64_t N, int64_t K, const void *x, int64_t M, const float *y) {
    if (ql::block_bytes_of(type) < 0) return QL_ERR_TYPE;
    if (N < 1 || M < 1 || K < 256 || K % 256 != 0) return QL_ERR_SHAPE;
    // 32-bit indexing limits inside the kernels
    if (N > (int64_t(1) << 30) || K > (int64_t(1) << 24) || M > kMaxTokens) return QL_ERR_SHAPE;
    if (M * K > (int64_t(1) << 40) || M * N > (int64_t(1) << 40)) return QL_ERR_SHAPE;
    if (!W || !x || !y) return QL_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u)
        return QL_ERR_ALIGN;
    return QL_OK;
}

enum class Path { Auto, Gemv, Gemm };

// The status word's value, cleared in the same atomic operation.
__global__ void status_take_kernel(unsigned *word, unsigned *out) { *out = atomicExch(word, 0u); }

// Does nothing: launched the ordinary way (no programmatic dependent launch) it orders the stream.
__global__ void stream_fence_kernel() {}

// qlinear_copy's kernel: 16 bytes per thread and step where both ends are 16-byte aligned, else
// byte by byte. It lets the next kernel launch first and waits for the preceding one before
// touching either buffer.
__global__ void copy_kernel(uint8_t *dst, const uint8_t *src, int64_t bytes) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t head = 0;
    if (((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0) {
        const int64_t n16 = bytes / 16;
        for (int64_t i = tid; i < n16; i += nthr)
            reinterpret_cast<uint4 *>(dst)[i] = reinterpret_cast<const uint4 *>(src)[i];
        head = n16 * 16;
    }
    for (int64_t i = head + tid; i < bytes; i += nthr) dst[i] = src[i];
}

// The address a kernel uses for `ptr`: itself for device (or managed) memory of the current
// device, the mapped device address for page-locked host memory; nullptr for anything else.
void *kernel_address(const DeviceState &s, const void *ptr) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
        (void)cudaGetLastError();   // an unknown pointer: not an error of the context
        return nullptr;
    }
    if ((at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == s.dev)
        return const_cast<void *>(ptr);
    if (at.type == cudaMemoryTypeHost && at.devicePointer != nullptr) return at.devicePointer;
    return nullptr;
}

// One thread waits, with the library's bounded wait, on a barrier phase that never
// completes; when the wait runs out it records the timeout in the status word.
__global__ void wait_timeout_selftest_kernel(unsigned *status) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = ql::smem_u32(&bar);
    if (threadIdx.x == 0) {
        ql::mbar_init(b, 1);
        ql::fence_mbar_init();
        if (!ql::mbar_wait(b, 0)) atomicOr(status, ql::kStatusTimeout);
    }
}

int run_gemv(const DeviceState &s, int type, const void *W, int64_t N, int64_t K, const void *x, int64_t M, float *y,
             cudaStream_t st) {
    // tokens in groups of kGemvMaxM: one launch per group (the weights stream once per group)
    for (int64_t m0 = 0; m0 < M; m0 += ql::kGemvMaxM) {
        const int mg = static_cast<int>(M - m0 < ql::kGemvMaxM ? M - m0 : ql::kGemvMaxM);
        cudaError_t e = ql::gemv_launch(type, static_cast<const uint8_t *>(W),
                                        static_cast<const __half *>(x) + m0 * K, y + m0 * N, N, K, mg,
                                        s.status_word, s.num_sms, s.pdl, st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return QL_OK;
}

int run(Path path, int type, const void *W, int64_t N, int64_t K, const void *x, int64_t M, float *y, void *stream) {
    int rc = validate(type, W, N, K, x, M, y);
    if (rc != QL_OK) return rc;
    DeviceState *s = nullptr;
    if ((rc = device_state(&s)) != QL_OK) return rc;
    if ((rc = check_on_device(*s, {W, x, y})) != QL_OK) return rc;
    if (launch_refused(*s)) return QL_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (path == Path::Gemv || (path == Path::Auto && M <= ql::kGemvMaxM))
        return run_gemv(*s, type, W, N, K, x, M, y, st);
    cudaError_t e = ql::gemm_launch(type, static_cast<const uint8_t *>(W), static_cast<const __half *>(x), y, N, K, M,
                                    s->status_word, s->num_sms, s->pdl, st);
    if (e == cudaErrorNotSupported) return QL_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return cuda_fail(e);
    return QL_OK;
}

// Several projections sharing x: each (W_j, N_j, y_j) is checked like a single call.
int run_multi(int type, int n_proj, const void *const *W, const int64_t *N, int64_t K, const void *x, int64_t M,
              float *const *y, void *stream) {
    if (!W || !N || !y) return QL_ERR_NULL;
    if (n_proj < 1 || n_proj > ql::kGemvMaxProj) return QL_ERR_SHAPE;
    for (int j = 0; j < n_proj; ++j) {
        const int rc = validate(type, W[j], N[j], K, x, M, y[j]);
        if (rc != QL_OK) return rc;
    }
    DeviceState *s = nullptr;
    int rc = device_state(&s);
    if (rc != QL_OK) return rc;
    if ((rc = check_on_device(*s, {x})) != QL_OK) return rc;
    for (int j = 0; j < n_proj; ++j)
        if ((rc = check_on_device(*s, {W[j], y[j]})) != QL_OK) return rc;
    if (launch_refused(*s)) return QL_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (M > ql::kGemvMaxM) {   // prefill: one GEMM per projection
        for (int j = 0; j < n_proj; ++j) {
            cudaError_t e = ql::gemm_launch(type, static_cast<const uint8_t *>(W[j]), static_cast<const __half *>(x),
                                            y[j], N[j], K, M, s->status_word, s->num_sms, s->pdl, st);
            if (e == cudaErrorNotSupported) return QL_ERR_UNSUPPORTED;
            if (e != cudaSuccess) return cuda_fail(e);
        }
        return QL_OK;
    }
    ql::GemvProj proj[ql::kGemvMaxProj];
    for (int j = 0; j < n_proj; ++j) proj[j] = ql::GemvProj{static_cast<const uint8_t *>(W[j]), y[j], N[j]};
    cudaError_t e = ql::gemv_launch_multi(type, n_proj, proj, static_cast<const __half *>(x), K, static_cast<int>(M),
                                          s->status_word, s->num_sms, s->pdl, st);
    return e == cudaSuccess ? QL_OK : cuda_fail(e);
}

bool misaligned(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; }

// A decode launch with a fused prologue (SiLU-gated or RMSNorm x) and optional residual.
int run_fused(int type, const void *W, int64_t N, int64_t K, int64_t M, const ql::GemvFusion &f, const void *a,
              const void *b, float *y, void *stream) {
    int rc = validate(type, W, N, K, a, M, y);   // a: the [M, K] input that stands in for x
    if (rc != QL_OK) return rc;
    if (!b) return QL_ERR_NULL;
    if (misaligned(b) || (f.residual && misaligned(f.residual)) || (f.xnorm && misaligned(f.xnorm))) return QL_ERR_ALIGN;
    if (!(f.eps >= 0.f) || f.eps > 3.0e38f) return QL_ERR_SHAPE;   // also rejects NaN
    if (M > ql::kGemvMaxM) return QL_ERR_UNSUPPORTED;
    DeviceState *s = nullptr;
    if ((rc = device_state(&s)) != QL_OK) return rc;
    if ((rc = check_on_device(*s, {W, a, b, y, f.residual, f.xnorm, f.norm_w})) != QL_OK) return rc;
    if (launch_refused(*s)) return QL_ERR_CUDA;
    cudaError_t e = ql::gemv_launch_fused(type, static_cast<const uint8_t *>(W), y, N, K, static_cast<int>(M), f,
                                          s->status_word, s->num_sms, s->pdl, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return QL_ERR_UNSUPPORTED;
    return e == cudaSuccess ? QL_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

int qlinear(int type, const void *W_blocks, int64_t N, int64_t K, const void *x_fp16, int64_t M, float *y_fp32,
            void *stream) {
    return run(Path::Auto, type, W_blocks, N, K, x_fp16, M, y_fp32, stream);
}

int qlinear_gemv(int type, const void *W_blocks, int64_t N, int64_t K, const void *x_fp16, int64_t M, float *y_fp32,
                 void *stream) {
    return run(Path::Gemv, type, W_blocks, N, K, x_fp16, M, y_fp32, stream);
}

int qlinear_gemm(int type, const void *W_blocks, int64_t N, int64_t K, const void *x_fp16, int64_t M, float *y_fp32,
                 void *stream) {
    return run(Path::Gemm, type, W_blocks, N, K, x_fp16, M, y_fp32, stream);
}

int qlinear_multi(int type, int n_proj, const void *const *W_blocks, const int64_t *N, int64_t K, const void *x_fp16,
                  int64_t M, float *const *y_fp32, void *stream) {
    return run_multi(type, n_proj, W_blocks, N, K, x_fp16, M, y_fp32, stream);
}

int qlinear_max_projections(void) { return ql::kGemvMaxProj; }

int qlinear_repack(int type, const void *W_src, int64_t N, int64_t K, void *W_dst, void *stream) {
    if (type != QL_Q6_K) return QL_ERR_TYPE;
    if (N < 1 || K < 256 || K % 256 != 0 || N > (int64_t(1) << 30) || K > (int64_t(1) << 24)) return QL_ERR_SHAPE;
    if (!W_src || !W_dst) return QL_ERR_NULL;
    if (misaligned(W_src) || misaligned(W_dst)) return QL_ERR_ALIGN;
    DeviceState *s = nullptr;
    int rc = device_state(&s);
    if (rc != QL_OK) return rc;
    if ((rc = check_on_device(*s, {W_src, W_dst})) != QL_OK) return rc;
    if (launch_refused(*s)) return QL_ERR_CUDA;
    cudaError_t e = ql::repack_q6k_aligned(static_cast<const uint8_t *>(W_src), N, K, static_cast<uint8_t *>(W_dst),
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    // The layer kernels read W before their dependency wait (programmatic dependent launch): the
    // kernel right after the repack must not be one of them. An empty kernel launched the ordinary
    // way starts only once the repack has completed and its writes are visible, and a layer call
    // that follows may then start early without seeing W_dst half written.
    stream_fence_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>();
    e = cudaGetLastError();
    return e == cudaSuccess ? QL_OK : cuda_fail(e);
}

int qlinear_copy(void *dst, const void *src, int64_t bytes, void *stream) {
    if (bytes < 0) return QL_ERR_SHAPE;
    if (bytes == 0) return QL_OK;
    if (!dst || !src) return QL_ERR_NULL;
    DeviceState *s = nullptr;
    int rc = device_state(&s);
    if (rc != QL_OK) return rc;
    void *d = kernel_address(*s, dst);
    const void *sp = kernel_address(*s, src);
    if (!d || !sp) return QL_ERR_DEVICE;
    if (launch_refused(*s)) return QL_ERR_CUDA;
    constexpr int kThreadsCopy = 256;
    const int64_t units = (bytes + 15) / 16;
    const int64_t blocks = std::min<int64_t>((units + kThreadsCopy - 1) / kThreadsCopy, int64_t(4) * s->num_sms);
    void *args[] = {&d, const_cast<void **>(&sp), &bytes};
    const cudaError_t e = ql::launch_pdl(reinterpret_cast<const void *>(copy_kernel), dim3(static_cast<unsigned>(blocks)),
                                         dim3(kThreadsCopy), 0, static_cast<cudaStream_t>(stream), s->pdl, args);
    return e == cudaSuccess ? QL_OK : cuda_fail(e);
}

int qlinear_argmax(int type, const void *W_blocks, int64_t N, int64_t K, const void *x_fp16, int64_t M,
                   int64_t *index_out, float *value_out, void *stream) {
    int rc = validate(type, W_blocks, N, K, x_fp16, M, reinterpret_cast<const float *>(index_out));
    if (rc != QL_OK) return rc;
    if (value_out && misaligned(value_out)) return QL_ERR_ALIGN;
    if (M > ql::kGemvMaxM) return QL_ERR_UNSUPPORTED;
    DeviceState *s = nullptr;
    if ((rc = device_state(&s)) != QL_OK) return rc;
    if ((rc = check_on_device(*s, {W_blocks, x_fp16, index_out, value_out})) != QL_OK) return rc;
    if (launch_refused(*s)) return QL_ERR_CUDA;
    cudaError_t e = ql::gemv_launch_argmax(type, static_cast<const uint8_t *>(W_blocks), N, K,
                                           static_cast<const __half *>(x_fp16), static_cast<int>(M),
                                           reinterpret_cast<long long *>(index_out), value_out, s->status_word,
                                           s->num_sms, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return QL_ERR_UNSUPPORTED;
    return e == cudaSuccess ? QL_OK : cuda_fail(e);
}

int qlinear_embed(int type, const void *W_blocks, int64_t N, int64_t K, const int32_t *ids, int64_t M, void *out,
                  int out_fp16, void *stream) {
    if (ql::block_bytes_of(type) < 0) return QL_ERR_TYPE;
    if (N < 1 || M < 1 || K < 256 || K % 256 != 0 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 24) ||
        M > (int64_t(1) << 30))
        return QL_ERR_SHAPE;
    if (!W_blocks || !ids || !out) return QL_ERR_NULL;
    if (misaligned(W_blocks) || misaligned(out) || (reinterpret_cast<uintptr_t>(ids) & 3u)) return QL_ERR_ALIGN;
    DeviceState *s = nullptr;
    int rc = device_state(&s);
    if (rc != QL_OK) return rc;
    if ((rc = check_on_device(*s, {W_blocks, ids, out})) != QL_OK) return rc;
    if (launch_refused(*s)) return QL_ERR_CUDA;
    cudaError_t e = ql::embed_launch(type, static_cast<const uint8_t *>(W_blocks), ids, N, K, M, out, out_fp16 != 0,
                                     s->status_word, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QL_OK : cuda_fail(e);
}

int qlinear_silu_mul(int type, const void *W_blocks, int64_t N, int64_t K, const void *gate_fp16, const float *up_fp32,
                     int64_t M, const float *residual, float *y_fp32, void *stream) {
    ql::GemvFusion f;
    f.pro = 1;
    f.gate = static_cast<const __half *>(gate_fp16);
    f.up_or_h = up_fp32;
    f.residual = residual;
    return run_fused(type, W_blocks, N, K, M, f, gate_fp16, up_fp32, y_fp32, stream);
}

int qlinear_rmsnorm(int type, const void *W_blocks, int64_t N, int64_t K, const float *h_fp32, const float *norm_w_fp32,
                    float eps, int64_t M, const float *residual, float *y_fp32, void *xnorm_fp16, void *stream) {
    ql::GemvFusion f;
    f.pro = 2;
    f.up_or_h = h_fp32;
    f.norm_w = norm_w_fp32;
    f.eps = eps;
    f.xnorm = static_cast<__half *>(xnorm_fp16);
    f.residual = residual;
    return run_fused(type, W_blocks, N, K, M, f, h_fp32, norm_w_fp32, y_fp32, stream);
}

int qlinear_block_bytes(int type) {
    const int b = ql::block_bytes_of(type);
    return b < 0 ? QL_ERR_TYPE : b;
}

int qlinear_gemv_max_m(void) { return ql::kGemvMaxM; }

const char *qlinear_strerror(int status) {
    switch (status) {
    case QL_OK: return "success";
    case QL_ERR_TYPE: return "unsupported type (expected Q4_K=12, Q5_K=13, Q6_K=14, IQ4_XS=23, aligned Q6_K=270)";
    case QL_ERR_SHAPE: return "bad shape (need K % 256 == 0, K >= 256, N >= 1, M >= 1, within 32-bit indexing)";
    case QL_ERR_NULL: return "null pointer argument";
    case QL_ERR_ALIGN: return "W, x and y must be 16-byte aligned";
    case QL_ERR_CUDA: return "CUDA runtime error (see qlinear_last_cuda_error)";
    case QL_ERR_TIMEOUT: return "a device-side bounded wait ran out";
    case QL_ERR_UNSUPPORTED: return "the requested kernel cannot run this shape";
    case QL_ERR_DEVICE: return "current device is not an sm_103 (GB300) GPU";
    case QL_ERR_INDEX: return "an index read on the device was out of range (embedding id)";
    case QL_ERR_BOUNDS: return "a bounds check of the QL_DEBUG build failed (the access was skipped)";
    default: return "unknown status";
    }
}

int qlinear_last_cuda_error(void) { return t_last_cuda_error; }

int qlinear_selftest_wait_timeout(void *stream) {
    DeviceState *s = nullptr;
    int rc = device_state(&s);
    if (rc != QL_OK) return rc;
    if (launch_refused(*s)) return QL_ERR_CUDA;
    wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(s->status_word);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QL_OK : cuda_fail(e);
}

int qlinear_device_status(void *stream) {
    DeviceState *s = nullptr;
    int rc = device_state(&s);
    if (rc != QL_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(s->status_mutex);
    // read and clear in one device operation, after the stream's work: a bit another stream sets
    // meanwhile is either taken now or kept for the next check, never lost
    status_take_kernel<<<1, 1, 0, st>>>(s->status_word, s->status_taken);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned word = 0;
    if ((e = cudaMemcpyAsync(&word, s->status_taken, sizeof(word), cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return cuda_fail(e);
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e);
    if (word & ql::kStatusBounds) return QL_ERR_BOUNDS;
    if (word & ql::kStatusTimeout) return QL_ERR_TIMEOUT;
    return word ? QL_ERR_INDEX : QL_OK;
}

int qlinear_gemm_plan(int type, int64_t N, int64_t K, int64_t M, int num_sms, const int *cluster_capacity,
                      int64_t *plan) {
    if (ql::block_bytes_of(type) < 0) return QL_ERR_TYPE;
    if (N < 1 || M < 1 || K < 256 || K % 256 != 0 || N > (int64_t(1) << 30) || K > (int64_t(1) << 24) ||
        M > kMaxTokens || num_sms < 1)
        return QL_ERR_SHAPE;
    if (!plan) return QL_ERR_NULL;
    const int rc = ql::gemm_plan_info(type, N, K, M, num_sms, cluster_capacity, plan);
    return rc == 0 ? QL_OK : rc == -1 ? QL_ERR_TYPE : QL_ERR_UNSUPPORTED;
}

int qlinear_launch_count(int type, int64_t N, int64_t K, int64_t M) {
    if (ql::block_bytes_of(type) < 0) return QL_ERR_TYPE;
    if (N < 1 || M < 1 || K < 256 || K % 256 != 0) return QL_ERR_SHAPE;
    if (M <= ql::kGemvMaxM) return 1;
    return ql::gemm_launch_count(type, N, K, M);
}

}  // extern "C"
