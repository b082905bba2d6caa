/*
 * qlinear.h -- C ABI of the GB300 (sm_103a) GGUF weight-only quantized linear layer.
 *
 * The layer computes, for a weight matrix W stored as GGUF/ggml superblocks of 256 weights,
 *
 *     y[m][n] = sum_{k<K} x[m][k] * dequant(W)[n][k]          m < M, n < N
 *
 * with fp16 activations x, fp32 accumulation and an fp32 result y. Supported block formats
 * (ggml type id: bytes per 256-weight superblock), from the _GGML_QUANT table of
 * tinygrad/llm/gguf.py:
 *     Q4_K   = 12 : 144     d, dmin fp16; 12-byte packed 6-bit scales/mins; 128 B of 4-bit q
 *     Q5_K   = 13 : 176     as Q4_K plus a 32-byte high-bit array (commit log of explicit-dev,
 *                           commit "custom kernels: Q4_K support (ggml type 12)")
 *     Q6_K   = 14 : 210     128 B low 4 bits, 64 B high 2 bits, 16 int8 scales, d fp16 last
 *     IQ4_XS = 23 : 136     d fp16; 6-bit per-32 scales; 4-bit indices into a 16-entry
 *                           non-linear codebook (test/unit/test_llm_quant_cpu.py,
 *                           test_unpack_lut_dot_uop)
 * Dequantised weight: K-quants d*sc*q - dmin*m; Q6_K d*sc*(q-32); IQ4_XS d*(ls-32)*kv[q].
 *
 * Layouts (all row-major, contiguous, little-endian):
 *   W_blocks : N rows x (K/256) superblocks; row n, superblock b at byte (n*K/256 + b)*BB.
 *              This is the packed slice a GGUF file stores for an (N, K) tensor (dims
 *              reversed, K fastest: tinygrad/llm/gguf.py, _gguf_parse).
 *   x_fp16   : M x K IEEE binary16.
 *   y_fp32   : M x N fp32, overwritten (never accumulated into).
 *
 * Ownership and execution: every pointer is a device pointer owned by the caller, on the
 * current CUDA device (device or managed memory of another GPU, or plain host memory, is
 * refused with QL_ERR_DEVICE before any launch). W and x are read-only. The call is
 * asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream): it validates,
 * enqueues and returns without synchronising. The library keeps a small per-device state (SM
 * count, the device status word, kernel attributes) created on first use and never frees
 * caller memory. Calls on distinct streams may run concurrently; no scratch memory is shared
 * between calls.
 *
 * Weights and the preceding kernel: the layer kernels are launched with programmatic dependent
 * launch (unless the environment sets QL_PDL=0) and start fetching W before the kernel ahead of
 * them in the stream has finished; only x (and the other inputs) are read after it completes.
 * So W must not be written by the kernel that immediately precedes the call on its stream, nor
 * by an earlier one linked to the call through kernels that also start early (qlinear_copy is
 * one). qlinear_repack keeps this by ending with an empty ordinary launch; a caller that writes
 * W with its own kernel right before a call puts any other work (or an event wait) in between,
 * or sets QL_PDL=0.
 *
 * Errors: arguments are checked on the host before any launch, and a failing check
 * returns a negative ql_status with nothing enqueued. A failed launch returns
 * QL_ERR_CUDA (qlinear_last_cuda_error() gives the cudaError_t, per calling thread).
 * Device-side pipeline waits are bounded; a wait that runs out sets the device's status
 * word, which qlinear_device_status() reports as QL_ERR_TIMEOUT. The status word is one per
 * device, shared by all streams.
 */
#ifndef QLINEAR_H_
#define QLINEAR_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QL_Q4_K = 12,
    QL_Q5_K = 13,
    QL_Q6_K = 14,
    QL_IQ4_XS = 23,
    QL_Q6_K_A16 = 270   /* Q6_K repacked by qlinear_repack: 224-byte blocks, 16-byte aligned */
} ql_type;

typedef enum {
    QL_OK = 0,
    QL_ERR_TYPE = -1,        /* unsupported ggml type */
    QL_ERR_SHAPE = -2,       /* K % 256 != 0, N < 1, M < 1, M > 65535*32, or beyond int32 indexing */
    QL_ERR_NULL = -3,        /* a required pointer is NULL */
    QL_ERR_ALIGN = -4,       /* W, x or y not 16-byte aligned */
    QL_ERR_CUDA = -5,        /* a CUDA runtime call or kernel launch failed */
    QL_ERR_TIMEOUT = -6,     /* a device-side bounded wait ran out (see qlinear_device_status) */
    QL_ERR_UNSUPPORTED = -7, /* the forced path cannot run this shape on this device */
    QL_ERR_DEVICE = -8,      /* the current device is not an sm_103 (GB300) part, or a pointer
                                is not device memory of the current device */
    QL_ERR_INDEX = -9,       /* an index read on the device was out of range (see qlinear_embed) */
    QL_ERR_BOUNDS = -10      /* a QL_DEBUG build's bounds check failed; the access was skipped */
} ql_status;

/*
 * qlinear: y = x . dequant(W)^T, dispatched on M.
 *   M <= qlinear_gemv_max_m()  -> decode kernel (tensor-core mma.sync GEMV, weights
 *                                 streamed once from HBM through a TMA-fed shared ring)
 *   otherwise                   -> prefill kernel (tcgen05 MMA with TMEM accumulators)
 * Chunked prefill pads M to the MMA tile internally; padded rows are never stored
 * (commit log of explicit-dev: "quant linears pad to the chunk bucket").
 * Arguments: type = ql_type; W_blocks = packed weights (N*K/256*BB bytes, 16-byte aligned);
 * N, K = output / input features (K % 256 == 0); x_fp16 = activations (M*K halves,
 * 16-byte aligned); M = tokens; y_fp32 = output (M*N floats, 16-byte aligned);
 * stream = cudaStream_t or NULL. Returns QL_OK or a negative ql_status.
 */
int qlinear(int type, const void *W_blocks, int64_t N, int64_t K, const void *x_fp16, int64_t M,
            float *y_fp32, void *stream);

/* Same contract, forcing the decode (GEMV) kernel for any M >= 1. Tokens are processed in
 * groups of 8 per MMA; the packed weights are decoded once per call. */
int qlinear_gemv(int type, const void *W_blocks, int64_t N, int64_t K, const void *x_fp16, int64_t M,
                 float *y_fp32, void *stream);

/* Same contract, forcing the prefill (tcgen05) kernel for any M >= 1. */
int qlinear_gemm(int type, const void *W_blocks, int64_t N, int64_t K, const void *x_fp16, int64_t M,
                 float *y_fp32, void *stream);

/*
 * qlinear_multi: several projections of the same activations in one pass,
 *     y_j = x . dequant(W_j)^T          j < n_proj
 * for weights that share `type` and K (a transformer's Q/K/V or gate/up projections). The
 * pages fuse such pairs in their engine and check that the fused result equals the separate
 * layers (test/unit/test_llm_quant_cpu.py, test_q8_linear_pair_matches_separate).
 * For M <= qlinear_gemv_max_m() one decode launch covers all projections: the row tiles of
 * every W_j form one work list split evenly over the SMs, and each slice of x is loaded once;
 * for larger M each projection runs the prefill kernel in turn.
 * Arguments: n_proj in [1, qlinear_max_projections()]; W_blocks, N and y_fp32 are HOST arrays
 * of n_proj entries (W_blocks[j] and y_fp32[j] are device pointers with the layouts and
 * alignment of qlinear(), y_fp32[j] holding M*N[j] floats); K, x_fp16, M, stream as in
 * qlinear(). Every projection is validated as a qlinear() call; NULL arrays give QL_ERR_NULL
 * and n_proj out of range QL_ERR_SHAPE, with nothing enqueued. The outputs must not overlap.
 */
int qlinear_multi(int type, int n_proj, const void *const *W_blocks, const int64_t *N, int64_t K,
                  const void *x_fp16, int64_t M, float *const *y_fp32, void *stream);

/* Most projections one qlinear_multi() call takes (4). */
int qlinear_max_projections(void);

/*
 * qlinear_repack: Q6_K weights (type QL_Q6_K, 210-byte blocks) rewritten into the aligned
 * layout QL_Q6_K_A16: every block followed by 14 zero bytes (224 bytes), so each block and
 * each row starts on a 16-byte boundary. A 210-byte block fits a 2-D tensor copy only in stages
 * of 8 blocks starting at multiples of 8 (the copy's inner extent and start must be 16-byte
 * multiples), so Q6_K rows are otherwise fetched with one bulk copy per row; in the aligned
 * layout both kernels use 2-D tensor copies. The pages leave the packed layout to the engine
 * (test/unit/test_llm_quant_cpu.py repacks weights for its own kernels: q8_repack).
 * Pass the result to any call with type = QL_Q6_K_A16; it decodes to the same weights.
 * W_src: N*K/256*210 bytes; W_dst: N*K/256*224 bytes (device, 16-byte aligned, not
 * overlapping). Asynchronous on `stream` (the repack kernel, then an empty ordinary launch
 * that makes a layer call right after it safe: see "Weights and the preceding kernel").
 * type must be QL_Q6_K (else QL_ERR_TYPE).
 */
int qlinear_repack(int type, const void *W_src, int64_t N, int64_t K, void *W_dst, void *stream);

/*
 * qlinear_copy: copies `bytes` from src to dst on `stream` with a kernel, for moving a layer's
 * inputs in and its outputs out around the layer calls of a step. Each pointer is device
 * memory of the current device or page-locked host memory mapped into the device's address
 * space (cudaHostAlloc / cudaHostRegister memory on a system with unified addressing); a
 * host pointer is read or written by the kernel directly, with no staging buffer. Anything
 * else gives QL_ERR_DEVICE before any launch. The regions must not overlap; bytes == 0 does
 * nothing; bytes < 0 gives QL_ERR_SHAPE; a NULL pointer (bytes > 0) gives QL_ERR_NULL.
 * The kernel is a programmatic dependent launch like the layer kernels (it lets the next
 * kernel start at once and waits for the preceding one before touching memory), so a layer
 * call right after it streams its weights while the copy runs, and a copy right after a
 * layer call starts as that call drains. For the same reason it is for a step's inputs and
 * outputs, not for a layer's weights: copied W must be separated from the layer calls that read
 * it by an ordinary launch, an event wait or a synchronisation (see "Weights and the preceding
 * kernel"). Asynchronous; the bytes are in dst once the stream has reached the copy's end (e.g.
 * after a stream synchronize for a host dst).
 */
int qlinear_copy(void *dst, const void *src, int64_t bytes, void *stream);

/*
 * Decode calls with the layer's input produced inside the launch (fused prologue) and an
 * optional residual added to the output (fused epilogue). The pages fuse both element-wise
 * producers into the consuming linear and check the result equals the separate steps
 * (test/unit/test_llm_quant_cpu.py: test_q8_silu_linear_matches_separate,
 * test_f16_linear_matches_standard).
 *
 * qlinear_silu_mul: y = x . dequant(W)^T (+ residual) with x = fp16(silu(gate) * up),
 *   silu(g) = g / (1 + e^-g), evaluated in fp32 and rounded once to fp16 (the pages'
 *   silu_mul(gate, up).half()). gate_fp16: [M, K] binary16; up_fp32: [M, K] fp32.
 * qlinear_rmsnorm: y = x . dequant(W)^T (+ residual) with
 *   x = fp16(h * rsqrt(mean_k(h^2) + eps) * norm_w), h_fp32 [M, K], norm_w_fp32 [K], eps >= 0,
 *   evaluated in fp32. When xnorm_fp16 is not NULL the fp16 x is also written there ([M, K]).
 * Both: M <= qlinear_gemv_max_m() (else QL_ERR_UNSUPPORTED); residual is NULL or an [M, N]
 * fp32 array, and may be y_fp32 itself (y += x . W^T). Device pointers are 16-byte aligned
 * (QL_ERR_ALIGN); W, gate/h, up/norm_w and y must not be NULL (QL_ERR_NULL); a negative or
 * non-finite eps gives QL_ERR_SHAPE. Validation, ownership and streams as for qlinear().
 * The result matches the oracle within the layer's tolerance widened by one fp16 rounding
 * step of each activation (the fp32 prologue may round across a boundary the fp64 one does not).
 */
/*
 * qlinear_argmax: the greedy output head. For each token m < M (M <= qlinear_gemv_max_m()),
 * index_out[m] = the first n with the largest y[m][n] of y = x . dequant(W)^T, and, when
 * value_out is not NULL, value_out[m] = that y (fp32), without materialising y: the decode
 * kernel keeps, per CTA and token, the best (value, row) and merges it across CTAs by one
 * 64-bit atomic maximum. Every y[m][n] is the value qlinear() computes for it, bit for bit, so
 * the choice equals the first maximum of qlinear()'s output (+0 and -0 compare equal; a NaN
 * ranks above every number). The pages pick the next token from a Q6_K head this way and check
 * it against the argmax of the materialised logits (test/unit/test_llm_quant_cpu.py,
 * test_q6_argmax_matches_materialized_logits).
 * index_out: M int64 (16-byte aligned), also used as scratch; value_out: M floats or NULL.
 * Enqueues a memset and two kernels on `stream`. Other arguments as for qlinear().
 */
int qlinear_argmax(int type, const void *W_blocks, int64_t N, int64_t K, const void *x_fp16, int64_t M,
                   int64_t *index_out, float *value_out, void *stream);

/*
 * qlinear_embed: the embedding gather, out[m][k] = dequant(W)[ids[m]][k] for m < M, k < K:
 * each weight is its exact value rounded once to fp32 (out_fp16 == 0) or to fp16, round to
 * nearest even (out_fp16 != 0). The pages' quantized Embedding returns the fp16 rounding of the
 * dequantised rows (test/unit/test_llm_quant_cpu.py, test_q4_embedding_matches_reference).
 * W_blocks: N rows as for qlinear(); ids: M int32 device indices (4-byte aligned); out: M*K
 * elements (16-byte aligned). An id outside [0, N) cannot be checked on the host: its row is
 * written as zeros and the next qlinear_device_status() reports QL_ERR_INDEX.
 */
int qlinear_embed(int type, const void *W_blocks, int64_t N, int64_t K, const int32_t *ids, int64_t M, void *out,
                  int out_fp16, void *stream);

int qlinear_silu_mul(int type, const void *W_blocks, int64_t N, int64_t K, const void *gate_fp16,
                     const float *up_fp32, int64_t M, const float *residual, float *y_fp32, void *stream);
int qlinear_rmsnorm(int type, const void *W_blocks, int64_t N, int64_t K, const float *h_fp32,
                    const float *norm_w_fp32, float eps, int64_t M, const float *residual, float *y_fp32,
                    void *xnorm_fp16, void *stream);

/* Bytes per 256-weight superblock of `type` (144/176/210/136), or QL_ERR_TYPE. */
int qlinear_block_bytes(int type);

/* Largest M that qlinear() sends to the decode kernel (8). */
int qlinear_gemv_max_m(void);

/* Static description of a status code; never NULL. */
const char *qlinear_strerror(int status);

/* cudaError_t recorded by the last QL_ERR_CUDA returned on the calling thread (0 if none). */
int qlinear_last_cuda_error(void);

/* After the work already enqueued on `stream`, reads and clears the device status word of the
 * current device in one atomic exchange (a one-thread kernel on `stream`), then synchronises
 * `stream`: QL_OK; QL_ERR_BOUNDS if a QL_DEBUG build's bounds check failed; else QL_ERR_TIMEOUT
 * if a bounded wait in a kernel ran out since the last check; else QL_ERR_INDEX if an embedding
 * id was out of range; QL_ERR_CUDA if a CUDA call failed. The word is per device: a bit set by
 * work on another stream is reported by whichever check takes it first, and none is lost. */
int qlinear_device_status(void *stream);

/* Number of kernels one qlinear() call of this shape launches (for launch accounting);
 * QL_ERR_* on invalid arguments. */
int qlinear_launch_count(int type, int64_t N, int64_t K, int64_t M);

/*
 * qlinear_gemm_plan: the launch plan of the prefill GEMM (M > 8) for this shape, computed on
 * the host without a device, for tests and tooling. num_sms: the device's SM count;
 * cluster_capacity[i]: how many thread-block clusters of i + 2 CTAs can be resident at once
 * (i = 0..6; NULL: none, so no split plan). plan[14] receives {n_tile, k, L, tail, S, xk,
 * a_col, a_slots, recv_off, bar_off, grid_x, grid_y, cluster, smem}:
 *   n_tile  tokens per tile;  k  heads per tail CTA (0: one CTA per row tile and token tile);
 *   L, tail superblocks [0, L) of a row tile go to its head, [L, K/256) to the tail;
 *   S       superblocks per weight stage;  xk  64-wide k chunks per x stage;
 *   a_col, a_slots  first TMEM column and depth (superblocks) of the dequantised-weight ring;
 *   recv_off, bar_off  shared-memory offsets of the split form's receive area and barriers;
 *   grid_x, grid_y, cluster, smem  the launch (cluster: CTAs per cluster, 1 = none).
 * The device call makes the same plan with the device's SM count and cudaOccupancyMaxActiveClusters.
 * QL_ERR_TYPE, QL_ERR_SHAPE (as qlinear, or num_sms < 1), QL_ERR_NULL (plan), or
 * QL_ERR_UNSUPPORTED when no plan fits in shared memory.
 */
int qlinear_gemm_plan(int type, int64_t N, int64_t K, int64_t M, int num_sms, const int *cluster_capacity,
                      int64_t *plan);

/* Diagnostic of the failure path: enqueues on `stream` one small kernel whose bounded wait
 * on a barrier that nothing completes runs out (after about 2 s) and sets the device status
 * word, exactly as an expired pipeline wait in the layer's kernels would. No fault is raised
 * and the context stays usable; the next qlinear_device_status() reports QL_ERR_TIMEOUT.
 * Returns QL_OK once enqueued, else an error. (Not part of the method; it tests the
 * library's own error reporting.) */
int qlinear_selftest_wait_timeout(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* QLINEAR_H_ */
