/*
 * transformer_epilogue_gb300 — C ABI of the fused transformer-block epilogue ops
 * (SkipLayerNormalization, BiasSoftmax, BiasAdd, QuickGelu) for one NVIDIA GB300
 * (sm_103a) GPU.
 *
 * The ops are the com.microsoft ONNX Runtime contrib ops whose definitions are
 * given by the manifest pages "com.microsoft.SkipLayerNormalization",
 * "com.microsoft.BiasSoftmax", "com.microsoft.BiasAdd" and
 * "com.microsoft.QuickGelu" (sections `description`, `inputs`, `outputs`,
 * `attributes`, `derive`).  Each entry point below cites the section that
 * defines what it computes.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are dense, contiguous, row-major device buffers of element type T
 *    (ep_dtype); every pointer is a device pointer owned by the caller.  The
 *    library allocates nothing and frees nothing.
 *  - Every call is asynchronous: it validates on the host, enqueues its kernel(s)
 *    on `stream` and returns without synchronising.  Outputs are valid once the
 *    stream reaches that point.  A NULL stream is the legacy default stream.
 *  - Kernels are launched as programmatic dependents of the work before them in
 *    the stream (CUDA programmatic dependent launch): their blocks may be
 *    scheduled while that work drains, but no block reads or writes global
 *    memory before every kernel ahead of it in the stream has completed, so the
 *    ordering seen by the caller is ordinary stream order.  Calls may be
 *    captured into CUDA graphs (the split-row workspace must then outlive the
 *    graph).
 *  - All validation happens before anything is enqueued.  A contract violation
 *    returns EP_ERR_INVALID_ARG, a legal op this library does not implement
 *    (another element type, an unsupported rank) returns EP_ERR_UNSUPPORTED, a
 *    split-row BiasSoftmax without enough workspace returns EP_ERR_WORKSPACE, and
 *    a launch error reported by the CUDA runtime returns EP_ERR_CUDA.  On any
 *    non-OK status nothing has been enqueued, except for EP_ERR_CUDA (the
 *    runtime's state is then whatever the failing launch left).  ep_last_error()
 *    gives a message for the calling thread's last non-OK status.
 *  - Empty tensors (numel 0) return EP_OK without launching anything; their
 *    pointers may be NULL.
 *  - Pointers must be aligned to sizeof(T).  16-byte alignment is not
 *    required: it selects the 128-bit vector path (BiasAdd and QuickGelu also
 *    when X, skip and Y share one offset within 16 bytes), and other alignments
 *    take a scalar path computing the same function (the results agree within
 *    the ops' tolerances).
 *  - An output may alias an input exactly (same address, same size: in place).
 *    Any other overlap between an output and another operand is rejected.
 *  - Counts and offsets are 64-bit.
 *  - Arithmetic is float32 for every element type; float16 and bfloat16
 *    results are rounded once, to nearest-even, when stored.
 */
#ifndef TRANSFORMER_EPILOGUE_EP_H
#define TRANSFORMER_EPILOGUE_EP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream; the same type as cudaStream_t (struct CUstream_st*). */
typedef struct CUstream_st* ep_stream_t;

/* Element type T.  The manifests' typeConstraints list float32 and float16
 * (typeConstraints of all four manifests); the op schemas also allow
 * bfloat16, which the WebGPU package leaves out (QuickGelu and
 * SkipLayerNormalization `description`) and this library implements. */
typedef enum { EP_F32 = 0, EP_F16 = 1, EP_BF16 = 2 } ep_dtype;

typedef enum {
  EP_OK = 0,
  EP_ERR_INVALID_ARG = 1,   /* shape, attribute, pointer or overlap contract violated   */
  EP_ERR_UNSUPPORTED = 2,   /* legal for the op, not implemented here (dtype, rank)     */
  EP_ERR_WORKSPACE = 3,     /* split-row BiasSoftmax: workspace NULL or too small       */
  EP_ERR_CUDA = 4           /* the CUDA runtime reported an error for a launch          */
} ep_status;

/* Message for the calling thread's last non-OK status ("" if none).  The string
 * belongs to the library and stays valid until the thread's next call. */
const char* ep_last_error(void);

/* Name of a status code, e.g. "EP_ERR_INVALID_ARG". */
const char* ep_status_name(ep_status s);

/* Number of kernels this library has enqueued in this process (all threads). */
uint64_t ep_kernel_launch_count(void);

/* Version of this ABI (incremented on any incompatible change). */
int ep_abi_version(void);

/* Failure detection.  Every shared-memory barrier wait in the staged kernels
 * is bounded (1 s); a wait that runs out is counted on the device, the kernel
 * stops its remaining work without leaving copies in flight, and the affected
 * outputs are not written.  ep_pipeline_timeouts() adds up those counts on the
 * current device into *count (0 when nothing timed out) and, if clear != 0,
 * resets them.  It synchronises with the device.  No op definition covers
 * this; it exists because the library's kernels wait on barriers. */
ep_status ep_pipeline_timeouts(uint64_t* count, int clear);

/* Self-test of that mechanism: launches a one-CTA kernel on `stream` whose
 * barrier wait is set up to run out (it expects 16 bytes that no copy
 * delivers) with a limit of timeout_us microseconds (1..1000000), waits for the
 * stream, and stores in *timeouts_seen how many timed-out waits the library
 * counted meanwhile (1 expected).  The kernel returns normally after the
 * limit; the device stays usable.  EP_ERR_INVALID_ARG for a limit out of
 * range or a NULL timeouts_seen. */
ep_status ep_selftest_bounded_wait(uint32_t timeout_us, uint64_t* timeouts_seen, ep_stream_t stream);

/*
 * SkipLayerNormalization
 *   com.microsoft.SkipLayerNormalization manifest: `description`, `inputs`,
 *   `outputs`, `attributes.epsilon`, `derive.rank2CoreContract`,
 *   `derive.broadcastSkipShapeOk`.
 *
 *   s = (input + skip) + bias          (float32, in this order; bias optional)
 *   input_skip_bias_sum = T(s)         (optional output)
 *   mu = mean(s), var = mean((s-mu)^2) over the last (hidden) axis, population
 *   output = (s - mu) / sqrt(var + epsilon) * gamma + beta   (beta optional)
 *
 * input      [in_rank dims], in_rank 2 (rows, H) or 3 (N, S, H); H > 0.
 * skip       rank 2: the shape of input.  rank-3 input: the shape of input,
 *            (1, S, H) or (S, H); row r of input uses skip row r mod skipRows,
 *            skipRows = numel(skip) / H.
 * gamma      H elements (required).  beta, bias: H elements or NULL.
 * epsilon    >= 0 (the op's default is 9.999999960041972e-13, float32 1e-12).
 * output     shape of input.
 * input_skip_bias_sum   shape of input, or NULL.
 *
 * Errors: EP_ERR_UNSUPPORTED for a dtype other than EP_F32/EP_F16/EP_BF16 or a rank
 * other than 2/3; EP_ERR_INVALID_ARG for a non-positive H, a skip shape not
 * listed above, a negative or NaN epsilon, a NULL required pointer, a
 * misaligned pointer or an overlap other than exact in-place aliasing.
 */
ep_status ep_skip_layer_norm(ep_dtype t,
                             const void* input, const int64_t* in_shape, int in_rank,
                             const void* skip, const int64_t* skip_shape, int skip_rank,
                             const void* gamma, const void* beta, const void* bias,
                             float epsilon,
                             void* output, void* input_skip_bias_sum,
                             ep_stream_t stream);

/*
 * SkipLayerNormalization with the RMS form and the per-row statistics.
 *   The manifests' SkipLayerNormalization shaders carry a `simplified` flag
 *   (always false in the package; the RMS form of the contrib op family,
 *   SkipSimplifiedLayerNormalization), and the op's `description` names the
 *   training-statistics outputs it does not implement.  This entry point adds
 *   both to ep_skip_layer_norm (same arguments, layout and errors otherwise):
 *
 * simplified   0: as ep_skip_layer_norm.  1: RMS form, no mean subtraction:
 *              output = s / sqrt(mean(s^2) + epsilon) * gamma (+ beta)
 *              (beta is normally NULL in this form).
 * mean         NULL, or numel(input)/H float32 values: the mean of each row's s
 *              (0 when simplified).
 * inv_std_dev  NULL, or numel(input)/H float32 values: 1/sqrt(var + epsilon)
 *              (1/sqrt(mean(s^2) + epsilon) when simplified).
 * The float32 outputs must be 4-byte aligned and overlap no other operand.
 */
ep_status ep_skip_layer_norm_ex(ep_dtype t,
                                const void* input, const int64_t* in_shape, int in_rank,
                                const void* skip, const int64_t* skip_shape, int skip_rank,
                                const void* gamma, const void* beta, const void* bias,
                                float epsilon, int simplified,
                                void* output, void* input_skip_bias_sum,
                                float* mean, float* inv_std_dev,
                                ep_stream_t stream);

/*
 * BiasSoftmax
 *   com.microsoft.BiasSoftmax manifest: `description`, `attributes.axis`,
 *   `attributeDescriptions.is_inner_broadcast`, `derive` (axisNorm, batchCount,
 *   blockSize, biasBlockCount, biasContract).
 *
 *   axisN = axis < 0 ? axis + rank : axis           (0 <= axisN < rank)
 *   batchCount = prod(shape[0:axisN]); blockSize = prod(shape[axisN:rank])
 *   biasRows = bias_numel / blockSize; innerRepeat = batchCount / biasRows
 *   bias row of data row r: r / innerRepeat if is_inner_broadcast != 0,
 *                           r % biasRows    otherwise
 *   output[r, :] = softmax(data[r, :] + bias[bias row, :])
 *
 * data, output  `rank` dims given by `shape` (1 <= rank <= 16).
 * bias          bias_numel elements; only its element count matters.
 * The biasContract must hold: bias_numel % blockSize == 0,
 * 0 < biasRows <= batchCount and batchCount % biasRows == 0, or data and bias
 * are both empty.
 * workspace     device scratch for rows too long to keep on chip (the split-row
 *               path); ep_bias_softmax_workspace_size() gives the bytes needed
 *               (0 when the row path is taken; then workspace may be NULL).
 *               16-byte aligned; its contents on entry do not matter.
 *
 * Errors: EP_ERR_INVALID_ARG for an axis out of range, a violated biasContract,
 * NULL/misaligned pointers or overlaps; EP_ERR_WORKSPACE when the split-row
 * path needs more than workspace_bytes or workspace is NULL/misaligned.
 */
ep_status ep_bias_softmax(ep_dtype t,
                          const void* data, const int64_t* shape, int rank,
                          const void* bias, int64_t bias_numel,
                          int axis, int is_inner_broadcast,
                          void* output,
                          void* workspace, size_t workspace_bytes,
                          ep_stream_t stream);

/* Workspace bytes ep_bias_softmax needs for this dtype, shape and axis (0 if
 * none).  Returns 0 as well for arguments ep_bias_softmax would reject. */
size_t ep_bias_softmax_workspace_size(ep_dtype t, const int64_t* shape, int rank, int axis);

/*
 * BiasSoftmax without a caller-provided workspace.
 *   The op definition has no counterpart to this entry point: it is a variant
 *   of ep_bias_softmax for callers that cannot allocate device memory, e.g. a
 *   plugin or engine whose device memory is all reserved at start-up, code
 *   running inside an allocator or memory-pool callback, or a loop that cannot
 *   afford the device-wide synchronisation cudaMalloc/cudaFree may cause.  Such
 *   callers have no way to provide the scratch the split-row path needs.
 *
 * Same arguments, results and errors as ep_bias_softmax, minus the workspace.
 * The split-row scratch comes from a fixed 1 MiB device array inside the
 * library (held by every device that loads the library until process exit),
 * so rows * ceil(blockSize / chunk) must not exceed 131072 when blockSize >
 * 16384, with chunk = 4096 for float32 and 8192 for float16/bfloat16; larger shapes
 * return EP_ERR_WORKSPACE before anything is enqueued.
 * Rows of up to 16384 elements need no scratch and have no such limit.
 * This entry point allocates nothing.
 *
 * The first call on a device that needs the scratch looks up its device
 * address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.  All calls share the one array, which keeps
 * the previous call's contents: every entry a call reads is written earlier in
 * the same call, so nothing needs clearing, but calls that may overlap on the
 * GPU (other streams, other threads) race on the array and must be ordered by
 * the caller.
 */
ep_status ep_bias_softmax_noalloc(ep_dtype t,
                                  const void* data, const int64_t* shape, int rank,
                                  const void* bias, int64_t bias_numel,
                                  int axis, int is_inner_broadcast,
                                  void* output, ep_stream_t stream);

/*
 * BiasAdd
 *   com.microsoft.BiasAdd manifest: `description`, `inputs`, `outputs`.
 *
 *   Y[n, s, c] = (X[n, s, c] + bias[c]) + skip[n, s, c]
 *
 * shape   3 dims (N, S, C) of X, skip and Y; bias has C elements.
 * For float32 the three-term sum is compensated (error-free two-sums), so Y
 * is within one rounding of the exact sum even under cancellation.
 *
 * Errors: EP_ERR_INVALID_ARG for negative dims, NULL/misaligned pointers or
 * overlaps.
 */
ep_status ep_bias_add(ep_dtype t, const void* X, const int64_t* shape,
                      const void* bias, const void* skip, void* Y,
                      ep_stream_t stream);

/*
 * QuickGelu
 *   com.microsoft.QuickGelu manifest: `description`, `attributes.alpha`.
 *
 *   Y = X * sigmoid(alpha * X)       elementwise over numel elements
 *
 * alpha   the op's default is 1.702.
 *
 * Errors: EP_ERR_INVALID_ARG for numel < 0, NULL/misaligned pointers or
 * overlaps.
 */
ep_status ep_quick_gelu(ep_dtype t, const void* X, int64_t numel, float alpha,
                        void* Y, ep_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* TRANSFORMER_EPILOGUE_EP_H */
