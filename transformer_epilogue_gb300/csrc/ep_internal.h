// Internal interface between the C ABI layer (ep_api.cpp, validation and
// bookkeeping) and the CUDA translation units (kernels + launch planning).
// Arguments reaching a launcher have been validated: shapes are consistent,
// pointers are non-NULL where needed and aligned to sizeof(T), and every count
// is positive.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace ep {

enum class DType : int { F32 = 0, F16 = 1, BF16 = 2 };

inline int dtype_size(DType t) { return t == DType::F32 ? 4 : 2; }

struct SlnArgs {
  DType t;
  const void* input;
  const void* skip;
  const void* gamma;
  const void* beta;     // nullable
  const void* bias;     // nullable
  void* output;
  void* sum_out;        // nullable: input_skip_bias_sum
  float* mean_out;      // nullable: per-row float32 mean (0 when simplified)
  float* inv_std_out;   // nullable: per-row float32 1/sqrt(var + eps)
  int64_t rows;         // > 0
  int64_t skip_rows;    // divides rows
  int64_t H;            // > 0
  float eps;
  bool simplified;      // RMS form: no mean subtraction
};

struct SoftmaxArgs {
  DType t;
  const void* data;
  const void* bias;
  void* output;
  int64_t rows;         // batchCount > 0
  int64_t cols;         // blockSize > 0
  int64_t bias_rows;    // biasBlockCount, divides rows
  int64_t inner_repeat; // rows / bias_rows
  bool inner;           // is_inner_broadcast != 0
  void* workspace;      // split-row statistics (nullable when not needed)
  size_t workspace_bytes;
};

struct BiasAddArgs {
  DType t;
  const void* x;
  const void* bias;
  const void* skip;
  void* y;
  int64_t n;            // numel(X) > 0
  int64_t C;            // channels > 0
};

struct QuickGeluArgs {
  DType t;
  const void* x;
  void* y;
  int64_t n;            // numel > 0
  float alpha;
};

// Each launcher enqueues its kernel(s) on `stream`, adds the number of kernels
// enqueued to *launches, and returns the first CUDA error seen (cudaSuccess
// otherwise).  `sm_count` is the device's multiprocessor count.
cudaError_t launch_skip_layer_norm(const SlnArgs& a, int sm_count, cudaStream_t stream, int* launches);
// `l2_bytes` (the device's L2 size) sizes the row windows of the split-row path.
cudaError_t launch_bias_softmax(const SoftmaxArgs& a, int sm_count, int l2_bytes, cudaStream_t stream,
                                int* launches);
cudaError_t launch_bias_add(const BiasAddArgs& a, int sm_count, cudaStream_t stream, int* launches);
cudaError_t launch_quick_gelu(const QuickGeluArgs& a, int sm_count, cudaStream_t stream, int* launches);

// Bytes of split-row workspace BiasSoftmax needs for (rows, cols) of type t;
// 0 when the rows fit the on-chip row kernel.  Depends only on the shape, not
// on pointer alignment.
size_t softmax_workspace_bytes(DType t, int64_t rows, int64_t cols);

// Fixed device scratch of ep_bias_softmax_noalloc: its size, and its device
// address on the current device (looked up on the first call per device).
size_t static_softmax_scratch_bytes();
cudaError_t static_softmax_scratch(void** addr);

// Bounded-wait timeouts counted by each translation unit's staged kernels on
// the current device (synchronous read; `clear` resets the counter).
cudaError_t sln_pipe_timeouts(unsigned int* count, bool clear);
cudaError_t softmax_pipe_timeouts(unsigned int* count, bool clear);
cudaError_t elementwise_pipe_timeouts(unsigned int* count, bool clear);

// One-CTA kernel whose bounded wait is made to run out after timeout_ns.
cudaError_t launch_selftest_bounded_wait(uint64_t timeout_ns, cudaStream_t stream, int* launches);

}  // namespace ep
