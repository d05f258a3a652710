// C ABI of the epilogue library: argument validation (the op definitions'
// contracts), overlap and alignment checks, device queries, error strings and
// the launch counter.  Kernels and their launch planning live in the .cu files.
#include "ep.h"

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <cuda_runtime.h>

#include "ep_internal.h"

namespace {

constexpr int kAbiVersion = 1;
constexpr int kMaxRank = 16;
constexpr int kMaxDevices = 64;

thread_local char g_err[512] = "";
std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_l2_bytes[kMaxDevices];

ep_status fail(ep_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

ep_status ok() {
  g_err[0] = '\0';
  return EP_OK;
}

bool valid_dtype(ep_dtype t) { return t == EP_F32 || t == EP_F16 || t == EP_BF16; }
int esize(ep_dtype t) { return t == EP_F32 ? 4 : 2; }
ep::DType to_dtype(ep_dtype t) {
  return t == EP_F32 ? ep::DType::F32 : t == EP_F16 ? ep::DType::F16 : ep::DType::BF16;
}

// Product of dims [b, e); false if a dim is negative or the product overflows 2^62.
bool dims_product(const int64_t* d, int b, int e, int64_t* out) {
  int64_t p = 1;
  for (int i = b; i < e; ++i) {
    if (d[i] < 0) return false;
    if (d[i] != 0 && p > (int64_t(1) << 62) / d[i]) return false;
    p *= d[i];
  }
  *out = p;
  return true;
}

bool aligned(const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) % uintptr_t(a)) == 0; }

struct Span {
  const void* p;
  int64_t bytes;
};

bool overlap(Span a, Span b) {
  if (a.p == nullptr || b.p == nullptr || a.bytes <= 0 || b.bytes <= 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + uintptr_t(b.bytes) && b0 < a0 + uintptr_t(a.bytes);
}

bool exact_alias(Span a, Span b) { return a.p == b.p && a.bytes == b.bytes; }

// An output may share storage with an input only as an exact alias.
bool bad_overlap_inplace_ok(Span out, Span in) { return overlap(out, in) && !exact_alias(out, in); }

struct DevInfo {
  int sm_count;
  int l2_bytes;
};

ep_status device_info(DevInfo* info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(EP_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < kMaxDevices) {
    const int sm = g_sm_count[dev].load(std::memory_order_relaxed);
    if (sm > 0) {
      info->sm_count = sm;
      info->l2_bytes = g_l2_bytes[dev].load(std::memory_order_relaxed);
      return EP_OK;
    }
  }
  int sm = 0, l2 = 0;
  e = cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
  if (e != cudaSuccess || sm <= 0)
    return fail(EP_ERR_CUDA, "device attribute query failed: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < kMaxDevices) {
    g_l2_bytes[dev].store(l2, std::memory_order_relaxed);
    g_sm_count[dev].store(sm, std::memory_order_relaxed);
  }
  info->sm_count = sm;
  info->l2_bytes = l2;
  return EP_OK;
}

ep_status finish(cudaError_t e, int launches, const char* op) {
  g_launches.fetch_add(uint64_t(launches), std::memory_order_relaxed);
  if (e != cudaSuccess) return fail(EP_ERR_CUDA, "%s: kernel launch failed: %s", op, cudaGetErrorString(e));
  return ok();
}

}  // namespace

extern "C" {

const char* ep_last_error(void) { return g_err; }

const char* ep_status_name(ep_status s) {
  switch (s) {
    case EP_OK: return "EP_OK";
    case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG";
    case EP_ERR_UNSUPPORTED: return "EP_ERR_UNSUPPORTED";
    case EP_ERR_WORKSPACE: return "EP_ERR_WORKSPACE";
    case EP_ERR_CUDA: return "EP_ERR_CUDA";
  }
  return "EP_STATUS_UNKNOWN";
}

uint64_t ep_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int ep_abi_version(void) { return kAbiVersion; }

namespace {
cudaError_t sum_pipe_timeouts(unsigned int* total, bool clear) {
  unsigned int a = 0, b = 0, c = 0;
  cudaError_t e = ep::sln_pipe_timeouts(&a, clear);
  if (e == cudaSuccess) e = ep::softmax_pipe_timeouts(&b, clear);
  if (e == cudaSuccess) e = ep::elementwise_pipe_timeouts(&c, clear);
  *total = a + b + c;
  return e;
}
}  // namespace

ep_status ep_pipeline_timeouts(uint64_t* count, int clear) {
  if (count == nullptr) return fail(EP_ERR_INVALID_ARG, "pipeline_timeouts: NULL count");
  unsigned int total = 0;
  cudaError_t e = sum_pipe_timeouts(&total, clear != 0);
  if (e != cudaSuccess) return fail(EP_ERR_CUDA, "pipeline_timeouts: %s", cudaGetErrorString(e));
  *count = total;
  return ok();
}

ep_status ep_selftest_bounded_wait(uint32_t timeout_us, uint64_t* timeouts_seen, ep_stream_t stream) {
  if (timeouts_seen == nullptr) return fail(EP_ERR_INVALID_ARG, "selftest_bounded_wait: NULL timeouts_seen");
  if (timeout_us < 1 || timeout_us > 1000000)
    return fail(EP_ERR_INVALID_ARG, "selftest_bounded_wait: limit %u us outside 1..1000000", timeout_us);
  unsigned int before = 0, after = 0;
  cudaError_t e = sum_pipe_timeouts(&before, false);
  if (e != cudaSuccess) return fail(EP_ERR_CUDA, "selftest_bounded_wait: %s", cudaGetErrorString(e));
  int launches = 0;
  e = ep::launch_selftest_bounded_wait(uint64_t(timeout_us) * 1000u, reinterpret_cast<cudaStream_t>(stream),
                                       &launches);
  g_launches.fetch_add(uint64_t(launches), std::memory_order_relaxed);
  if (e == cudaSuccess) e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = sum_pipe_timeouts(&after, false);
  if (e != cudaSuccess) return fail(EP_ERR_CUDA, "selftest_bounded_wait: %s", cudaGetErrorString(e));
  *timeouts_seen = uint64_t(after - before);
  return ok();
}

ep_status ep_skip_layer_norm_ex(ep_dtype t, const void* input, const int64_t* in_shape, int in_rank,
                                const void* skip, const int64_t* skip_shape, int skip_rank,
                                const void* gamma, const void* beta, const void* bias, float epsilon,
                                int simplified, void* output, void* input_skip_bias_sum, float* mean,
                                float* inv_std_dev, ep_stream_t stream) {
  if (!valid_dtype(t)) return fail(EP_ERR_UNSUPPORTED, "skip_layer_norm: dtype %d is not float32/float16/bfloat16", int(t));
  if (in_rank != 2 && in_rank != 3)
    return fail(EP_ERR_UNSUPPORTED, "skip_layer_norm: input rank %d (rank 2 or 3 supported)", in_rank);
  if (in_shape == nullptr || skip_shape == nullptr)
    return fail(EP_ERR_INVALID_ARG, "skip_layer_norm: NULL shape array");
  int64_t numel = 0;
  if (!dims_product(in_shape, 0, in_rank, &numel))
    return fail(EP_ERR_INVALID_ARG, "skip_layer_norm: negative or overflowing input dims");
  const int64_t H = in_shape[in_rank - 1];
  if (H <= 0) return fail(EP_ERR_INVALID_ARG, "skip_layer_norm: hidden size must be > 0, got %lld", (long long)H);
  const int64_t rows = numel / H;
  // skip shapes (rank2CoreContract; broadcastSkipShapeOk)
  bool skip_ok = false;
  if (skip_rank == in_rank) {
    skip_ok = true;
    for (int i = 0; i < in_rank; ++i) skip_ok = skip_ok && skip_shape[i] == in_shape[i];
    if (!skip_ok && in_rank == 3)
      skip_ok = skip_shape[0] == 1 && skip_shape[1] == in_shape[1] && skip_shape[2] == in_shape[2];
  } else if (in_rank == 3 && skip_rank == 2) {
    skip_ok = skip_shape[0] == in_shape[1] && skip_shape[1] == in_shape[2];
  }
  if (!skip_ok)
    return fail(EP_ERR_INVALID_ARG,
                "skip_layer_norm: skip shape must equal the input shape, or be (1,S,H) or (S,H) for rank-3 input");
  int64_t skip_numel = 0;
  dims_product(skip_shape, 0, skip_rank, &skip_numel);
  const int64_t skip_rows = skip_numel / H;
  if (!(epsilon >= 0.0f)) return fail(EP_ERR_INVALID_ARG, "skip_layer_norm: epsilon must be >= 0");
  if (simplified != 0 && simplified != 1)
    return fail(EP_ERR_INVALID_ARG, "skip_layer_norm: simplified must be 0 or 1");
  if (rows == 0) return ok();
  if (skip_rows == 0 || rows % skip_rows != 0)
    return fail(EP_ERR_INVALID_ARG, "skip_layer_norm: skip rows do not tile the input rows");
  if (input == nullptr || skip == nullptr || gamma == nullptr || output == nullptr)
    return fail(EP_ERR_INVALID_ARG, "skip_layer_norm: input, skip, gamma and output are required");
  const int es = esize(t);
  const void* ptrs[] = {input, skip, gamma, beta, bias, output, input_skip_bias_sum};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned(p, es))
      return fail(EP_ERR_INVALID_ARG, "skip_layer_norm: pointer %p is not aligned to the element size", p);
  if ((mean != nullptr && !aligned(mean, 4)) || (inv_std_dev != nullptr && !aligned(inv_std_dev, 4)))
    return fail(EP_ERR_INVALID_ARG, "skip_layer_norm: mean / inv_std_dev must be 4-byte aligned");
  const int64_t nb = numel * es;
  const Span in{input, nb}, sk{skip, skip_numel * es}, g{gamma, H * es}, b{beta, H * es}, bi{bias, H * es};
  const Span outs[] = {{output, nb}, {input_skip_bias_sum, nb}};
  for (const Span& o : outs) {
    if (o.p == nullptr) continue;
    if (bad_overlap_inplace_ok(o, in) || bad_overlap_inplace_ok(o, sk) || overlap(o, g) || overlap(o, b) ||
        overlap(o, bi))
      return fail(EP_ERR_INVALID_ARG, "skip_layer_norm: an output overlaps an input other than as an exact alias");
  }
  if (overlap(outs[0], outs[1])) return fail(EP_ERR_INVALID_ARG, "skip_layer_norm: output and input_skip_bias_sum overlap");
  const Span stat_spans[] = {{mean, rows * 4}, {inv_std_dev, rows * 4}};
  for (const Span& st : stat_spans) {
    if (st.p == nullptr) continue;
    if (overlap(st, in) || overlap(st, sk) || overlap(st, g) || overlap(st, b) || overlap(st, bi) ||
        overlap(st, outs[0]) || overlap(st, outs[1]))
      return fail(EP_ERR_INVALID_ARG, "skip_layer_norm: mean / inv_std_dev overlap another operand");
  }
  if (overlap(stat_spans[0], stat_spans[1]))
    return fail(EP_ERR_INVALID_ARG, "skip_layer_norm: mean and inv_std_dev overlap");
  DevInfo dv;
  if (ep_status s = device_info(&dv); s != EP_OK) return s;
  ep::SlnArgs a{to_dtype(t), input, skip, gamma, beta, bias, output, input_skip_bias_sum, mean, inv_std_dev,
                rows, skip_rows, H, epsilon, simplified != 0};
  int launches = 0;
  cudaError_t e = ep::launch_skip_layer_norm(a, dv.sm_count, reinterpret_cast<cudaStream_t>(stream), &launches);
  return finish(e, launches, "skip_layer_norm");
}

ep_status ep_skip_layer_norm(ep_dtype t, const void* input, const int64_t* in_shape, int in_rank,
                             const void* skip, const int64_t* skip_shape, int skip_rank,
                             const void* gamma, const void* beta, const void* bias, float epsilon,
                             void* output, void* input_skip_bias_sum, ep_stream_t stream) {
  return ep_skip_layer_norm_ex(t, input, in_shape, in_rank, skip, skip_shape, skip_rank, gamma, beta, bias,
                               epsilon, 0, output, input_skip_bias_sum, nullptr, nullptr, stream);
}

namespace {

struct SoftmaxDims {
  int64_t batch, block, numel, bias_rows;
};

ep_status softmax_dims(const char* op, ep_dtype t, const int64_t* shape, int rank, int axis, SoftmaxDims* d) {
  if (!valid_dtype(t)) return fail(EP_ERR_UNSUPPORTED, "%s: dtype %d is not float32/float16/bfloat16", op, int(t));
  if (rank < 1) return fail(EP_ERR_INVALID_ARG, "%s: data rank must be >= 1", op);
  if (rank > kMaxRank) return fail(EP_ERR_UNSUPPORTED, "%s: rank %d > %d", op, rank, kMaxRank);
  if (shape == nullptr) return fail(EP_ERR_INVALID_ARG, "%s: NULL shape array", op);
  if (!(axis + rank >= 0 && axis < rank))
    return fail(EP_ERR_INVALID_ARG, "%s: axis %d out of range for rank %d", op, axis, rank);
  const int an = axis < 0 ? axis + rank : axis;
  if (!dims_product(shape, 0, an, &d->batch) || !dims_product(shape, an, rank, &d->block) ||
      !dims_product(shape, 0, rank, &d->numel))
    return fail(EP_ERR_INVALID_ARG, "%s: negative or overflowing dims", op);
  return EP_OK;
}

}  // namespace

size_t ep_bias_softmax_workspace_size(ep_dtype t, const int64_t* shape, int rank, int axis) {
  SoftmaxDims d;
  char saved[sizeof(g_err)];
  std::memcpy(saved, g_err, sizeof(g_err));
  const ep_status s = softmax_dims("bias_softmax_workspace_size", t, shape, rank, axis, &d);
  std::memcpy(g_err, saved, sizeof(g_err));
  if (s != EP_OK || d.numel == 0) return 0;
  return ep::softmax_workspace_bytes(to_dtype(t), d.batch, d.block);
}

ep_status ep_bias_softmax(ep_dtype t, const void* data, const int64_t* shape, int rank, const void* bias,
                          int64_t bias_numel, int axis, int is_inner_broadcast, void* output, void* workspace,
                          size_t workspace_bytes, ep_stream_t stream) {
  SoftmaxDims d;
  if (ep_status s = softmax_dims("bias_softmax", t, shape, rank, axis, &d); s != EP_OK) return s;
  if (bias_numel < 0) return fail(EP_ERR_INVALID_ARG, "bias_softmax: negative bias_numel");
  // derive.biasContract
  const int64_t bias_rows = d.block > 0 ? bias_numel / d.block : 0;
  const bool contract = (d.numel == 0 && bias_numel == 0) ||
                        (d.block > 0 && bias_rows > 0 && bias_numel % d.block == 0 && bias_rows <= d.batch &&
                         d.batch % bias_rows == 0);
  if (!contract)
    return fail(EP_ERR_INVALID_ARG,
                "bias_softmax: biasContract violated (bias numel %lld, blockSize %lld, batchCount %lld)",
                (long long)bias_numel, (long long)d.block, (long long)d.batch);
  if (d.numel == 0) return ok();
  if (data == nullptr || bias == nullptr || output == nullptr)
    return fail(EP_ERR_INVALID_ARG, "bias_softmax: data, bias and output are required");
  const int es = esize(t);
  if (!aligned(data, es) || !aligned(bias, es) || !aligned(output, es))
    return fail(EP_ERR_INVALID_ARG, "bias_softmax: pointer not aligned to the element size");
  const Span dt{data, d.numel * es}, bs{bias, bias_numel * es}, out{output, d.numel * es};
  if (bad_overlap_inplace_ok(out, dt) || overlap(out, bs))
    return fail(EP_ERR_INVALID_ARG, "bias_softmax: output overlaps an input other than as an exact alias of data");
  const size_t need = ep::softmax_workspace_bytes(to_dtype(t), d.batch, d.block);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 16))
      return fail(EP_ERR_WORKSPACE, "bias_softmax: split-row path needs %zu bytes of 16-byte-aligned workspace, got %zu%s",
                  need, workspace == nullptr ? size_t(0) : workspace_bytes,
                  (workspace != nullptr && !aligned(workspace, 16)) ? " (misaligned)" : "");
    const Span ws{workspace, int64_t(need)};
    if (overlap(ws, dt) || overlap(ws, bs) || overlap(ws, out))
      return fail(EP_ERR_WORKSPACE, "bias_softmax: workspace overlaps data, bias or output");
  }
  DevInfo dv;
  if (ep_status s = device_info(&dv); s != EP_OK) return s;
  ep::SoftmaxArgs a{to_dtype(t), data, bias, output, d.batch, d.block, bias_rows, d.batch / bias_rows,
                    is_inner_broadcast != 0, need > 0 ? workspace : nullptr, need};
  int launches = 0;
  cudaError_t e = ep::launch_bias_softmax(a, dv.sm_count, dv.l2_bytes, reinterpret_cast<cudaStream_t>(stream),
                                          &launches);
  return finish(e, launches, "bias_softmax");
}

ep_status ep_bias_softmax_noalloc(ep_dtype t, const void* data, const int64_t* shape, int rank, const void* bias,
                                  int64_t bias_numel, int axis, int is_inner_broadcast, void* output,
                                  ep_stream_t stream) {
  SoftmaxDims d;
  if (ep_status s = softmax_dims("bias_softmax_noalloc", t, shape, rank, axis, &d); s != EP_OK) return s;
  if (bias_numel < 0) return fail(EP_ERR_INVALID_ARG, "bias_softmax_noalloc: negative bias_numel");
  const int64_t bias_rows = d.block > 0 ? bias_numel / d.block : 0;
  const bool contract = (d.numel == 0 && bias_numel == 0) ||
                        (d.block > 0 && bias_rows > 0 && bias_numel % d.block == 0 && bias_rows <= d.batch &&
                         d.batch % bias_rows == 0);
  if (!contract)
    return fail(EP_ERR_INVALID_ARG,
                "bias_softmax_noalloc: biasContract violated (bias numel %lld, blockSize %lld, batchCount %lld)",
                (long long)bias_numel, (long long)d.block, (long long)d.batch);
  if (d.numel == 0) return ok();
  if (data == nullptr || bias == nullptr || output == nullptr)
    return fail(EP_ERR_INVALID_ARG, "bias_softmax_noalloc: data, bias and output are required");
  const int es = esize(t);
  if (!aligned(data, es) || !aligned(bias, es) || !aligned(output, es))
    return fail(EP_ERR_INVALID_ARG, "bias_softmax_noalloc: pointer not aligned to the element size");
  const Span dt{data, d.numel * es}, bs{bias, bias_numel * es}, out{output, d.numel * es};
  if (bad_overlap_inplace_ok(out, dt) || overlap(out, bs))
    return fail(EP_ERR_INVALID_ARG,
                "bias_softmax_noalloc: output overlaps an input other than as an exact alias of data");
  const size_t need = ep::softmax_workspace_bytes(to_dtype(t), d.batch, d.block);
  const size_t cap = ep::static_softmax_scratch_bytes();
  if (need > cap)
    return fail(EP_ERR_WORKSPACE,
                "bias_softmax_noalloc: this shape needs %zu bytes of split-row scratch, more than the fixed %zu "
                "(rows * ceil(blockSize / %d) must be <= %zu); use ep_bias_softmax with a workspace",
                need, cap, t == EP_F32 ? 4096 : 8192, cap / 8);
  DevInfo dv;
  if (ep_status s = device_info(&dv); s != EP_OK) return s;
  void* scratch = nullptr;
  if (need > 0) {
    cudaError_t e = ep::static_softmax_scratch(&scratch);
    if (e != cudaSuccess)
      return fail(EP_ERR_CUDA, "bias_softmax_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
  }
  ep::SoftmaxArgs a{to_dtype(t), data, bias, output, d.batch, d.block, bias_rows, d.batch / bias_rows,
                    is_inner_broadcast != 0, scratch, need};
  int launches = 0;
  cudaError_t e = ep::launch_bias_softmax(a, dv.sm_count, dv.l2_bytes, reinterpret_cast<cudaStream_t>(stream),
                                          &launches);
  return finish(e, launches, "bias_softmax_noalloc");
}

ep_status ep_bias_add(ep_dtype t, const void* X, const int64_t* shape, const void* bias, const void* skip, void* Y,
                      ep_stream_t stream) {
  if (!valid_dtype(t)) return fail(EP_ERR_UNSUPPORTED, "bias_add: dtype %d is not float32/float16/bfloat16", int(t));
  if (shape == nullptr) return fail(EP_ERR_INVALID_ARG, "bias_add: NULL shape array");
  int64_t n = 0;
  if (!dims_product(shape, 0, 3, &n)) return fail(EP_ERR_INVALID_ARG, "bias_add: negative or overflowing dims");
  const int64_t C = shape[2];
  if (n == 0) return ok();
  if (X == nullptr || bias == nullptr || skip == nullptr || Y == nullptr)
    return fail(EP_ERR_INVALID_ARG, "bias_add: X, bias, skip and Y are required");
  const int es = esize(t);
  if (!aligned(X, es) || !aligned(bias, es) || !aligned(skip, es) || !aligned(Y, es))
    return fail(EP_ERR_INVALID_ARG, "bias_add: pointer not aligned to the element size");
  const Span x{X, n * es}, b{bias, C * es}, s{skip, n * es}, y{Y, n * es};
  if (bad_overlap_inplace_ok(y, x) || bad_overlap_inplace_ok(y, s) || overlap(y, b))
    return fail(EP_ERR_INVALID_ARG, "bias_add: Y overlaps an input other than as an exact alias of X or skip");
  DevInfo dv;
  if (ep_status st = device_info(&dv); st != EP_OK) return st;
  ep::BiasAddArgs a{to_dtype(t), X, bias, skip, Y, n, C};
  int launches = 0;
  cudaError_t e = ep::launch_bias_add(a, dv.sm_count, reinterpret_cast<cudaStream_t>(stream), &launches);
  return finish(e, launches, "bias_add");
}

ep_status ep_quick_gelu(ep_dtype t, const void* X, int64_t numel, float alpha, void* Y, ep_stream_t stream) {
  if (!valid_dtype(t)) return fail(EP_ERR_UNSUPPORTED, "quick_gelu: dtype %d is not float32/float16/bfloat16", int(t));
  if (numel < 0) return fail(EP_ERR_INVALID_ARG, "quick_gelu: negative numel");
  if (numel == 0) return ok();
  if (X == nullptr || Y == nullptr) return fail(EP_ERR_INVALID_ARG, "quick_gelu: X and Y are required");
  const int es = esize(t);
  if (!aligned(X, es) || !aligned(Y, es))
    return fail(EP_ERR_INVALID_ARG, "quick_gelu: pointer not aligned to the element size");
  if (bad_overlap_inplace_ok(Span{Y, numel * es}, Span{X, numel * es}))
    return fail(EP_ERR_INVALID_ARG, "quick_gelu: Y overlaps X other than as an exact alias");
  DevInfo dv;
  if (ep_status s = device_info(&dv); s != EP_OK) return s;
  ep::QuickGeluArgs a{to_dtype(t), X, Y, numel, alpha};
  int launches = 0;
  cudaError_t e = ep::launch_quick_gelu(a, dv.sm_count, reinterpret_cast<cudaStream_t>(stream), &launches);
  return finish(e, launches, "quick_gelu");
}

}  // extern "C"
