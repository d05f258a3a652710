// SkipLayerNormalization kernels.
//
// Definition: com.microsoft.SkipLayerNormalization manifest, `description`,
// `inputs` (skip shapes, optional beta/bias), `outputs` (input_skip_bias_sum)
// and `attributes.epsilon`; its shaders carry a `simplified` flag (the RMS form)
// that the same kernel implements.
//
// Design (GB300): a row is owned by a group of TPR threads; each thread keeps
// NV fragments of VW elements of s = (input + skip) + bias in float32 registers,
// so input, skip and the outputs each cross HBM exactly once.  The mean and the
// variance are two reductions over the registers (warp shuffles, then shared
// memory across the warps of a group): a two-pass variance with no second
// global read.  gamma/beta/bias and a broadcast skip are read through the
// read-only path at normal L2 priority (they are reused by every row); the
// streamed tensors use evict-first loads and stores.  Rows too long for the
// register budget fall back to a CTA-per-row kernel that re-reads the row
// (three passes) instead of holding it.
#include <algorithm>

#include "device_common.cuh"
#include "ep_internal.h"

namespace ep {
namespace {

using dev::Frag;

struct SlnKernelArgs {
  const void* input;
  const void* skip;
  const void* gamma;
  const void* beta;
  const void* bias;
  void* output;
  void* sum_out;
  float* mean_out;
  float* inv_std_out;
  int64_t rows;
  int64_t skip_rows;
  int64_t H;
  float eps;
  bool simplified;
  bool skip_bcast;  // skip_rows < rows: skip is reused, keep it cached
};

template <typename T, int VW, int TPR, int NV>
__global__ void __launch_bounds__(TPR > 256 ? TPR : 256)
k_skip_layer_norm(const SlnKernelArgs a) {
  constexpr int BS = TPR > 256 ? TPR : 256;
  constexpr int RPC = BS / TPR;  // rows per CTA
  __shared__ float red_a[BS / 32];
  __shared__ float red_b[BS / 32];

  // input/skip may be the same buffers as output/sum_out (exact in-place
  // aliasing), so only the never-written vectors are marked __restrict__.
  const T* in = static_cast<const T*>(a.input);
  const T* sk = static_cast<const T*>(a.skip);
  const T* __restrict__ gamma = static_cast<const T*>(a.gamma);
  const T* __restrict__ beta = static_cast<const T*>(a.beta);
  const T* __restrict__ bias = static_cast<const T*>(a.bias);
  T* out = static_cast<T*>(a.output);
  T* sum_out = static_cast<T*>(a.sum_out);

  const int g = threadIdx.x / TPR;
  const int lane = threadIdx.x % TPR;
  const int64_t H = a.H;

  for (int64_t base = static_cast<int64_t>(blockIdx.x) * RPC; base < a.rows;
       base += static_cast<int64_t>(gridDim.x) * RPC) {
    const int64_t r = base + g;
    const bool active = r < a.rows;
    const int64_t off = r * H;
    const int64_t soff = a.skip_bcast ? (r % a.skip_rows) * H : off;

    Frag<T, VW> s[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int e = 0; e < VW; ++e) s[v].v[e] = 0.f;

    if (active) {
      Frag<T, VW> k[NV];
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int64_t c = static_cast<int64_t>(v * TPR + lane) * VW;
        if (c < H) {
          s[v].load_stream(in + off + c);
          if (a.skip_bcast) k[v].load_keep(sk + soff + c);
          else k[v].load_stream(sk + soff + c);
        }
      }
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int64_t c = static_cast<int64_t>(v * TPR + lane) * VW;
        if (c < H) {
#pragma unroll
          for (int e = 0; e < VW; ++e) s[v].v[e] = __fadd_rn(s[v].v[e], k[v].v[e]);
          if (bias != nullptr) {
            Frag<T, VW> b;
            b.load_keep(bias + c);
#pragma unroll
            for (int e = 0; e < VW; ++e) s[v].v[e] = __fadd_rn(s[v].v[e], b.v[e]);
          }
          if (sum_out != nullptr) s[v].store_stream(sum_out + off + c);
        }
      }
    }

    float mean = 0.f;
    if (!a.simplified) {
      float t = 0.f;
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int e = 0; e < VW; ++e) t += s[v].v[e];
      mean = dev::group_sum<TPR>(t, red_a) / static_cast<float>(H);
    }
    float q = 0.f;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int64_t c = static_cast<int64_t>(v * TPR + lane) * VW;
      if (c < H) {
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          const float d = s[v].v[e] - mean;
          q = fmaf(d, d, q);
        }
      }
    }
    const float var = dev::group_sum<TPR>(q, red_b) / static_cast<float>(H);
    const float rstd = 1.0f / sqrtf(var + a.eps);

    if (active) {
      if (lane == 0) {
        if (a.mean_out != nullptr) a.mean_out[r] = mean;
        if (a.inv_std_out != nullptr) a.inv_std_out[r] = rstd;
      }
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int64_t c = static_cast<int64_t>(v * TPR + lane) * VW;
        if (c < H) {
          Frag<T, VW> gm, bt, y;
          gm.load_keep(gamma + c);
          if (beta != nullptr) bt.load_keep(beta + c);
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            const float n = (s[v].v[e] - mean) * rstd;
            y.v[e] = beta != nullptr ? fmaf(n, gm.v[e], bt.v[e]) : n * gm.v[e];
          }
          y.store_stream(out + off + c);
        }
      }
    }
  }
}

// Rows longer than the register budget: one 1024-thread CTA per row, three
// passes over the row (sum; squared deviations; outputs).  Each pass recomputes
// s from input/skip/bias; the outputs are written only in the last pass, each
// element by the thread that read it, so exact in-place aliasing stays valid.
template <typename T>
__global__ void __launch_bounds__(1024) k_skip_layer_norm_long(const SlnKernelArgs a) {
  __shared__ float red_a[32];
  __shared__ float red_b[32];
  const T* in = static_cast<const T*>(a.input);
  const T* sk = static_cast<const T*>(a.skip);
  const T* gamma = static_cast<const T*>(a.gamma);
  const T* beta = static_cast<const T*>(a.beta);
  const T* bias = static_cast<const T*>(a.bias);
  T* out = static_cast<T*>(a.output);
  T* sum_out = static_cast<T*>(a.sum_out);
  const int64_t H = a.H;

  auto s_at = [&](int64_t off, int64_t soff, int64_t c) {
    const float k = a.skip_bcast ? dev::ld1_keep(sk + soff + c) : dev::ld1_stream(sk + soff + c);
    float s = __fadd_rn(dev::ld1_stream(in + off + c), k);
    if (bias != nullptr) s = __fadd_rn(s, dev::ld1_keep(bias + c));
    return s;
  };

  for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
    const int64_t off = r * H;
    const int64_t soff = a.skip_bcast ? (r % a.skip_rows) * H : off;
    float mean = 0.f;
    if (!a.simplified) {
      float t = 0.f;
      for (int64_t c = threadIdx.x; c < H; c += blockDim.x) t += s_at(off, soff, c);
      mean = dev::group_sum<1024>(t, red_a) / static_cast<float>(H);
    }
    float q = 0.f;
    for (int64_t c = threadIdx.x; c < H; c += blockDim.x) {
      const float d = s_at(off, soff, c) - mean;
      q = fmaf(d, d, q);
    }
    const float var = dev::group_sum<1024>(q, red_b) / static_cast<float>(H);
    const float rstd = 1.0f / sqrtf(var + a.eps);
    if (threadIdx.x == 0) {
      if (a.mean_out != nullptr) a.mean_out[r] = mean;
      if (a.inv_std_out != nullptr) a.inv_std_out[r] = rstd;
    }
    for (int64_t c = threadIdx.x; c < H; c += blockDim.x) {
      const float s = s_at(off, soff, c);
      if (sum_out != nullptr) dev::st1_stream(sum_out + off + c, s);
      const float n = (s - mean) * rstd;
      const float gm = dev::ld1_keep(gamma + c);
      dev::st1_stream(out + off + c, beta != nullptr ? fmaf(n, gm, dev::ld1_keep(beta + c)) : n * gm);
    }
    // red_a/red_b are reused by the next row: the next write to red_a follows
    // this row's second barrier, which every thread passes only after reading red_a.
  }
}

// ---------------------------------------------------------------------------
// launch planning
// ---------------------------------------------------------------------------

using KernelFn = void (*)(SlnKernelArgs);

// Row-group shapes (threads per row TPR, fragments per thread NV) compiled for
// each (T, VW), in order of capacity TPR*NV*VW; the first that holds the row is
// taken.  Every shape keeps at most 32 floats of the row per thread, so the row
// stays in registers without spilling; the largest holds kRowMax elements.
// Longer rows use the three-pass kernel.
constexpr int64_t kRowMax = 16384;

template <typename T, int VW>
KernelFn pick_kernel(int64_t H, int* tpr_out) {
  const int64_t nfrag = H / VW;
#define EP_SLN_CASE(TPR_, NV_)                          \
  if (nfrag <= int64_t(TPR_) * NV_) {                   \
    *tpr_out = TPR_;                                    \
    return k_skip_layer_norm<T, VW, TPR_, NV_>;         \
  }
  if constexpr (VW == 8) {
    EP_SLN_CASE(32, 1) EP_SLN_CASE(32, 2) EP_SLN_CASE(32, 4) EP_SLN_CASE(64, 4)
    EP_SLN_CASE(128, 4) EP_SLN_CASE(256, 4) EP_SLN_CASE(512, 4)
  } else if constexpr (VW == 4) {
    EP_SLN_CASE(32, 1) EP_SLN_CASE(32, 2) EP_SLN_CASE(32, 4) EP_SLN_CASE(32, 8)
    EP_SLN_CASE(64, 8) EP_SLN_CASE(128, 8) EP_SLN_CASE(256, 8) EP_SLN_CASE(512, 8)
  } else {
    EP_SLN_CASE(32, 1) EP_SLN_CASE(32, 2) EP_SLN_CASE(32, 4) EP_SLN_CASE(32, 8)
    EP_SLN_CASE(64, 8) EP_SLN_CASE(128, 8) EP_SLN_CASE(256, 8) EP_SLN_CASE(512, 8)
    EP_SLN_CASE(512, 16) EP_SLN_CASE(512, 32)
  }
#undef EP_SLN_CASE
  return nullptr;
}

template <typename T>
cudaError_t launch_t(const SlnArgs& a, int sm_count, cudaStream_t stream, int* launches) {
  SlnKernelArgs k{a.input, a.skip, a.gamma, a.beta, a.bias, a.output, a.sum_out,
                  a.mean_out, a.inv_std_out, a.rows, a.skip_rows, a.H, a.eps,
                  a.simplified, a.skip_rows < a.rows};
  constexpr int VW = dev::Vec16<T>::N;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool vec = (a.H % VW == 0) && al16(a.input) && al16(a.skip) && al16(a.gamma) &&
                   al16(a.beta) && al16(a.bias) && al16(a.output) && al16(a.sum_out);
  int tpr = 0;
  KernelFn fn = vec ? pick_kernel<T, VW>(a.H, &tpr) : pick_kernel<T, 1>(a.H, &tpr);
  if (fn != nullptr) {
    const int bs = std::max(tpr, 256);
    const int rpc = bs / tpr;
    const int64_t need = (a.rows + rpc - 1) / rpc;
    const int64_t cap = int64_t(sm_count) * 64 * (2048 / bs);  // many waves, then grid-stride
    const unsigned grid = static_cast<unsigned>(std::min(need, cap));
    fn<<<grid, bs, 0, stream>>>(k);
  } else {
    const int64_t cap = int64_t(sm_count) * 2 * 16;
    const unsigned grid = static_cast<unsigned>(std::min(a.rows, cap));
    k_skip_layer_norm_long<T><<<grid, 1024, 0, stream>>>(k);
  }
  *launches += 1;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_skip_layer_norm(const SlnArgs& a, int sm_count, cudaStream_t stream, int* launches) {
  return a.t == DType::F32 ? launch_t<float>(a, sm_count, stream, launches)
                           : launch_t<__half>(a, sm_count, stream, launches);
}

}  // namespace ep
