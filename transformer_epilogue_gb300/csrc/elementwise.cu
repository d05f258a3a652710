// BiasAdd and QuickGelu kernels.
//
// Definitions: com.microsoft.BiasAdd manifest (`description`, `inputs`:
// Y = X + bias[c] + skip over (N, S, C)) and com.microsoft.QuickGelu manifest
// (`description`, `attributes.alpha`: Y = X * sigmoid(alpha * X)).
//
// Design (GB300): a persistent grid (a whole number of CTAs per SM) strides
// over 128-bit fragments; each thread loads U independent fragments of every
// streamed operand before it uses any, so an SM keeps tens of KB of loads in
// flight.  Streamed data is loaded/stored evict-first; bias is read through the
// read-only path and stays in L1/L2.  The manifests' vec4 / vec4-tail / scalar
// variants become one kernel per op: a vector body, plus a scalar head (to
// reach 16-byte alignment) and a scalar tail.  Misaligned operands with
// different offsets take the same kernel with VW = 1.
#include <algorithm>

#include "device_common.cuh"
#include "ep_internal.h"

namespace ep {
namespace {

using dev::Frag;

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ float two_sum3(float a, float b, float c) {
  // (a + b) + c with error-free transformations (Knuth's TwoSum), so that the
  // float32 result is within one rounding of the exact sum, even when it cancels.
  const float s1 = __fadd_rn(a, b);
  const float bb1 = __fsub_rn(s1, a);
  const float e1 = __fadd_rn(__fsub_rn(a, __fsub_rn(s1, bb1)), __fsub_rn(b, bb1));
  const float s2 = __fadd_rn(s1, c);
  const float bb2 = __fsub_rn(s2, s1);
  const float e2 = __fadd_rn(__fsub_rn(s1, __fsub_rn(s2, bb2)), __fsub_rn(c, bb2));
  return __fadd_rn(s2, __fadd_rn(e1, e2));
}

template <typename T>
__device__ __forceinline__ float bias_add_elem(float x, float b, float s) {
  if constexpr (sizeof(T) == 4) return two_sum3(x, b, s);
  else return __fadd_rn(__fadd_rn(x, b), s);  // float16 terms: far below an f16 ulp
}

// BiasAdd: every fragment lies inside one row because C % VW == 0.
template <typename T, int VW>
__global__ void __launch_bounds__(kThreads)
k_bias_add(const T* x, const T* __restrict__ bias, const T* skip, T* y, int64_t nfrag, int64_t C) {
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  const int64_t cfrag = C / VW;
  for (int64_t i0 = int64_t(blockIdx.x) * kThreads + threadIdx.x; i0 < nfrag; i0 += stride * kUnroll) {
    Frag<T, VW> fx[kUnroll], fs[kUnroll], fb[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < nfrag) {
        fx[u].load_stream(x + i * VW);
        fs[u].load_stream(skip + i * VW);
        fb[u].load_keep(bias + (i % cfrag) * VW);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < nfrag) {
        Frag<T, VW> fy;
#pragma unroll
        for (int e = 0; e < VW; ++e) fy.v[e] = bias_add_elem<T>(fx[u].v[e], fb[u].v[e], fs[u].v[e]);
        fy.store_stream(y + i * VW);
      }
    }
  }
}

// x * sigmoid(alpha x), float32 result within a few ulp (relative).
//  z = alpha*x is split into z + zlo exactly (FMA), and exp(z + zlo) is taken
//  as exp(z)*(1 + zlo), which removes the error of rounding alpha*x.
//  z >= 0 : x / (1 + e^{-z});   -64 < z < 0 : x * t/(1 + t), t = e^{z};
//  z <= -64: 1/(1+e^z) rounds to 1, and x*e^z is formed as (x*e^{z+64})*e^{-64}
//  so that no intermediate leaves the normal range before the last product.
__device__ __forceinline__ float quick_gelu_f32(float x, float alpha) {
  const float z = __fmul_rn(alpha, x);
  float zlo = fmaf(alpha, x, -z);
  if (!isfinite(zlo)) zlo = 0.f;
  if (z >= 0.f) {
    float u = expf(-z);
    u = fmaf(-u, zlo, u);
    return __fdiv_rn(x, __fadd_rn(1.0f, u));
  }
  if (z > -64.f) {
    float t = expf(z);
    t = fmaf(t, zlo, t);
    return __fmul_rn(x, __fdiv_rn(t, __fadd_rn(1.0f, t)));
  }
  float t = expf(__fadd_rn(z, 64.0f));
  t = fmaf(t, zlo, t);
  return __fmul_rn(__fmul_rn(x, t), 1.60381089e-28f /* e^-64 */);
}

// float16 results: float32 arithmetic with the fast exponential and divide;
// their error (a few float32 ulp) is far below the float16 rounding.
__device__ __forceinline__ float quick_gelu_f16(float x, float alpha) {
  const float u = __expf(-alpha * x);
  return __fdividef(x, 1.0f + u);
}

template <typename T>
__device__ __forceinline__ float quick_gelu_elem(float x, float alpha) {
  if constexpr (sizeof(T) == 4) return quick_gelu_f32(x, alpha);
  else return quick_gelu_f16(x, alpha);
}

// Elements [0, head) and [head + nfrag*VW, n) are scalar; [head, head + nfrag*VW)
// is the 16-byte-aligned vector body (VW == 1: everything is "body").
template <typename T, int VW>
__global__ void __launch_bounds__(kThreads)
k_quick_gelu(const T* x, T* y, int64_t head, int64_t nfrag, int64_t n, float alpha) {
  const int64_t tid = int64_t(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  const T* xb = x + head;
  T* yb = y + head;
  for (int64_t i0 = tid; i0 < nfrag; i0 += stride * kUnroll) {
    Frag<T, VW> f[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < nfrag) f[u].load_stream(xb + i * VW);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < nfrag) {
#pragma unroll
        for (int e = 0; e < VW; ++e) f[u].v[e] = quick_gelu_elem<T>(f[u].v[e], alpha);
        f[u].store_stream(yb + i * VW);
      }
    }
  }
  if (VW > 1) {
    const int64_t tail0 = head + nfrag * VW;
    const int64_t tail = n - tail0;
    if (tid < head) dev::st1_stream(y + tid, quick_gelu_elem<T>(dev::ld1_stream(x + tid), alpha));
    if (tid < tail) dev::st1_stream(y + tail0 + tid, quick_gelu_elem<T>(dev::ld1_stream(x + tail0 + tid), alpha));
  }
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline unsigned grid_for(int64_t work_items, int sm_count) {
  const int64_t per_sm = 2048 / kThreads;  // full residency at <= 32 registers... and otherwise fewer
  const int64_t need = (work_items + kThreads - 1) / kThreads;
  return static_cast<unsigned>(std::max<int64_t>(1, std::min(need, int64_t(sm_count) * per_sm)));
}

template <typename T>
cudaError_t bias_add_t(const BiasAddArgs& a, int sm_count, cudaStream_t stream, int* launches) {
  constexpr int VW = dev::Vec16<T>::N;
  const T* x = static_cast<const T*>(a.x);
  const T* b = static_cast<const T*>(a.bias);
  const T* s = static_cast<const T*>(a.skip);
  T* y = static_cast<T*>(a.y);
  if (a.C % VW == 0 && al16(x) && al16(b) && al16(s) && al16(y)) {
    const int64_t nfrag = a.n / VW;
    k_bias_add<T, VW><<<grid_for(nfrag, sm_count), kThreads, 0, stream>>>(x, b, s, y, nfrag, a.C);
  } else {
    k_bias_add<T, 1><<<grid_for(a.n, sm_count), kThreads, 0, stream>>>(x, b, s, y, a.n, a.C);
  }
  *launches += 1;
  return cudaGetLastError();
}

template <typename T>
cudaError_t quick_gelu_t(const QuickGeluArgs& a, int sm_count, cudaStream_t stream, int* launches) {
  constexpr int VW = dev::Vec16<T>::N;
  const T* x = static_cast<const T*>(a.x);
  T* y = static_cast<T*>(a.y);
  const uintptr_t ox = reinterpret_cast<uintptr_t>(x) & 15u;
  const uintptr_t oy = reinterpret_cast<uintptr_t>(y) & 15u;
  if (ox == oy) {
    const int64_t head = std::min<int64_t>(a.n, int64_t((16 - ox) & 15u) / int64_t(sizeof(T)));
    const int64_t nfrag = (a.n - head) / VW;
    k_quick_gelu<T, VW><<<grid_for(std::max<int64_t>(nfrag, VW), sm_count), kThreads, 0, stream>>>(
        x, y, head, nfrag, a.n, a.alpha);
  } else {
    k_quick_gelu<T, 1><<<grid_for(a.n, sm_count), kThreads, 0, stream>>>(x, y, 0, a.n, a.n, a.alpha);
  }
  *launches += 1;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bias_add(const BiasAddArgs& a, int sm_count, cudaStream_t stream, int* launches) {
  return a.t == DType::F32 ? bias_add_t<float>(a, sm_count, stream, launches)
                           : bias_add_t<__half>(a, sm_count, stream, launches);
}

cudaError_t launch_quick_gelu(const QuickGeluArgs& a, int sm_count, cudaStream_t stream, int* launches) {
  return a.t == DType::F32 ? quick_gelu_t<float>(a, sm_count, stream, launches)
                           : quick_gelu_t<__half>(a, sm_count, stream, launches);
}

}  // namespace ep
