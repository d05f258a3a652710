// Device helpers shared by the epilogue kernels: 128-bit fragments of T
// unpacked to float32, cache-hinted global loads/stores, and row-group
// reductions (warp shuffles, then shared memory across warps).
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace ep {
namespace dev {

// Elements of T in one 16-byte vector.
template <typename T> struct Vec16;
template <> struct Vec16<float> { static constexpr int N = 4; };
template <> struct Vec16<__half> { static constexpr int N = 8; };
template <> struct Vec16<__nv_bfloat16> { static constexpr int N = 8; };

// ---------------------------------------------------------------------------
// global memory access
//   stream : touched once (inputs/outputs of the op) -> evict-first in L1/L2
//   keep   : reused across rows (gamma, beta, bias, a broadcast skip) and never
//            written by the kernel -> read-only path, normal L2 priority
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint4 ld16_stream(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint4 ld16_keep(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st16_stream(void* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

__device__ __forceinline__ float ld1_stream(const float* p) { return __ldcs(p); }
__device__ __forceinline__ float ld1_stream(const __half* p) { return __half2float(__ldcs(p)); }
__device__ __forceinline__ float ld1_stream(const __nv_bfloat16* p) { return __bfloat162float(__ldcs(p)); }
__device__ __forceinline__ float ld1_keep(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ld1_keep(const __half* p) { return __half2float(__ldg(p)); }
__device__ __forceinline__ float ld1_keep(const __nv_bfloat16* p) { return __bfloat162float(__ldg(p)); }
__device__ __forceinline__ void st1_stream(float* p, float v) { __stcs(p, v); }
__device__ __forceinline__ void st1_stream(__half* p, float v) { __stcs(p, __float2half_rn(v)); }
__device__ __forceinline__ void st1_stream(__nv_bfloat16* p, float v) { __stcs(p, __float2bfloat16_rn(v)); }

// 16 bytes <-> float32 lanes, per element type (conversions to float32 are
// exact; conversions from float32 round to nearest-even).
template <typename T> struct Conv;
template <> struct Conv<float> {
  static __device__ __forceinline__ void unpack(uint4 u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  static __device__ __forceinline__ uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};
template <> struct Conv<__half> {
  static __device__ __forceinline__ void unpack(uint4 u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = t.x; f[2 * i + 1] = t.y;
    }
  }
  static __device__ __forceinline__ uint4 pack(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <> struct Conv<__nv_bfloat16> {
  static __device__ __forceinline__ void unpack(uint4 u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      f[2 * i] = t.x; f[2 * i + 1] = t.y;
    }
  }
  static __device__ __forceinline__ uint4 pack(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// Programmatic dependent launch.  pdl_wait returns once the grids this one
// depends on have completed and their memory is visible (at once for a grid
// launched without that dependency); every kernel calls it before its first
// global memory access.  pdl_trigger, called after it, lets a dependent grid
// launch once every CTA of this one has triggered or exited, so a dependent
// never starts before this grid's own predecessors have completed.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 2^x and 1/x with the hardware approximations (flush-to-zero): relative
// errors of a few float32 ulp, used where the result is rounded to float16 or
// must only meet an absolute tolerance.  e^x is taken as 2^(x * log2(e)).
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16-byte shared-memory load of T elements, unpacked to float32; and a
// 16-byte evict-first global store of float32 lanes packed to T.
template <typename T, int VW>
__device__ __forceinline__ void lds_unpack(const T* p, float (&f)[VW]) {
  Conv<T>::unpack(*reinterpret_cast<const uint4*>(p), f);
}
template <typename T, int VW>
__device__ __forceinline__ void stg_pack_stream(T* p, const float (&f)[VW]) {
  st16_stream(p, Conv<T>::pack(f));
}

// A fragment of VW consecutive elements held as float32.  VW == Vec16<T>::N
// uses one 128-bit access (the address must be 16-byte aligned); VW == 1 is
// the scalar path.
template <typename T, int VW> struct Frag {
  float v[VW];
  __device__ __forceinline__ void load_stream(const T* p) {
    if constexpr (VW == 1) v[0] = ld1_stream(p);
    else Conv<T>::unpack(ld16_stream(p), v);
  }
  __device__ __forceinline__ void load_keep(const T* p) {
    if constexpr (VW == 1) v[0] = ld1_keep(p);
    else Conv<T>::unpack(ld16_keep(p), v);
  }
  __device__ __forceinline__ void store_stream(T* p) const {
    if constexpr (VW == 1) st1_stream(p, v[0]);
    else st16_stream(p, Conv<T>::pack(v));
  }
};

// ---------------------------------------------------------------------------
// reductions over a row group of TPR consecutive threads (TPR a power of two).
// TPR <= 32: shuffles inside the warp segment.  TPR > 32: shuffles, then one
// shared-memory slot per warp and a __syncthreads(); every thread of the group
// then adds the group's slots in the same order, so all of them hold the same
// value.  `red` has blockDim.x / 32 floats.  Every thread of the block must
// call the TPR > 32 form the same number of times.
// ---------------------------------------------------------------------------

template <int TPR>
__device__ __forceinline__ float group_sum(float x, float* red) {
  if constexpr (TPR <= 32) {
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
  } else {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    constexpr int W = TPR / 32;
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[warp] = x;
    __syncthreads();
    const float* g = red + (warp / W) * W;
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < W; ++i) t += g[i];
    return t;
  }
}

template <int TPR>
__device__ __forceinline__ float group_max(float x, float* red) {
  if constexpr (TPR <= 32) {
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
  } else {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    constexpr int W = TPR / 32;
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[warp] = x;
    __syncthreads();
    const float* g = red + (warp / W) * W;
    float t = g[0];
#pragma unroll
    for (int i = 1; i < W; ++i) t = fmaxf(t, g[i]);
    return t;
  }
}

// Row-group reductions that synchronise only the group: TPR <= 32 uses
// shuffles within the warp segment; TPR > 32 (whole warps) uses a named
// barrier `bar_id` over the group's TPR threads and the group's slots of
// `red` (indexed by warp within the group: `gwarp0` is the group's first warp).
template <int TPR>
__device__ __forceinline__ float group_sum_named(float x, float* red, int bar_id, int gwarp0) {
  if constexpr (TPR <= 32) {
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
  } else {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    constexpr int W = TPR / 32;
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[warp] = x;
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(TPR) : "memory");
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < W; ++i) t += red[gwarp0 + i];
    return t;
  }
}

template <int TPR>
__device__ __forceinline__ float group_max_named(float x, float* red, int bar_id, int gwarp0) {
  if constexpr (TPR <= 32) {
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
  } else {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    constexpr int W = TPR / 32;
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[warp] = x;
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(TPR) : "memory");
    float t = red[gwarp0];
#pragma unroll
    for (int i = 1; i < W; ++i) t = fmaxf(t, red[gwarp0 + i]);
    return t;
  }
}

}  // namespace dev
}  // namespace ep
