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

// max(a, b, c) in one instruction (NaN operands ignored, as fmaxf does).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// z = data + bias for one 16-byte fragment: the bias unpacked to float32, each
// 16-bit data element added to it by one mixed-precision add (the exact
// float32 value of the element plus the float32 bias, rounded once, as a
// conversion followed by a float32 add).  float32 fragments add in pairs.
template <typename T> struct MixAdd;
template <> struct MixAdd<__half> {
  static __device__ __forceinline__ void add(uint32_t w, float b0, float b1, float& z0, float& z1) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.f16 %0, l, %3;\n\tadd.rn.f32.f16 %1, h, %4;\n\t}"
        : "=&f"(z0), "=f"(z1) : "r"(w), "f"(b0), "f"(b1));
  }
};
template <> struct MixAdd<__nv_bfloat16> {
  static __device__ __forceinline__ void add(uint32_t w, float b0, float b1, float& z0, float& z1) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %3;\n\tadd.rn.f32.bf16 %1, h, %4;\n\t}"
        : "=&f"(z0), "=f"(z1) : "r"(w), "f"(b0), "f"(b1));
  }
};

// z += b for a raw 16-byte fragment b of T (16-bit: one mixed-precision add
// per element; float32: packed adds), each sum rounded once to float32.
template <typename T, int VW>
__device__ __forceinline__ void add_raw(uint4 b, float (&z)[VW]);

// Element-wise z += b and z *= k over a fragment, two lanes per packed
// float32 instruction (each lane rounded exactly as the scalar operation).
template <int VW>
__device__ __forceinline__ void add_pairs(float (&z)[VW], const float (&b)[VW]) {
#pragma unroll
  for (int e = 0; e < VW; e += 2) {
    const float2 t = __fadd2_rn(make_float2(z[e], z[e + 1]), make_float2(b[e], b[e + 1]));
    z[e] = t.x;
    z[e + 1] = t.y;
  }
}
template <int VW>
__device__ __forceinline__ void scale_pairs(float (&z)[VW], float k) {
#pragma unroll
  for (int e = 0; e < VW; e += 2) {
    const float2 t = __fmul2_rn(make_float2(z[e], z[e + 1]), make_float2(k, k));
    z[e] = t.x;
    z[e + 1] = t.y;
  }
}

template <typename T, int VW>
__device__ __forceinline__ void add_raw(uint4 b, float (&z)[VW]) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) MixAdd<T>::add(w[i], z[2 * i], z[2 * i + 1], z[2 * i], z[2 * i + 1]);
  } else {
    float fb[VW];
    Conv<T>::unpack(b, fb);
    add_pairs(z, fb);
  }
}

template <typename T, int VW>
__device__ __forceinline__ void lds_add(const T* d, const T* b, float (&z)[VW]) {
  if constexpr (sizeof(T) == 2) {
    float fb[VW];
    Conv<T>::unpack(*reinterpret_cast<const uint4*>(b), fb);
    const uint4 u = *reinterpret_cast<const uint4*>(d);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) MixAdd<T>::add(w[i], fb[2 * i], fb[2 * i + 1], z[2 * i], z[2 * i + 1]);
  } else {
    float fb[VW];
    Conv<T>::unpack(*reinterpret_cast<const uint4*>(d), z);
    Conv<T>::unpack(*reinterpret_cast<const uint4*>(b), fb);
    add_pairs(z, fb);
  }
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
    if constexpr (W > 8) {
      const int l = threadIdx.x & 31;
      float t = l < W ? g[l] : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      return t;
    } else {
      float t = 0.f;
#pragma unroll
      for (int i = 0; i < W; ++i) t += g[i];
      return t;
    }
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
    if constexpr (W > 8) {
      const int l = threadIdx.x & 31;
      float t = l < W ? g[l] : -INFINITY;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
      return t;
    } else {
      float t = g[0];
#pragma unroll
      for (int i = 1; i < W; ++i) t = fmaxf(t, g[i]);
      return t;
    }
  }
}

// Row-group reductions that synchronise only the group: TPR <= 32 uses
// shuffles within the warp segment; TPR > 32 (whole warps) uses a named
// barrier `bar_id` over the group's TPR threads and the group's slots of
// `red` (indexed by warp within the group: `gwarp0` is the group's first warp).
// Groups of more than 8 warps combine the warps' slots lane-parallel (lane i
// reads slot i, then a butterfly over the warp), which takes fewer
// instructions than every thread adding all the slots in turn.
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
    if constexpr (W > 8) {
      const int l = threadIdx.x & 31;
      float t = l < W ? red[gwarp0 + l] : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      return t;
    } else {
      float t = 0.f;
#pragma unroll
      for (int i = 0; i < W; ++i) t += red[gwarp0 + i];
      return t;
    }
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
    if constexpr (W > 8) {
      const int l = threadIdx.x & 31;
      float t = l < W ? red[gwarp0 + l] : -INFINITY;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
      return t;
    } else {
      float t = red[gwarp0];
#pragma unroll
      for (int i = 1; i < W; ++i) t = fmaxf(t, red[gwarp0 + i]);
      return t;
    }
  }
}

}  // namespace dev
}  // namespace ep
