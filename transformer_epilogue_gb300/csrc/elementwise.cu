// BiasAdd and QuickGelu kernels.
//
// Definitions: com.microsoft.BiasAdd manifest (`description`, `inputs`:
// Y = X + bias[c] + skip over (N, S, C)) and com.microsoft.QuickGelu manifest
// (`description`, `attributes.alpha`: Y = X * sigmoid(alpha * X)).
//
// Design (GB300), two kernel families per op:
//  * 16-byte-aligned operands (at least one tile): the shared-memory-staged,
//    warp-specialised kernel (k_elementwise_tma): a producer warp bulk-copies
//    16 KB tiles into a ring of shared-memory stages, eight consumer warps
//    compute and store; one CTA per tile, running CTAs take over the tiles of
//    CTAs they cancel (cluster launch control).
//  * Anything else: register kernels whose grid strides over 128-bit
//    fragments; each thread loads U independent fragments of every streamed
//    operand before it uses any, so an SM keeps tens of KB of loads in flight.
//    A vector body, plus a scalar head (to reach 16-byte alignment) and a
//    scalar tail; misaligned operands with different offsets use VW = 1.
// Streamed data is loaded/stored evict-first; bias stays in shared memory or
// the read-only path.  Every launch is a programmatic dependent of the work
// before it in the stream.
#include <algorithm>
#include <climits>
#include <type_traits>

#include "device_common.cuh"
#include "ep_internal.h"
#include "launch_util.h"
#include "tma_pipe.cuh"
#include "tuning.h"

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

// (a + b) + c for bfloat16 results: the rounding error e of a + b (Knuth's
// TwoSum) is added after c.  Where a + b and c cancel, their sum is exact
// (Sterbenz) and e is added with one rounding; elsewhere |(a + b) + c| is at
// least about half of |a + b| and e is below its float32 ulp.  Either way the
// float32 result is within two float32 ulp of the exact sum, far inside a
// bfloat16 ulp.
__device__ __forceinline__ float sum3_bf16(float a, float b, float c) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return __fadd_rn(__fadd_rn(s, c), e);
}

template <typename T>
__device__ __forceinline__ float bias_add_elem(float x, float b, float s) {
  // float16 terms span at most 40 bits, so the float32 sum is within a float16
  // ulp without compensation; bfloat16 (float32's exponent range) compensates
  // the first addition, float32 both.
  if constexpr (std::is_same_v<T, __half>) return __fadd_rn(__fadd_rn(x, b), s);
  else if constexpr (std::is_same_v<T, __nv_bfloat16>) return sum3_bf16(x, b, s);
  else return two_sum3(x, b, s);
}

// BiasAdd: every fragment lies inside one row because C % VW == 0.
template <typename T, int VW>
__global__ void __launch_bounds__(kThreads)
k_bias_add(const T* x, const T* __restrict__ bias, const T* skip, T* y, int64_t nfrag, int64_t C) {
  dev::pdl_wait();
  dev::pdl_trigger();
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

// x * sigmoid(alpha x), float32 result within a few ulp (relative), with the
// hardware 2^x and reciprocal instead of a library exponential and a divide.
//  * w = -|alpha x| is carried as wh + wl, exact (TwoProduct: the rounding
//    error of a product is one FMA away, Dekker / Ogita-Rump-Oishi), and so
//    is p = wh log2(e) = ph + pl, with log2(e) itself split into a float and
//    its remainder.
//  * u = e^{w} = 2^{ph} * e^{pl ln2 + wl} ~ 2^{ph} (1 + c), c = pl ln2 + wl:
//    |c| < 2^-16, so the dropped c^2/2 is far below a float32 ulp.
//  * z >= 0: y = x / (1 + u);  z < 0: y = x u / (1 + u);  1 + u is in [1, 2],
//    so the approximate reciprocal stays in the normal range.
//  * For ph < -100, 1 + u rounds to 1: z >= 0 gives y = x; z < 0 gives
//    y = (x 2^{ph + 64} (1 + c)) 2^-64 (2^{ph} itself would leave the normal
//    range below -126), one last product into the subnormal range; below
//    ph = -200, |y| < 2^-180 and rounds to (signed) zero.
__device__ __forceinline__ float quick_gelu_f32(float x, float alpha) {
  constexpr float kL = 1.44269502162933349609375f;  // log2(e) rounded to float32
  constexpr float kLlo = 1.92596298909109e-08f;     // log2(e) - kL
  constexpr float kLn2 = 0.6931471805599453f;
  const float zh = __fmul_rn(alpha, x);
  float zl = fmaf(alpha, x, -zh);
  if (!isfinite(zl)) zl = 0.f;  // alpha x overflowed (or x is not finite)
  const bool pos = zh >= 0.f;
  const float wh = pos ? -zh : zh;
  const float wl = pos ? -zl : zl;
  const float ph = __fmul_rn(wh, kL);
  if (!(ph >= -200.f)) return pos ? x : __fmul_rn(x, 0.f);  // also ph = NaN: x is NaN
  const float pl = fmaf(wh, kLlo, fmaf(wh, kL, -ph));
  const float c = fmaf(pl, kLn2, wl);
  if (ph >= -100.f) {
    float u = dev::ex2_approx(ph);
    u = fmaf(u, c, u);
    const float r = dev::rcp_approx(__fadd_rn(1.0f, u));
    return pos ? __fmul_rn(x, r) : __fmul_rn(__fmul_rn(x, u), r);
  }
  // u < 2^-100: 1 / (1 + u) rounds to 1
  if (pos) return x;
  float u = dev::ex2_approx(__fadd_rn(ph, 64.0f));
  u = fmaf(u, c, u);
  return __fmul_rn(__fmul_rn(x, u), 5.42101086242752217e-20f /* 2^-64 */);
}

// float16 results: float32 arithmetic with the fast exponential and divide;
// their error (a few float32 ulp) is far below the float16 rounding.
__device__ __forceinline__ float quick_gelu_f16(float x, float alpha) {
  const float u = __expf(-alpha * x);
  return __fdividef(x, 1.0f + u);
}

// bfloat16 results: float32 arithmetic with the hardware 2^x and reciprocal,
// t = -alpha x log2(e) rounded once; the errors (a few float32 ulp, and
// |t| 2^-24 from rounding t) are far below a bfloat16 ulp.  bfloat16 keeps
// float32's exponent range, down to 2^-133, but the hardware 2^x flushes
// results below 2^-126: where e^{alpha x} < 2^-64, 1 + e^{alpha x} rounds to 1
// and x e^{alpha x} is formed as (x 2^{64 - t}) 2^-64.  nal2e = -alpha log2(e).
__device__ __forceinline__ float quick_gelu_bf16(float x, float nal2e) {
  const float t = __fmul_rn(x, nal2e);
  if (t > 64.f) return __fmul_rn(__fmul_rn(x, dev::ex2_approx(__fsub_rn(64.f, t))), 5.42101086242752217e-20f);
  return __fmul_rn(x, dev::rcp_approx(__fadd_rn(1.0f, dev::ex2_approx(t))));
}

// float16 results use the fast form, bfloat16 the fast form with its
// underflow branch, float32 the accurate one.
template <typename T>
__device__ __forceinline__ float quick_gelu_elem(float x, float alpha) {
  if constexpr (std::is_same_v<T, __half>) return quick_gelu_f16(x, alpha);
  else if constexpr (std::is_same_v<T, __nv_bfloat16>) return quick_gelu_bf16(x, -alpha * dev::kLog2e);
  else return quick_gelu_f32(x, alpha);
}

// Elements [0, head) and [head + nfrag*VW, n) are scalar; [head, head + nfrag*VW)
// is the 16-byte-aligned vector body (VW == 1: everything is "body").
template <typename T, int VW>
__global__ void __launch_bounds__(kThreads)
k_quick_gelu(const T* x, T* y, int64_t head, int64_t nfrag, int64_t n, float alpha) {
  dev::pdl_wait();
  dev::pdl_trigger();
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

// ---------------------------------------------------------------------------
// Shared-memory-staged, warp-specialised kernels (the fast path when every
// operand is 16-byte aligned).  A CTA has kEwConsumers consumer threads and one
// producer warp; tiles are kEwTileFrags 16-byte fragments, and each of its
// stages holds one tile of X (and of skip, for BiasAdd), filled by the producer
// with cp.async.bulk copies, with a header naming the tile (-1: no more work)
// and, for BiasAdd, the bias column of its first element.  `full`/`empty`
// mbarriers per stage hand stages between producer and consumers, with no
// CTA-wide barrier.  With EP_EW_CLC the grid has one CTA per tile and running
// CTAs take over the tiles of CTAs they cancel (cluster launch control);
// otherwise a persistent grid takes tiles round-robin.  BiasAdd's bias vector
// is bulk-copied into shared memory once per CTA; within a tile the bias column
// of each fragment advances incrementally (no division per fragment).
// Elements after the last whole fragment are done by block 0's consumers with
// scalar loads.
// ---------------------------------------------------------------------------

constexpr int kEwConsumers = 256;
constexpr int kEwThreads = kEwConsumers + 32;
constexpr int kEwConsumerWarps = kEwConsumers / 32;
constexpr int kEwTileFrags = 1024;  // 16 KB per operand per tile
constexpr int kEwFragsPerThread = kEwTileFrags / kEwConsumers;
constexpr int kEwMaxStages = 8;

// float16 QuickGelu on the fast path: x / (1 + 2^(x * (-alpha log2 e))) with
// the hardware 2^x and reciprocal.  u = inf gives x * 0 (NaN for x = -inf).
__device__ __forceinline__ float quick_gelu_fast(float x, float nal2e) {
  const float u = dev::ex2_approx(x * nal2e);
  return x * dev::rcp_approx(1.0f + u);
}

template <typename T, bool BIAS_ADD>
__global__ void __launch_bounds__(kEwThreads, EP_EW_TMA_MIN_CTAS)
k_elementwise_tma(const T* x, const T* skip, const T* bias, T* y, int64_t nfrag, int64_t n, int64_t C,
                  float alpha, int stages, uint32_t bias_bytes, uint32_t col_step_frag, int head, int bias_rot) {
  constexpr int VW = dev::Vec16<T>::N;
  constexpr int NOPS = BIAS_ADD ? 2 : 1;
  constexpr uint32_t kTileBytes = kEwTileFrags * 16u;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[kEwMaxStages];
  __shared__ __align__(8) uint64_t empty[kEwMaxStages];
  __shared__ __align__(8) uint64_t bias_bar;
  __shared__ __align__(8) uint64_t clc_bar;
  __shared__ __align__(16) uint4 clc_resp;
  __shared__ int64_t tile_of[kEwMaxStages];  // stage header: the tile, or -1
  __shared__ uint32_t col_of[kEwMaxStages];  // BiasAdd: bias column of the tile's first element
  const int tid = threadIdx.x;
  unsigned char* stage0 = smem + bias_bytes;  // bias_bytes is a multiple of 128
  const uint32_t stage_bytes = NOPS * kTileBytes;
  const int64_t ntiles = (nfrag + kEwTileFrags - 1) / kEwTileFrags;
  // the 16-byte-aligned body: elements [head, head + nfrag * VW)
  const T* xb = x + head;
  const T* skb = BIAS_ADD ? skip + head : nullptr;
  T* yb = y + head;

  if (tid == 0) {
    for (int st = 0; st < stages; ++st) {
      dev::mbar_init(&full[st], 1);
      dev::mbar_init(&empty[st], kEwConsumerWarps);
    }
    dev::mbar_init(&bias_bar, 1);
    dev::mbar_init(&clc_bar, 1);
    dev::mbar_init_fence();
  }
  __syncthreads();
  dev::pdl_wait();
  dev::pdl_trigger();
  const bool have_tiles = int64_t(blockIdx.x) < ntiles;

  if (tid >= kEwConsumers) {
    // ---- producer ----
    if (tid != kEwConsumers || !have_tiles) return;
    const uint64_t pol_stream = dev::policy_evict_first();
    if constexpr (BIAS_ADD) {
      if (!bias_rot) {  // else the consumers fill shared memory themselves
        const uint32_t cb = uint32_t(C) * uint32_t(sizeof(T));
        dev::mbar_arrive_expect_tx(&bias_bar, cb);
        dev::bulk_g2s(smem, bias, cb, &bias_bar, dev::policy_evict_last());
      }
    }
    // one CTA per tile: take over the tiles of cancelled CTAs; else round-robin
    const bool use_clc = EP_EW_CLC && int64_t(gridDim.x) == ntiles;
    dev::ClcStream clc(&clc_resp, &clc_bar);
    if (use_clc) clc.request();
    int64_t tile = blockIdx.x;
    dev::Ring ring(stages);
    for (int64_t j = 0;; ++j, ring.next()) {
      const int st = ring.st;
      if (j >= stages && !dev::mbar_wait(&empty[st], ring.phase ^ 1u)) {
        if constexpr (BIAS_ADD) {
          if (!bias_rot) dev::mbar_wait(&bias_bar, 0);
        }
        for (int64_t k = j - stages; k < j; ++k)
          dev::mbar_wait(&full[k % stages], static_cast<uint32_t>((k / stages) & 1));
        clc.drain();
        return;
      }
      tile_of[st] = tile;  // released to the consumers by the arrive below
      if (tile < 0) {
        dev::mbar_arrive(&full[st]);
        break;
      }
      const int64_t f0 = tile * int64_t(kEwTileFrags);
      if constexpr (BIAS_ADD) col_of[st] = static_cast<uint32_t>((f0 * VW) % C);
      const uint32_t bytes = static_cast<uint32_t>(min(int64_t(kEwTileFrags), nfrag - f0)) * 16u;
      unsigned char* dst = stage0 + size_t(st) * stage_bytes;
      dev::mbar_arrive_expect_tx(&full[st], NOPS * bytes);
      dev::bulk_g2s(dst, xb + f0 * VW, bytes, &full[st], pol_stream);
      if constexpr (BIAS_ADD) dev::bulk_g2s(dst + kTileBytes, skb + f0 * VW, bytes, &full[st], pol_stream);
      if (use_clc) {
        tile = clc.next();
      } else {
        tile += gridDim.x;
        if (tile >= ntiles) tile = -1;
      }
    }
    clc.drain();
    return;
  }

  // ---- consumers ----
  const float nal2e = -alpha * dev::kLog2e;
  if (blockIdx.x == 0) {  // scalar head (before the aligned body) and tail (past its last fragment)
    const int64_t tail0 = head + nfrag * VW;
    for (int64_t k = tid; k < head + (n - tail0); k += kEwConsumers) {
      const int64_t e = k < head ? k : tail0 + (k - head);
      const float xv = dev::ld1_stream(x + e);
      float yv;
      if constexpr (BIAS_ADD) yv = bias_add_elem<T>(xv, dev::ld1_keep(bias + e % C), dev::ld1_stream(skip + e));
      else if constexpr (std::is_same_v<T, float>) yv = quick_gelu_f32(xv, alpha);
      else if constexpr (std::is_same_v<T, __nv_bfloat16>) yv = quick_gelu_bf16(xv, nal2e);
      else yv = quick_gelu_fast(xv, nal2e);
      dev::st1_stream(y + e, yv);
    }
  }
  if (!have_tiles) return;
  bool ok = true;
  if constexpr (BIAS_ADD) {
    if (bias_rot) {
      // bias rotated by `head`, so that the body's fragments (which start at
      // element head) read it at 16-byte boundaries: slot j = bias[(j + head) mod C]
      T* sbias = reinterpret_cast<T*>(smem);
      for (int64_t j = tid; j < C; j += kEwConsumers) {
        const int64_t src = j + head < C ? j + head : j + head - C;
        sbias[j] = bias[src];
      }
      dev::named_barrier_sync(1, kEwConsumers);
    } else {
      ok = dev::mbar_wait(&bias_bar, 0);
    }
  }
  const uint32_t Cu = static_cast<uint32_t>(C);
  dev::Ring ring(stages);
  for (;; ring.next()) {
    const int st = ring.st;
    ok = dev::mbar_wait(&full[st], ring.phase) && ok;
    if (!__all_sync(0xffffffffu, ok)) return;
    const int64_t tile = tile_of[st];  // the header is read before the stage is released
    if (tile < 0) return;
    const uint32_t col0 = BIAS_ADD ? col_of[st] : 0u;
    const int64_t f0 = tile * int64_t(kEwTileFrags);
    const int nf = static_cast<int>(min(int64_t(kEwTileFrags), nfrag - f0));
    const unsigned char* src = stage0 + size_t(st) * stage_bytes;
    float a[kEwFragsPerThread][VW];
    float sk[BIAS_ADD ? kEwFragsPerThread : 1][VW];
#pragma unroll
    for (int u = 0; u < kEwFragsPerThread; ++u) {
      const int f = u * kEwConsumers + tid;
      if (f < nf) {
        dev::lds_unpack(reinterpret_cast<const T*>(src) + f * VW, a[u]);
        if constexpr (BIAS_ADD) dev::lds_unpack(reinterpret_cast<const T*>(src + kTileBytes) + f * VW, sk[u]);
      }
    }
    dev::release_stage(&empty[st]);
    uint32_t c = 0;
    if constexpr (BIAS_ADD) {
      c = col0 + uint32_t(tid) * VW;
      c = c % Cu;
    }
#pragma unroll
    for (int u = 0; u < kEwFragsPerThread; ++u) {
      const int f = u * kEwConsumers + tid;
      if (f < nf) {
        if constexpr (BIAS_ADD) {
          float b[VW];
          dev::lds_unpack(reinterpret_cast<const T*>(smem) + c, b);
#pragma unroll
          for (int e = 0; e < VW; ++e) a[u][e] = bias_add_elem<T>(a[u][e], b[e], sk[u][e]);
        } else if constexpr (std::is_same_v<T, float>) {
#pragma unroll
          for (int e = 0; e < VW; ++e) a[u][e] = quick_gelu_f32(a[u][e], alpha);
        } else if constexpr (std::is_same_v<T, __nv_bfloat16>) {
#pragma unroll
          for (int e = 0; e < VW; ++e) a[u][e] = quick_gelu_bf16(a[u][e], nal2e);
        } else {
#pragma unroll
          for (int e = 0; e < VW; ++e) a[u][e] = quick_gelu_fast(a[u][e], nal2e);
        }
        dev::stg_pack_stream(yb + (f0 + f) * VW, a[u]);
      }
      if constexpr (BIAS_ADD) {
        c += col_step_frag;
        if (c >= Cu) c -= Cu;
      }
    }
  }
}

constexpr uint32_t kEwStageBudget = EP_EW_TMA_STAGE_BUDGET;
constexpr int64_t kEwMaxBiasBytes = 64 * 1024;

// `head` elements precede the 16-byte-aligned body (x, skip and y share their
// offset within 16 bytes); `bias_rot`: BiasAdd's bias is staged rotated by
// head (needed when head > 0 or the bias itself is not 16-byte aligned).
template <typename T, bool BIAS_ADD>
cudaError_t launch_ew_tma(const T* x, const T* skip, const T* bias, T* y, int64_t n, int64_t C, float alpha,
                          int sm_count, cudaStream_t stream, int head, bool bias_rot) {
  constexpr int VW = dev::Vec16<T>::N;
  auto fn = k_elementwise_tma<T, BIAS_ADD>;
  const int64_t nfrag = (n - head) / VW;
  const uint32_t bias_bytes = BIAS_ADD ? uint32_t((C * int64_t(sizeof(T)) + 127) / 128 * 128) : 0u;
  const uint32_t stage_bytes = (BIAS_ADD ? 2u : 1u) * kEwTileFrags * 16u;
  const int stages = std::min<int>(kEwMaxStages, std::max<int>(2, kEwStageBudget / stage_bytes));
  const size_t smem = bias_bytes + size_t(stages) * stage_bytes;
  int per_sm = 1;
  cudaError_t e = resident_ctas(reinterpret_cast<const void*>(fn), kEwThreads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t ntiles = (nfrag + kEwTileFrags - 1) / kEwTileFrags;
  // one CTA per tile under launch control, else a persistent grid
  const bool clc = EP_EW_CLC && ntiles <= int64_t(INT32_MAX);
  const unsigned grid = static_cast<unsigned>(
      std::max<int64_t>(1, clc ? ntiles : std::min<int64_t>(ntiles, int64_t(sm_count) * per_sm)));
  const uint32_t step_frag = BIAS_ADD ? uint32_t((int64_t(kEwConsumers) * VW) % C) : 0u;
  return launch(fn, dim3(grid), dim3(kEwThreads), smem, stream, x, skip, bias, y, nfrag, n, C, alpha, stages,
                bias_bytes, step_frag, head, int(bias_rot));
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
  // X, skip and Y at the same offset within 16 bytes: a scalar head, then an
  // aligned body for the staged kernel (the bias may have any alignment)
  const uintptr_t ox = reinterpret_cast<uintptr_t>(x) & 15u;
  const bool same = ox == (reinterpret_cast<uintptr_t>(s) & 15u) && ox == (reinterpret_cast<uintptr_t>(y) & 15u);
  const int64_t head = same ? std::min<int64_t>(a.n, int64_t((16 - ox) & 15u) / int64_t(sizeof(T))) : 0;
  if (EP_EW_TMA && same && a.C % VW == 0 && a.C * int64_t(sizeof(T)) <= kEwMaxBiasBytes &&
      (a.n - head) / VW >= kEwTileFrags) {
    *launches += 1;
    return launch_ew_tma<T, true>(x, s, b, y, a.n, a.C, 0.f, sm_count, stream, int(head), head != 0 || !al16(b));
  }
  cudaError_t e;
  if (a.C % VW == 0 && al16(x) && al16(b) && al16(s) && al16(y)) {
    const int64_t nfrag = a.n / VW;
    e = launch(k_bias_add<T, VW>, dim3(grid_for(nfrag, sm_count)), dim3(kThreads), 0, stream, x, b, s, y, nfrag, a.C);
  } else {
    e = launch(k_bias_add<T, 1>, dim3(grid_for(a.n, sm_count)), dim3(kThreads), 0, stream, x, b, s, y, a.n, a.C);
  }
  if (e == cudaSuccess) *launches += 1;
  return e;
}

template <typename T>
cudaError_t quick_gelu_t(const QuickGeluArgs& a, int sm_count, cudaStream_t stream, int* launches) {
  constexpr int VW = dev::Vec16<T>::N;
  const T* x = static_cast<const T*>(a.x);
  T* y = static_cast<T*>(a.y);
  const uintptr_t ox = reinterpret_cast<uintptr_t>(x) & 15u;
  const uintptr_t oy = reinterpret_cast<uintptr_t>(y) & 15u;
  if (EP_EW_TMA && ox == oy) {  // same offset within 16 bytes: a scalar head, then the aligned body
    const int64_t head = std::min<int64_t>(a.n, int64_t((16 - ox) & 15u) / int64_t(sizeof(T)));
    if ((a.n - head) / VW >= kEwTileFrags) {
      *launches += 1;
      return launch_ew_tma<T, false>(x, nullptr, nullptr, y, a.n, 1, a.alpha, sm_count, stream, int(head), false);
    }
  }
  cudaError_t e;
  if (ox == oy) {
    const int64_t head = std::min<int64_t>(a.n, int64_t((16 - ox) & 15u) / int64_t(sizeof(T)));
    const int64_t nfrag = (a.n - head) / VW;
    e = launch(k_quick_gelu<T, VW>, dim3(grid_for(std::max<int64_t>(nfrag, VW), sm_count)), dim3(kThreads), 0, stream,
               x, y, head, nfrag, a.n, a.alpha);
  } else {
    e = launch(k_quick_gelu<T, 1>, dim3(grid_for(a.n, sm_count)), dim3(kThreads), 0, stream, x, y, int64_t(0), a.n,
               a.n, a.alpha);
  }
  if (e == cudaSuccess) *launches += 1;
  return e;
}

}  // namespace

cudaError_t launch_bias_add(const BiasAddArgs& a, int sm_count, cudaStream_t stream, int* launches) {
  switch (a.t) {
    case DType::F32: return bias_add_t<float>(a, sm_count, stream, launches);
    case DType::F16: return bias_add_t<__half>(a, sm_count, stream, launches);
    default: return bias_add_t<__nv_bfloat16>(a, sm_count, stream, launches);
  }
}

cudaError_t launch_quick_gelu(const QuickGeluArgs& a, int sm_count, cudaStream_t stream, int* launches) {
  switch (a.t) {
    case DType::F32: return quick_gelu_t<float>(a, sm_count, stream, launches);
    case DType::F16: return quick_gelu_t<__half>(a, sm_count, stream, launches);
    default: return quick_gelu_t<__nv_bfloat16>(a, sm_count, stream, launches);
  }
}

// Failure-detection self-test: one thread arms a shared-memory barrier for 16
// bytes that no copy will deliver and waits for it with the given limit, so the
// bounded wait runs out, is counted, and the kernel returns normally.  Nothing
// is in flight when it exits.
__global__ void k_selftest_bounded_wait(uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    dev::mbar_init(&bar, 1);
    dev::mbar_init_fence();
    dev::mbar_arrive_expect_tx(&bar, 16);
    (void)dev::mbar_wait_for(&bar, 0, timeout_ns);
  }
}

cudaError_t launch_selftest_bounded_wait(uint64_t timeout_ns, cudaStream_t stream, int* launches) {
  k_selftest_bounded_wait<<<1, 32, 0, stream>>>(timeout_ns);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t elementwise_pipe_timeouts(unsigned int* count, bool clear) { return read_pipe_timeouts(count, clear); }

}  // namespace ep
