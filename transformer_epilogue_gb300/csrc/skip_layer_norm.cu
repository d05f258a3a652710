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
// variance are two reductions over the registers (warp shuffles, then a named
// barrier or shared memory across the warps of a group): a two-pass variance
// with no second global read.  16-byte-aligned rows take the staged kernel
// (k_skip_layer_norm_tma: rows bulk-copied into shared memory by a producer
// warp, gamma/beta/bias held in shared memory, tiles handed out by cluster
// launch control); other rows the register kernel, which reads gamma/beta/bias
// and a broadcast skip through the read-only path; rows too long for the
// register budget a CTA-per-row kernel that re-reads the row (three passes).
// The streamed tensors use evict-first loads and stores, and every launch is a
// programmatic dependent of the work before it in the stream.
#include <algorithm>
#include <climits>

#include "device_common.cuh"
#include "ep_internal.h"
#include "launch_util.h"
#include "tma_pipe.cuh"
#include "tuning.h"

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
  dev::pdl_wait();
  dev::pdl_trigger();
  constexpr int BS = TPR > 256 ? TPR : 256;
  constexpr int RPC = BS / TPR;  // rows per CTA
  // red_a: the mean; red_b: the variance, by row parity.  A row's reads of a
  // buffer precede the next write to it only through a barrier between them:
  // red_a is next written after this row's variance barrier, and the variance
  // buffer two rows on, after the next row's variance barrier (the RMS form has
  // no mean barrier).
  __shared__ float red_a[BS / 32];
  __shared__ float red_b[2][BS / 32];
  int par = 0;

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
    const float var = dev::group_sum<TPR>(q, red_b[par]) / static_cast<float>(H);
    par ^= 1;
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
  dev::pdl_wait();
  dev::pdl_trigger();
  __shared__ float red_a[32];
  __shared__ float red_b[2][32];  // by row parity, as in k_skip_layer_norm
  int par = 0;
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
    const float var = dev::group_sum<1024>(q, red_b[par]) / static_cast<float>(H);
    par ^= 1;
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
  }
}

// ---------------------------------------------------------------------------
// Shared-memory-staged, warp-specialised kernel (the fast path for 16-byte-
// aligned rows).
//
// A CTA has NC consumer threads (256; 512 for the widest rows) in row groups
// of TPR and one producer warp.  Tiles are RT = NC/TPR consecutive rows; each of the
// `stages` shared-memory stages holds one tile: the RT input rows, then the RT
// skip rows (for a broadcast skip, rows r mod skipRows), and the stage header
// names the tile (-1: no more work).  Per stage, `full` completes when the
// producer's cp.async.bulk copies have landed and `empty` when all consumer
// warps are done with it.  The producer refills a stage as soon as it is empty,
// so up to `stages` tiles are in flight per CTA; consumer groups synchronise
// only among themselves (shuffles, or a named barrier when a row spans several
// warps), never CTA-wide.  With EP_SLN_CLC the grid has one CTA per tile and
// each running CTA takes over the tiles of CTAs it cancels (cluster launch
// control), so faster SMs take more tiles; otherwise a persistent grid takes
// tiles round-robin.  The arithmetic is that of k_skip_layer_norm, reading rows
// from shared memory.
// ---------------------------------------------------------------------------

constexpr int kWsConsumers = 256;
constexpr int kTmaMaxStages = 8;

// Dynamic shared memory: [gamma | beta | bias] (each `param_stride` bytes,
// beta/bias only when present), then the stages.  EXACT: the row is exactly
// TPR*NV fragments, so no column needs a bounds check.
template <typename T, int TPR, int NV, bool EXACT, int PARTS = 1, int NC = kWsConsumers>
__global__ void __launch_bounds__(NC + 32, NC > kWsConsumers ? 1 : EP_SLN_TMA_MIN_CTAS)
k_skip_layer_norm_tma(const SlnKernelArgs a, int stages, int64_t ntiles, uint32_t param_stride) {
  constexpr int VW = dev::Vec16<T>::N;
  constexpr int RT = NC / TPR;
  constexpr int NCW = NC / 32;  // consumer warps
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[kTmaMaxStages];
  __shared__ __align__(8) uint64_t empty[kTmaMaxStages];
  __shared__ __align__(8) uint64_t params_bar;
  __shared__ __align__(8) uint64_t clc_bar;
  __shared__ __align__(16) uint4 clc_resp;
  __shared__ int64_t tile_of[kTmaMaxStages];  // stage header: the tile, or -1
  __shared__ float red_a[NCW];
  __shared__ float red_b[NCW];

  static_assert(PARTS == 1 || (RT == 1 && EXACT && NV % PARTS == 0), "parts: one exact row a tile");
  const int H = static_cast<int>(a.H);  // staged rows are at most 64 KB
  // a stage holds a tile of rows, or one part of a row (input, then skip)
  const uint32_t row_bytes = static_cast<uint32_t>(H) * uint32_t(sizeof(T)) / uint32_t(PARTS);
  const uint32_t tile_bytes = RT * row_bytes;
  const uint32_t stage_bytes = 2 * tile_bytes;
  const bool has_beta = a.beta != nullptr;
  const bool has_bias = a.bias != nullptr;
  // part-staged rows read bias through the read-only path, and gamma/beta too
  // unless they are 16-bit rows whose host gave gamma/beta room in shared
  // memory (param_stride != 0)
  constexpr bool kPartParams = PARTS > 1 && sizeof(T) == 2;
  const uint32_t param_bytes = PARTS > 1 ? (kPartParams ? param_stride * (1u + has_beta) : 0u)
                                         : param_stride * (1u + has_beta + has_bias);
  unsigned char* stage0 = smem + param_bytes;
  const int tid = threadIdx.x;

  if (tid == 0) {
    for (int st = 0; st < stages; ++st) {
      dev::mbar_init(&full[st], 1);
      dev::mbar_init(&empty[st], NCW);
    }
    dev::mbar_init(&params_bar, 1);
    dev::mbar_init(&clc_bar, 1);
    dev::mbar_init_fence();
  }
  __syncthreads();
  dev::pdl_wait();
  dev::pdl_trigger();
  if (int64_t(blockIdx.x) >= ntiles) return;

  if (tid >= NC) {
    // ---- producer: one thread issues every copy of this CTA ----
    if (tid != NC) return;
    const T* in = static_cast<const T*>(a.input);
    const T* sk = static_cast<const T*>(a.skip);
    const uint64_t pol_stream = dev::policy_evict_first();
    const uint64_t pol_keep = dev::policy_evict_last();
    if constexpr (PARTS > 1) {
      if (!kPartParams || param_stride == 0) {
        dev::mbar_arrive(&params_bar);
      } else {
        const uint32_t full_row = static_cast<uint32_t>(H) * uint32_t(sizeof(T));
        dev::mbar_arrive_expect_tx(&params_bar, (1u + has_beta) * full_row);
        dev::bulk_g2s(smem, a.gamma, full_row, &params_bar, pol_keep);
        if (has_beta) dev::bulk_g2s(smem + param_stride, a.beta, full_row, &params_bar, pol_keep);
      }
    } else {
      dev::mbar_arrive_expect_tx(&params_bar, param_bytes / param_stride * row_bytes);
      dev::bulk_g2s(smem, a.gamma, row_bytes, &params_bar, pol_keep);
      if (has_beta) dev::bulk_g2s(smem + param_stride, a.beta, row_bytes, &params_bar, pol_keep);
      if (has_bias) dev::bulk_g2s(smem + param_stride * (1u + has_beta), a.bias, row_bytes, &params_bar, pol_keep);
    }
    // one CTA per tile: take over the tiles of cancelled CTAs; else round-robin
    const bool use_clc = EP_SLN_CLC && int64_t(gridDim.x) == ntiles;
    dev::ClcStream clc(&clc_resp, &clc_bar);
    if (use_clc) clc.request();  // the next tile is asked for while this CTA's own is copied
    int64_t tile = blockIdx.x;
    dev::Ring ring(stages);
    for (int64_t j = 0;; ++j, ring.next()) {
      const int st = ring.st;
      if (j >= stages && !dev::mbar_wait(&empty[st], ring.phase ^ 1u)) {
        // consumers stopped: wait (bounded) for the copies still in flight, then stop
        dev::mbar_wait(&params_bar, 0);
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
      const int64_t r0 = tile * RT;
      const uint32_t nr = static_cast<uint32_t>(min(int64_t(RT), a.rows - r0));
      unsigned char* dst = stage0 + size_t(st) * stage_bytes;
      if constexpr (PARTS > 1) {
        // part p of the input row and of its skip row in the p-th stage from here
        const int64_t sr = a.skip_bcast ? r0 % a.skip_rows : r0;
        const int part_cols = H / PARTS;
        for (int p = 0; p < PARTS; ++p) {
          int sp = st;
          if (p > 0) {
            ++j;
            ring.next();
            sp = ring.st;
            if (j >= stages && !dev::mbar_wait(&empty[sp], ring.phase ^ 1u)) {
              for (int64_t k = j - stages; k < j; ++k)
                dev::mbar_wait(&full[k % stages], static_cast<uint32_t>((k / stages) & 1));
              clc.drain();
              return;
            }
            tile_of[sp] = tile;
          }
          unsigned char* dp = stage0 + size_t(sp) * stage_bytes;
          dev::mbar_arrive_expect_tx(&full[sp], 2u * row_bytes);
          dev::bulk_g2s(dp, in + r0 * H + p * part_cols, row_bytes, &full[sp], pol_stream);
          dev::bulk_g2s(dp + tile_bytes, sk + sr * H + p * part_cols, row_bytes, &full[sp],
                        a.skip_bcast ? pol_keep : pol_stream);
        }
      } else {
      dev::mbar_arrive_expect_tx(&full[st], 2u * nr * row_bytes);
      dev::bulk_g2s(dst, in + r0 * H, nr * row_bytes, &full[st], pol_stream);
      if (!a.skip_bcast) {
        dev::bulk_g2s(dst + tile_bytes, sk + r0 * H, nr * row_bytes, &full[st], pol_stream);
      } else {
        int64_t sr = r0 % a.skip_rows;
        for (uint32_t q = 0; q < nr; ++q) {
          dev::bulk_g2s(dst + tile_bytes + q * row_bytes, sk + sr * H, row_bytes, &full[st], pol_keep);
          if (++sr == a.skip_rows) sr = 0;
        }
      }
      }
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
  T* out = static_cast<T*>(a.output);
  T* sum_out = static_cast<T*>(a.sum_out);
  const T* p_gamma = reinterpret_cast<const T*>(smem);
  const T* p_beta = reinterpret_cast<const T*>(smem + param_stride);
  const T* p_bias = reinterpret_cast<const T*>(smem + param_stride * (1u + has_beta));
  // a parameter fragment: from shared memory, or for part-staged rows from global
  auto param = [&](const T* staged, const void* global, int c, float (&f)[VW]) {
    if (PARTS > 1 && (!kPartParams || param_stride == 0 || global == a.bias)) {
      dev::Frag<T, VW> q;
      q.load_keep(static_cast<const T*>(global) + c);
#pragma unroll
      for (int e = 0; e < VW; ++e) f[e] = q.v[e];
    } else {
      dev::lds_unpack(staged + c, f);
    }
  };
  // the same fragment as 16 raw bytes
  auto param_raw = [&](const T* staged, const void* global, int c) -> uint4 {
    if (PARTS > 1 && (!kPartParams || param_stride == 0 || global == a.bias))
      return dev::ld16_keep(static_cast<const T*>(global) + c);
    return dev::lds16(staged + c);
  };
  // 16-bit types: mixed-precision adds and packed float32 pairs take fewer
  // instructions (16-bit rows of 12288-32768 elements went from 0.78-0.90 of
  // the copy bandwidth to 0.93-0.97); float32 rows, which hold up to 64 values
  // a thread, keep scalar arithmetic, which needs fewer registers
  constexpr bool kLean = sizeof(T) == 2;
  auto load_sum = [&](const T* in, const T* sk, float (&f)[VW]) {
    if constexpr (kLean) {
      dev::lds_add(in, sk, f);
    } else {
      float k[VW];
      dev::lds_unpack(in, f);
      dev::lds_unpack(sk, k);
#pragma unroll
      for (int e = 0; e < VW; ++e) f[e] = __fadd_rn(f[e], k[e]);
    }
  };
  const int g = tid / TPR;
  const int lane = tid % TPR;
  const int bar_id = 1 + g;            // named barrier of a multi-warp group
  const int gwarp0 = (g * TPR) >> 5;   // the group's first warp
  bool ok = dev::mbar_wait(&params_bar, 0);

  dev::Ring ring(stages);
  for (;; ring.next()) {
    const int st = ring.st;
    ok = dev::mbar_wait(&full[st], ring.phase) && ok;
    if constexpr (TPR > 32) ok = dev::named_barrier_and(bar_id, TPR, ok);
    else ok = __all_sync(0xffffffffu, ok);
    if (!ok) return;
    const int64_t tile = tile_of[st];  // the same for every consumer
    if (tile < 0) return;

    const int64_t r = tile * RT + g;
    const bool active = r < a.rows;
    float s[NV][VW];
    if constexpr (PARTS > 1) {
      // part p of the row (fragments [p PV, (p+1) PV)) is in the p-th stage
      constexpr int PV = NV / PARTS;
      const int part_cols = H / PARTS;
#pragma unroll
      for (int p = 0; p < PARTS; ++p) {
        if (p > 0) {
          ring.next();
          if (!dev::named_barrier_and(bar_id, TPR, dev::mbar_wait(&full[ring.st], ring.phase))) return;
        }
        const unsigned char* stage = stage0 + size_t(ring.st) * stage_bytes;
        const T* s_in = reinterpret_cast<const T*>(stage);
        const T* s_sk = reinterpret_cast<const T*>(stage + tile_bytes);
        // one row a tile (RT == 1): the tile's row always exists
#pragma unroll
        for (int v = p * PV; v < (p + 1) * PV; ++v) {
          const int c = (v * TPR + lane) * VW - p * part_cols;
          load_sum(s_in + c, s_sk + c, s[v]);
        }
        dev::release_stage(&empty[ring.st]);
      }
    } else {
      const unsigned char* stage = stage0 + size_t(st) * stage_bytes;
      const T* s_in = reinterpret_cast<const T*>(stage) + g * H;
      const T* s_sk = reinterpret_cast<const T*>(stage + tile_bytes) + g * H;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int c = (v * TPR + lane) * VW;
        if (active && (EXACT || c < H)) {
          load_sum(s_in + c, s_sk + c, s[v]);
        } else {
#pragma unroll
          for (int e = 0; e < VW; ++e) s[v][e] = 0.f;
        }
      }
      dev::release_stage(&empty[st]);
    }

    const int64_t off = r * H;
    if (active && (has_bias || sum_out != nullptr)) {
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int c = (v * TPR + lane) * VW;
        if (EXACT || c < H) {
          if (has_bias) {
            if constexpr (kLean) {
              dev::add_raw<T>(param_raw(p_bias, a.bias, c), s[v]);
            } else {
              float b[VW];
              param(p_bias, a.bias, c, b);
#pragma unroll
              for (int e = 0; e < VW; ++e) s[v][e] = __fadd_rn(s[v][e], b[e]);
            }
          }
          if (sum_out != nullptr) dev::stg_pack_stream(sum_out + off + c, s[v]);
        }
      }
    }
    float mean = 0.f;
    float var;
    if constexpr (kLean) {
      // sums over pairs of lanes (packed float32), then the two halves
      if (!a.simplified) {
        float2 t2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
          for (int e = 0; e < VW; e += 2) t2 = __fadd2_rn(t2, make_float2(s[v][e], s[v][e + 1]));
        mean = dev::group_sum_named<TPR>(t2.x + t2.y, red_a, bar_id, gwarp0) / static_cast<float>(H);
      }
      // s becomes s - mean from here on
      float2 q2 = make_float2(0.f, 0.f);
      const float2 nm = make_float2(-mean, -mean);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int c = (v * TPR + lane) * VW;
#pragma unroll
        for (int e = 0; e < VW; e += 2) {
          const float2 d = __fadd2_rn(make_float2(s[v][e], s[v][e + 1]), nm);
          s[v][e] = d.x;
          s[v][e + 1] = d.y;
          if (EXACT || c < H) q2 = __ffma2_rn(d, d, q2);
        }
      }
      var = dev::group_sum_named<TPR>(q2.x + q2.y, red_b, bar_id, gwarp0) / static_cast<float>(H);
    } else {
      if (!a.simplified) {
        float t = 0.f;
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
          for (int e = 0; e < VW; ++e) t += s[v][e];
        mean = dev::group_sum_named<TPR>(t, red_a, bar_id, gwarp0) / static_cast<float>(H);
      }
      // s becomes s - mean from here on
      float q = 0.f;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int c = (v * TPR + lane) * VW;
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          s[v][e] -= mean;
          if (EXACT || c < H) q = fmaf(s[v][e], s[v][e], q);
        }
      }
      var = dev::group_sum_named<TPR>(q, red_b, bar_id, gwarp0) / static_cast<float>(H);
    }
    const float rstd = 1.0f / sqrtf(var + a.eps);
    if (active) {
      if (lane == 0) {
        if (a.mean_out != nullptr) a.mean_out[r] = mean;
        if (a.inv_std_out != nullptr) a.inv_std_out[r] = rstd;
      }
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int c = (v * TPR + lane) * VW;
        if (EXACT || c < H) {
          float gm[VW], y[VW];
          param(p_gamma, a.gamma, c, gm);
          const float2 rs = make_float2(rstd, rstd);
          if constexpr (!kLean) {
            if (has_beta) {
              float bt[VW];
              param(p_beta, a.beta, c, bt);
#pragma unroll
              for (int e = 0; e < VW; ++e) y[e] = fmaf(s[v][e] * rstd, gm[e], bt[e]);
            } else {
#pragma unroll
              for (int e = 0; e < VW; ++e) y[e] = (s[v][e] * rstd) * gm[e];
            }
          } else if (has_beta) {
            float bt[VW];
            param(p_beta, a.beta, c, bt);
#pragma unroll
            for (int e = 0; e < VW; e += 2) {
              const float2 t = __ffma2_rn(__fmul2_rn(make_float2(s[v][e], s[v][e + 1]), rs),
                                          make_float2(gm[e], gm[e + 1]), make_float2(bt[e], bt[e + 1]));
              y[e] = t.x;
              y[e + 1] = t.y;
            }
          } else {
#pragma unroll
            for (int e = 0; e < VW; e += 2) {
              const float2 t = __fmul2_rn(__fmul2_rn(make_float2(s[v][e], s[v][e + 1]), rs),
                                          make_float2(gm[e], gm[e + 1]));
              y[e] = t.x;
              y[e + 1] = t.y;
            }
          }
          dev::stg_pack_stream(out + off + c, y);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// launch planning
// ---------------------------------------------------------------------------

using KernelFn = void (*)(SlnKernelArgs);

// Row-group shapes (threads per row TPR, fragments per thread NV) compiled for
// each (T, VW), in order of capacity TPR*NV*VW; the first that holds the row is
// taken.  Every shape keeps at most 32 floats of the row per thread.  The
// largest holds 32768 elements of a 16-byte-aligned row (1024 threads, one row
// per CTA: 64 registers a thread, with a few values spilled, which measured
// 2.7-3.2x faster than the three-pass kernel for rows of 20480-32768) and 16384
// of another row.  Longer rows use the three-pass kernel.

template <typename T, int VW>
KernelFn pick_kernel(int64_t H, int* tpr_out) {
  const int64_t nfrag = H / VW;
#define EP_SLN_CASE(TPR_, NV_)                          \
  if (nfrag <= int64_t(TPR_) * NV_) {                   \
    *tpr_out = TPR_;                                    \
    return k_skip_layer_norm<T, VW, TPR_, NV_>;         \
  }
  if constexpr (VW == 8) {
    EP_SLN_CASE(4, 1) EP_SLN_CASE(8, 1) EP_SLN_CASE(16, 1)
    EP_SLN_CASE(32, 1) EP_SLN_CASE(32, 2) EP_SLN_CASE(32, 4) EP_SLN_CASE(64, 4)
    EP_SLN_CASE(128, 4) EP_SLN_CASE(256, 4) EP_SLN_CASE(512, 4) EP_SLN_CASE(1024, 4)
  } else if constexpr (VW == 4) {
    EP_SLN_CASE(4, 1) EP_SLN_CASE(8, 1) EP_SLN_CASE(16, 1)
    EP_SLN_CASE(32, 1) EP_SLN_CASE(32, 2) EP_SLN_CASE(32, 4) EP_SLN_CASE(32, 8)
    EP_SLN_CASE(64, 8) EP_SLN_CASE(128, 8) EP_SLN_CASE(256, 8) EP_SLN_CASE(512, 8) EP_SLN_CASE(1024, 8)
  } else {
    EP_SLN_CASE(32, 1) EP_SLN_CASE(32, 2) EP_SLN_CASE(32, 4) EP_SLN_CASE(32, 8)
    EP_SLN_CASE(64, 8) EP_SLN_CASE(128, 8) EP_SLN_CASE(256, 8) EP_SLN_CASE(512, 8)
    EP_SLN_CASE(512, 16) EP_SLN_CASE(512, 32)
  }
#undef EP_SLN_CASE
  return nullptr;
}

// Row shapes of the staged kernel.  A row of nfrag = H/VW 16-byte fragments
// is split over TPR threads (a power of two, 4 to 256) holding NV fragments
// each; a CTA's 256 consumer threads take RT = 256/TPR rows per tile.
//
// Measured on GB300 (64-256 MB operands, hidden sizes 32 to 8192), a shape
// that covers the row exactly runs at the copy bandwidth when NV is 3 to 5;
// NV = 6 to 8 of 8-half fragments loses up to a fifth, and a ragged shape (idle
// lanes in the last fragment column) a quarter.  So the exact shape with the
// smallest NV >= 3 (TPR = nfrag/NV, the largest such power of two) is taken,
// then NV = 2 and 1 (rows of 8 and 4 fragments).  Short rows take 4 or 8
// threads a row (64 or 32 rows a tile): H = 32-128 in float16 went from 0.55-0.72
// of the copy bandwidth on the register kernel to 0.8-1.04.  Rows with no
// exact shape and at least 32 fragments take the first TPR whose NV <= 8
// fragments hold the row and whose tile is at most kTmaTileBytes (TPR = 256
// takes any tile); shorter ones the register kernel.
constexpr uint32_t kTmaTileBytes = EP_SLN_TMA_TILE_BYTES;
constexpr uint32_t kTmaStageBudget = EP_SLN_TMA_STAGE_BUDGET;  // shared memory for the stages of one CTA

using TmaFn = void (*)(SlnKernelArgs, int, int64_t, uint32_t);

// the power-of-two TPR in [4, 256] with TPR*nv == nfrag, else 0
inline int exact_tpr(int64_t nfrag, int nv) {
  if (nfrag % nv != 0) return 0;
  const int64_t t = nfrag / nv;
  return (t >= 4 && t <= 256 && (t & (t - 1)) == 0) ? static_cast<int>(t) : 0;
}

// Rows of 16385-32768 elements that 512 threads cover exactly and that the
// shapes below do not take (16-bit rows of 24576 and 32768; float32 rows of
// every multiple of 2048 up to 24576, and 32768): one row a tile on 512
// consumer threads holding NV fragments each (40-64 floats),
// staged in NV/2 parts of 16 KB (NV odd: NV parts of 8 KB), gamma/beta/bias
// through the read-only path; the CTA runs alone on its SM and takes as many
// stages as fit, so the next row streams in while the consumers reduce and
// write this one.
constexpr int kWideTpr = 512;
template <typename T, int NV>
TmaFn wide_kernel() {
  return k_skip_layer_norm_tma<T, kWideTpr, NV, true, (NV % 2 == 0 ? NV / 2 : NV), kWideTpr>;
}

// 16-bit rows of 18432-30720 elements (multiples of 2048 other than 24576): 4
// fragments a thread on nfrag / 4 consumer threads (576-960, whole warps); more warps than
// 512 threads holding 5-7 fragments hide more of each row's two reductions.
// The row is staged in halves, or in quarters above 24576 elements, so that
// gamma and beta still fit in shared memory beside three stages.  (Rows of
// 24576 stay on 512 threads of 6 fragments: 0.91 of the copy bandwidth
// against 0.88 on 768 threads of 4; 28672 went from 0.82 to 0.91 on 896.)
// float32 rows of 26624-30720 take 8 fragments (32 floats) a thread on the
// same H/32 threads, staged in quarters: 0.73-0.85 of the copy bandwidth on
// 512 threads of 13-15 fragments (which spill), 0.88-0.90 here; shorter float32
// rows measured 3-4 % slower this way and stay on 512 threads.
template <typename T, int TPR> constexpr int wide4_parts() {
  return sizeof(T) == 4 ? 4 : (TPR > 768 ? 4 : 2);
}
template <typename T, int TPR>
TmaFn wide4_kernel() {
  constexpr int NV = 32 / dev::Vec16<T>::N;  // 32 elements a thread
  return k_skip_layer_norm_tma<T, TPR, NV, true, wide4_parts<T, TPR>(), TPR>;
}

template <typename T>
TmaFn pick_wide4_kernel(int64_t nfrag, int* parts, int* consumers) {
  constexpr int NV = 32 / dev::Vec16<T>::N;
  if (nfrag % (64 * NV) != 0) return nullptr;
  const int64_t tpr = nfrag / NV;
  *parts = tpr > 768 ? wide4_parts<T, 832>() : wide4_parts<T, 576>();
  *consumers = static_cast<int>(tpr);
  if constexpr (sizeof(T) == 2) {
    switch (tpr) {
      case 576: return wide4_kernel<T, 576>();
      case 640: return wide4_kernel<T, 640>();
      case 704: return wide4_kernel<T, 704>();
      default: break;
    }
  }
  switch (tpr) {
    case 832: return wide4_kernel<T, 832>();
    case 896: return wide4_kernel<T, 896>();
    case 960: return wide4_kernel<T, 960>();
    default: return nullptr;
  }
}

template <typename T>
TmaFn pick_wide_kernel(int64_t nfrag, int* parts) {
  constexpr int VW = dev::Vec16<T>::N;
  if (nfrag % kWideTpr != 0) return nullptr;
  const int64_t nv = nfrag / kWideTpr;
  *parts = static_cast<int>(nv % 2 == 0 ? nv / 2 : nv);
  if constexpr (VW == 8) {
    switch (nv) {
      case 5: return wide_kernel<T, 5>();
      case 6: return wide_kernel<T, 6>();
      case 7: return wide_kernel<T, 7>();
      case 8: return wide_kernel<T, 8>();
      default: return nullptr;
    }
  } else {
    switch (nv) {
      case 9: return wide_kernel<T, 9>();
      case 10: return wide_kernel<T, 10>();
      case 11: return wide_kernel<T, 11>();
      case 12: return wide_kernel<T, 12>();
      case 13: return wide_kernel<T, 13>();
      case 14: return wide_kernel<T, 14>();
      case 15: return wide_kernel<T, 15>();
      case 16: return wide_kernel<T, 16>();
      default: return nullptr;
    }
  }
}

template <typename T>
TmaFn pick_tma_kernel(int64_t H, int* rows_per_tile, int* parts, int* consumers) {
  constexpr int VW = dev::Vec16<T>::N;
  const int64_t nfrag = H / VW;
  *parts = 1;
  *consumers = kWsConsumers;
  if (nfrag < 4) return nullptr;
  if (EP_SLN_WIDE && H > 16384) {
    *rows_per_tile = 1;
    if (VW == 8 ? EP_SLN_WIDE_NV4 : EP_SLN_WIDE_NV8)
      if (TmaFn f = pick_wide4_kernel<T>(nfrag, parts, consumers)) return f;
    *consumers = kWideTpr;
    return pick_wide_kernel<T>(nfrag, parts);
  }
  // exact shapes; the compiled set is every (TPR, NV) this search can return
  for (int nv : {3, 4, 5, 6, 7, 8, 2, 1, 12, 16}) {
    const int tpr = exact_tpr(nfrag, nv);
    if (tpr == 0) continue;
    *rows_per_tile = kWsConsumers / tpr;
    // float32 rows of 12288 and 16384 (48 and 64 floats a thread): staged in
    // 16 KB parts, gamma/beta/bias read through the read-only path (whole rows
    // of them would fill shared memory).  Measured at 256 MB: 0.62-0.69 of the
    // copy bandwidth on the register kernel, 0.93-0.97 here.  (16-bit rows of
    // 12288 in two parts measured no faster than whole rows.)
    if constexpr (VW == 4) {
      if (tpr == 256 && nv == 12) {
        *parts = 3;
        return k_skip_layer_norm_tma<T, 256, 12, true, 3>;
      }
      if (tpr == 256 && nv == 16) {
        *parts = 4;
        return k_skip_layer_norm_tma<T, 256, 16, true, 4>;
      }
    }
#define EP_SLN_TMA_EXACT(TPR_, NV_) \
    if (tpr == TPR_ && nv == NV_) return k_skip_layer_norm_tma<T, TPR_, NV_, true>;
    EP_SLN_TMA_EXACT(4, 3) EP_SLN_TMA_EXACT(8, 3) EP_SLN_TMA_EXACT(16, 3) EP_SLN_TMA_EXACT(32, 3)
    EP_SLN_TMA_EXACT(64, 3) EP_SLN_TMA_EXACT(128, 3) EP_SLN_TMA_EXACT(256, 3)
    EP_SLN_TMA_EXACT(4, 4) EP_SLN_TMA_EXACT(8, 4) EP_SLN_TMA_EXACT(16, 4) EP_SLN_TMA_EXACT(32, 4)
    EP_SLN_TMA_EXACT(64, 4) EP_SLN_TMA_EXACT(128, 4) EP_SLN_TMA_EXACT(256, 4)
    EP_SLN_TMA_EXACT(4, 5) EP_SLN_TMA_EXACT(8, 5) EP_SLN_TMA_EXACT(16, 5) EP_SLN_TMA_EXACT(32, 5)
    EP_SLN_TMA_EXACT(64, 5) EP_SLN_TMA_EXACT(128, 5) EP_SLN_TMA_EXACT(256, 5)
    EP_SLN_TMA_EXACT(256, 6)  // NV = 6 or 8 below TPR = 256 is NV = 3 or 4 at twice the TPR
    EP_SLN_TMA_EXACT(4, 7) EP_SLN_TMA_EXACT(8, 7) EP_SLN_TMA_EXACT(16, 7) EP_SLN_TMA_EXACT(32, 7)
    EP_SLN_TMA_EXACT(64, 7) EP_SLN_TMA_EXACT(128, 7) EP_SLN_TMA_EXACT(256, 7)
    EP_SLN_TMA_EXACT(256, 8)
    EP_SLN_TMA_EXACT(4, 2)    // NV = 2 and 1 are reached only for nfrag = 8 and 4
    EP_SLN_TMA_EXACT(4, 1)
#undef EP_SLN_TMA_EXACT
    return nullptr;
  }
  if (nfrag < 32) return nullptr;
  const int64_t row_bytes = H * int64_t(sizeof(T));
  for (int tpr : {16, 32, 64, 128, 256}) {
    const int64_t nv = (nfrag + tpr - 1) / tpr;
    if (nv > 8) continue;
    const int rt = kWsConsumers / tpr;
    if (rt * row_bytes > kTmaTileBytes && tpr != 256) continue;
    *rows_per_tile = rt;
#define EP_SLN_TMA_RAGGED(TPR_, NV_) \
    if (tpr == TPR_ && nv <= NV_) return k_skip_layer_norm_tma<T, TPR_, NV_, false>;
    EP_SLN_TMA_RAGGED(16, 4) EP_SLN_TMA_RAGGED(32, 4) EP_SLN_TMA_RAGGED(64, 4) EP_SLN_TMA_RAGGED(128, 4)
    EP_SLN_TMA_RAGGED(256, 4) EP_SLN_TMA_RAGGED(256, 8)
#undef EP_SLN_TMA_RAGGED
    return nullptr;
  }
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
  // rows of 2 or 3 fragments: one thread a row on the register kernel, which
  // runs no reduction across threads (256 MB: float32 H = 8 and 12 0.56-0.74 ->
  // 0.98-1.00 of the copy bandwidth, float16 H = 16 0.41 -> 0.69; rows of 4
  // fragments measured slower this way than on 4-thread staged rows)
  if (vec && EP_SLN_SHORT_REG && a.H / VW >= 2 && a.H / VW <= 3) {
    KernelFn fn = a.H / VW == 2 ? k_skip_layer_norm<T, VW, 1, 2> : k_skip_layer_norm<T, VW, 1, 3>;
    const int64_t need = (a.rows + 255) / 256;
    const int64_t cap = int64_t(sm_count) * 64 * 8;
    cudaError_t el = launch(fn, dim3(static_cast<unsigned>(std::min(need, cap))), dim3(256), 0, stream, k);
    if (el != cudaSuccess) return el;
    *launches += 1;
    return cudaGetLastError();
  }
  if (vec && EP_SLN_TMA) {
    int rt = 0, parts = 1, consumers = kWsConsumers;
    if (TmaFn f = pick_tma_kernel<T>(a.H, &rt, &parts, &consumers)) {
      const uint32_t row_bytes = uint32_t(a.H * int64_t(sizeof(T)));
      const uint32_t stage_bytes = 2u * uint32_t(rt) * row_bytes / uint32_t(parts);
      const uint32_t param_stride = (row_bytes + 127u) / 128u * 128u;
      uint32_t param_bytes = parts > 1 ? 0u : param_stride * (1u + (a.beta != nullptr) + (a.bias != nullptr));
      // 16-bit wide rows (more than 256 consumers): gamma and beta in shared
      // memory (they fit beside three stages up to 32768 elements)
      uint32_t pstride = param_stride;
      if (parts > 1) {
        const uint32_t gb = param_stride * (1u + (a.beta != nullptr));
        if (EP_SLN_WIDE_PARAMS && sizeof(T) == 2 && consumers > kWsConsumers && gb + 3u * stage_bytes <= 224u * 1024u) {
          param_bytes = gb;
        } else {
          pstride = 0;
        }
      }
      int stages = std::min<int>(kTmaMaxStages, std::max<int>(parts > 1 ? 3 : 2, kTmaStageBudget / stage_bytes));
      // A CTA whose parameters and two stages already exceed half of shared
      // memory, or whose threads fill the register file, runs alone on its SM:
      // give it as many stages as fit, so that more rows are in flight (f16
      // H = 10240-12288, f32 H = 5120-6144, and the wide rows).
      constexpr uint32_t kSmemForStages = 224u * 1024u;
      const bool alone = consumers > kWsConsumers ||
                         (param_bytes + 2u * stage_bytes > kSmemForStages / 2 &&
                          param_bytes + 2u * stage_bytes <= kSmemForStages);
      if (alone)
        stages = std::min<int>(kTmaMaxStages, std::max<int>(stages, int((kSmemForStages - param_bytes) / stage_bytes)));
      // never more stages than fit beside the parameters
      if (param_bytes + uint32_t(stages) * stage_bytes > kSmemForStages)
        stages = std::max<int>(2, int((kSmemForStages - std::min(param_bytes, kSmemForStages)) / stage_bytes));
      if (2 * stage_bytes <= 2 * kTmaStageBudget && (param_bytes <= 96u * 1024u || consumers > kWsConsumers)) {
        const size_t smem = param_bytes + size_t(stages) * stage_bytes;
        const int threads = consumers + 32;
        int per_sm = 1;
        cudaError_t e = resident_ctas(reinterpret_cast<const void*>(f), threads, smem, &per_sm);
        if (e != cudaSuccess) return e;
        const int64_t ntiles = (a.rows + rt - 1) / rt;
        // one CTA per tile under launch control, else a persistent grid
        const bool clc = EP_SLN_CLC && ntiles <= int64_t(INT32_MAX);
        const unsigned grid = static_cast<unsigned>(clc ? ntiles : std::min<int64_t>(ntiles, int64_t(sm_count) * per_sm));
        e = launch(f, dim3(grid), dim3(threads), smem, stream, k, stages, ntiles, pstride);
        if (e == cudaSuccess) *launches += 1;
        return e;
      }
    }
  }
  int tpr = 0;
  KernelFn fn = vec ? pick_kernel<T, VW>(a.H, &tpr) : pick_kernel<T, 1>(a.H, &tpr);
  if (fn != nullptr) {
    const int bs = std::max(tpr, 256);
    const int rpc = bs / tpr;
    const int64_t need = (a.rows + rpc - 1) / rpc;
    const int64_t cap = int64_t(sm_count) * 64 * (2048 / bs);  // many waves, then grid-stride
    const unsigned grid = static_cast<unsigned>(std::min(need, cap));
    cudaError_t e = launch(fn, dim3(grid), dim3(bs), 0, stream, k);
    if (e == cudaSuccess) *launches += 1;
    return e;
  }
  const int64_t cap = int64_t(sm_count) * 2 * 16;
  const unsigned grid = static_cast<unsigned>(std::min(a.rows, cap));
  cudaError_t e = launch(k_skip_layer_norm_long<T>, dim3(grid), dim3(1024), 0, stream, k);
  if (e == cudaSuccess) *launches += 1;
  return e;
}

}  // namespace

cudaError_t launch_skip_layer_norm(const SlnArgs& a, int sm_count, cudaStream_t stream, int* launches) {
  switch (a.t) {
    case DType::F32: return launch_t<float>(a, sm_count, stream, launches);
    case DType::F16: return launch_t<__half>(a, sm_count, stream, launches);
    default: return launch_t<__nv_bfloat16>(a, sm_count, stream, launches);
  }
}

cudaError_t sln_pipe_timeouts(unsigned int* count, bool clear) { return read_pipe_timeouts(count, clear); }

}  // namespace ep
