// BiasSoftmax kernels.
//
// Definition: com.microsoft.BiasSoftmax manifest, `description`, `derive`
// (axisNorm, batchCount, blockSize, biasBlockCount, biasContract) and
// `attributeDescriptions.is_inner_broadcast`: output[r] = softmax(data[r] +
// bias[br(r)]) over blockSize columns, br(r) = r / innerRepeat (inner) or
// r % biasBlockCount (outer).  The manifest's variants `adaptive_row` (one
// workgroup per row) and `longrow_split` (block_stats -> row_stats ->
// normalize, rows >= 65536) are the prior art for the two paths below.
//
// Row path (rows of at most 16384 elements): a group of TPR threads owns a row;
// z is kept in float32 registers, so data and output cross HBM once.  Max and
// sum are warp-shuffle (+ named-barrier) reductions.  16-byte-aligned rows take
// the staged kernel (k_bias_softmax_rows_tma) from 12 fragments on and the
// register kernel below that; other rows the register kernel; rows of at most
// 8 elements, other than aligned rows of exactly 8, a thread-per-row kernel.
//
// Split-row path (longer rows): rows are cut into 16 KB chunks and a pair of
// launches runs over them:
//   pass 1: per chunk (or per CTA's part of a row) (m_b, s_b) =
//           (max z, sum exp(z - m_b)) -> workspace
//   pass 2: M = max m_b, S = sum s_b exp(m_b - M) per row (the manifest's
//           separate row_stats pass is folded in here), then the chunk is
//           read again and exp(z - M) / S written.
// The staged pair (k_softmax_split_tma) serves 16-byte-aligned rows, the
// register pair (k_softmax_chunk_stats / k_softmax_chunk_normalize) the rest.
// The host runs the pair over windows of rows sized to stay resident in L2,
// so the second read of a chunk is normally served from L2, not HBM.  Every
// launch is a programmatic dependent of the work before it in the stream.
#include <algorithm>
#include <climits>
#include <atomic>
#include <cmath>

#include "device_common.cuh"
#include "ep_internal.h"
#include "launch_util.h"
#include "tma_pipe.cuh"
#include "tuning.h"

namespace ep {
namespace {

using dev::Frag;

struct SmKernelArgs {
  const void* data;
  const void* bias;
  void* output;
  int64_t rows;
  int64_t cols;
  int64_t bias_rows;
  int64_t inner_repeat;
  bool inner;
};

__device__ __forceinline__ int64_t bias_row(const SmKernelArgs& a, int64_t r) {
  return a.inner ? r / a.inner_repeat : r % a.bias_rows;
}

template <typename T, int VW, int TPR, int NV, bool EXACT = false>
__global__ void __launch_bounds__(TPR > 256 ? TPR : 256)
k_bias_softmax_rows(const SmKernelArgs a) {
  dev::pdl_wait();
  dev::pdl_trigger();
  constexpr int BS = TPR > 256 ? TPR : 256;
  constexpr int RPC = BS / TPR;
  // 16-byte fragments of a 16-bit type: data added to the bias by
  // mixed-precision adds, the exponent as a packed fused multiply-add
  constexpr bool k16 = sizeof(T) == 2 && VW == 8;
  __shared__ float red_a[BS / 32];
  __shared__ float red_b[BS / 32];
  const T* data = static_cast<const T*>(a.data);  // may alias output (in place)
  const T* __restrict__ bias = static_cast<const T*>(a.bias);
  T* out = static_cast<T*>(a.output);
  const int g = threadIdx.x / TPR;
  const int lane = threadIdx.x % TPR;
  const int64_t C = a.cols;

  for (int64_t base = int64_t(blockIdx.x) * RPC; base < a.rows; base += int64_t(gridDim.x) * RPC) {
    const int64_t r = base + g;
    const bool active = r < a.rows;
    const int64_t off = r * C;
    float z[NV][VW];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int e = 0; e < VW; ++e) z[v][e] = -INFINITY;
    if (active) {
      const int64_t boff = bias_row(a, r) * C;
      if constexpr (k16) {
        // all loads first (raw 16-byte fragments), then one fragment at a time
        uint4 du[NV], bu[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          const int c = (v * TPR + lane) * VW;
          if (EXACT || c < C) {
            du[v] = dev::ld16_stream(data + off + c);
            bu[v] = dev::ld16_keep(bias + boff + c);
          }
        }
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          const int c = (v * TPR + lane) * VW;
          if (EXACT || c < C) {
            float bz[VW];
            dev::Conv<T>::unpack(bu[v], bz);
            const uint32_t w[4] = {du[v].x, du[v].y, du[v].z, du[v].w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dev::MixAdd<T>::add(w[i], bz[2 * i], bz[2 * i + 1], z[v][2 * i], z[v][2 * i + 1]);
          }
        }
      } else {
        Frag<T, VW> d[NV], b[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          const int64_t c = int64_t(v * TPR + lane) * VW;
          if (EXACT || c < C) {
            d[v].load_stream(data + off + c);
            b[v].load_keep(bias + boff + c);
          }
        }
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          const int64_t c = int64_t(v * TPR + lane) * VW;
          if (EXACT || c < C) {
#pragma unroll
            for (int e = 0; e < VW; ++e) z[v][e] = d[v].v[e] + b[v].v[e];
          }
        }
      }
    }
    float m = -INFINITY;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      if constexpr (VW % 2 == 0) {
#pragma unroll
        for (int e = 0; e < VW; e += 2) m = dev::max3(m, z[v][e], z[v][e + 1]);
      } else {
#pragma unroll
        for (int e = 0; e < VW; ++e) m = fmaxf(m, z[v][e]);
      }
    }
    m = dev::group_max<TPR>(m, red_a);
    float s = 0.f;
    if constexpr (k16) {
      float2 acc = make_float2(0.f, 0.f);
      const float2 l2 = make_float2(dev::kLog2e, dev::kLog2e);
      const float2 ml = make_float2(-m * dev::kLog2e, -m * dev::kLog2e);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int c = (v * TPR + lane) * VW;
#pragma unroll
        for (int e = 0; e < VW; e += 2) {
          const float2 t = __ffma2_rn(make_float2(z[v][e], z[v][e + 1]), l2, ml);
          float e0 = dev::ex2_approx(t.x), e1 = dev::ex2_approx(t.y);
          if (!EXACT && c >= C) e0 = e1 = 0.f;
          z[v][e] = e0;
          z[v][e + 1] = e1;
          acc = __fadd2_rn(acc, make_float2(e0, e1));
        }
      }
      s = acc.x + acc.y;
    } else {
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int64_t c = int64_t(v * TPR + lane) * VW;
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          z[v][e] = (EXACT || c < C) ? __expf(z[v][e] - m) : 0.f;
          s += z[v][e];
        }
      }
    }
    s = dev::group_sum<TPR>(s, red_b);
    const float inv = 1.0f / s;
    if (active) {
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int64_t c = int64_t(v * TPR + lane) * VW;
        if (EXACT || c < C) {
          if constexpr (VW % 2 == 0) dev::scale_pairs(z[v], inv);
          else {
#pragma unroll
            for (int e = 0; e < VW; ++e) z[v][e] *= inv;
          }
          if constexpr (VW == 1) dev::st1_stream(out + off + c, z[v][0]);
          else dev::stg_pack_stream(out + off + c, z[v]);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Packed rows (blockSize <= 8, the manifest's `packed_rows` variant): one
// thread per row, grid-stride over rows; the row's few elements stay in
// registers.  Neighbouring threads read neighbouring rows, so a warp's loads
// cover contiguous memory.
// ---------------------------------------------------------------------------

constexpr int kPackedMax = 8;

template <typename T>
__global__ void __launch_bounds__(256) k_bias_softmax_packed(const SmKernelArgs a) {
  dev::pdl_wait();
  dev::pdl_trigger();
  const T* data = static_cast<const T*>(a.data);
  const T* __restrict__ bias = static_cast<const T*>(a.bias);
  T* out = static_cast<T*>(a.output);
  const int C = static_cast<int>(a.cols);
  const bool small = a.rows < (int64_t(1) << 31);
  for (int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; r < a.rows; r += int64_t(gridDim.x) * blockDim.x) {
    int64_t br;
    if (small) {  // 32-bit division when the indices fit
      const uint32_t r32 = static_cast<uint32_t>(r);
      br = a.inner ? r32 / static_cast<uint32_t>(a.inner_repeat) : r32 % static_cast<uint32_t>(a.bias_rows);
    } else {
      br = bias_row(a, r);
    }
    const T* d = data + r * C;
    const T* b = bias + br * C;
    float z[kPackedMax];
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kPackedMax; ++j) {
      if (j < C) {
        z[j] = dev::ld1_stream(d + j) + dev::ld1_keep(b + j);
        m = fmaxf(m, z[j]);
      }
    }
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < kPackedMax; ++j) {
      if (j < C) {
        z[j] = __expf(z[j] - m);
        sum += z[j];
      }
    }
    const float inv = 1.0f / sum;
    T* o = out + r * C;
#pragma unroll
    for (int j = 0; j < kPackedMax; ++j)
      if (j < C) dev::st1_stream(o + j, z[j] * inv);
  }
}

// ---------------------------------------------------------------------------
// Shared-memory-staged, warp-specialised row kernel (the fast path for
// 16-byte-aligned rows).
//
// A CTA has NC consumer threads (256; 512 for the widest rows) in row groups
// of TPR and one producer warp.  Tiles are RT = NC/TPR consecutive data rows.  A
// stage holds the tile's data rows and, after them, only the distinct bias
// rows those data rows use (at most `bias_slots`):
//   inner broadcast: bias rows r0/ir .. (r0+nr-1)/ir, one contiguous copy;
//   outer, biasRows <= RT: all bias rows;
//   outer, biasRows > RT: bias rows (r0 + j) mod biasRows, one or two copies.
// The producer also writes the tile (-1: no more work) and each row's bias
// slot into the stage's header, so consumers do no index division.
// `full`/`empty` mbarriers per stage hand stages between producer and
// consumers; consumer groups synchronise only among themselves.  With
// EP_SM_CLC the grid has one CTA per tile and running CTAs take over the tiles
// of CTAs they cancel (cluster launch control); otherwise a persistent grid
// takes tiles round-robin.
// ---------------------------------------------------------------------------

constexpr int kWsConsumers = 256;
constexpr int kTmaMaxStages = 8;
// CTAs of 257-416 consumer threads are sized to run two to an SM
constexpr int kWide2Max = 416;

// EXACT: the row is exactly TPR*NV fragments, so no column needs a bounds check.
// PARTS > 1 (one 256-thread row a tile, exact, NV a multiple of PARTS): a tile
// takes PARTS consecutive stages, stage p holding part p of the data row
// (columns [p C/PARTS, (p+1) C/PARTS)) and the same part of its bias row, so
// that stages stay small and two CTAs fit on an SM.  A lane's fragments
// v in [p NV/PARTS, (p+1) NV/PARTS) lie in part p.
template <typename T, int TPR, int NV, bool EXACT, int PARTS = 1, int NC = kWsConsumers>
__global__ void __launch_bounds__(NC + 32, NC > kWsConsumers ? (NC <= kWide2Max ? 2 : 1) : EP_SM_TMA_MIN_CTAS)
k_bias_softmax_rows_tma(const SmKernelArgs a, int stages, int bias_slots, int64_t ntiles) {
  constexpr int VW = dev::Vec16<T>::N;
  constexpr int RT = NC / TPR;
  constexpr int NCW = NC / 32;  // consumer warps
  static_assert(PARTS == 1 || (RT == 1 && EXACT && NV % PARTS == 0), "parts: one exact row a tile");
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[kTmaMaxStages];
  __shared__ __align__(8) uint64_t empty[kTmaMaxStages];
  __shared__ __align__(8) uint64_t clc_bar;
  __shared__ __align__(16) uint4 clc_resp;
  __shared__ int64_t tile_of[kTmaMaxStages];  // stage header: the tile, or -1
  __shared__ int slot_of[kTmaMaxStages][RT];  // sized per shape: static shared memory counts toward occupancy
  __shared__ float red_a[NCW];
  __shared__ float red_b[NCW];

  const int C = static_cast<int>(a.cols);  // staged rows are at most 64 KB
  // a stage holds rows, or one part of a row (and the same part of bias)
  const uint32_t row_bytes = static_cast<uint32_t>(C) * uint32_t(sizeof(T)) / uint32_t(PARTS);
  const uint32_t data_bytes = RT * row_bytes;
  const uint32_t stage_bytes = data_bytes + uint32_t(bias_slots) * row_bytes;
  const int tid = threadIdx.x;

  if (tid == 0) {
    for (int st = 0; st < stages; ++st) {
      dev::mbar_init(&full[st], 1);
      dev::mbar_init(&empty[st], NCW);
    }
    dev::mbar_init(&clc_bar, 1);
    dev::mbar_init_fence();
  }
  __syncthreads();
  dev::pdl_wait();
  dev::pdl_trigger();
  if (int64_t(blockIdx.x) >= ntiles) return;

  if (tid >= NC) {
    // ---- producer ----
    if (tid != NC) return;
    const T* data = static_cast<const T*>(a.data);
    const T* bias = static_cast<const T*>(a.bias);
    const uint64_t pol_stream = dev::policy_evict_first();
    const uint64_t pol_keep = dev::policy_evict_last();
    const bool outer_all = !a.inner && a.bias_rows <= RT;
    // one CTA per tile: take over the tiles of cancelled CTAs; else round-robin
    const bool use_clc = EP_SM_CLC && int64_t(gridDim.x) == ntiles;
    dev::ClcStream clc(&clc_resp, &clc_bar);
    if (use_clc) clc.request();
    int64_t tile = blockIdx.x;
    dev::Ring ring(stages);
    for (int64_t j = 0;; ++j, ring.next()) {
      const int st = ring.st;
      if (j >= stages && !dev::mbar_wait(&empty[st], ring.phase ^ 1u)) {
        for (int64_t k = j - stages; k < j; ++k)
          dev::mbar_wait(&full[k % stages], static_cast<uint32_t>((k / stages) & 1));
        clc.drain();
        return;
      }
      tile_of[st] = tile;  // released to the consumers with the header below
      if (tile < 0) {
        dev::mbar_arrive(&full[st]);
        break;
      }
      const int64_t r0 = tile * RT;
      const int nr = static_cast<int>(min(int64_t(RT), a.rows - r0));
      int64_t b0 = 0, n1 = 0, n2 = 0;  // bias rows [b0, b0+n1) then [0, n2)
      if (a.inner) {
        b0 = r0 / a.inner_repeat;
        n1 = (r0 + nr - 1) / a.inner_repeat - b0 + 1;
        int64_t b = b0, left = a.inner_repeat - (r0 - b0 * a.inner_repeat);
        for (int q = 0; q < nr; ++q) {
          slot_of[st][q] = static_cast<int>(b - b0);
          if (--left == 0) { ++b; left = a.inner_repeat; }
        }
      } else if (outer_all) {
        n1 = a.bias_rows;
        int64_t b = r0 % a.bias_rows;
        for (int q = 0; q < nr; ++q) {
          slot_of[st][q] = static_cast<int>(b);
          if (++b == a.bias_rows) b = 0;
        }
      } else {
        b0 = r0 % a.bias_rows;
        n1 = min(int64_t(nr), a.bias_rows - b0);
        n2 = int64_t(nr) - n1;
        for (int q = 0; q < nr; ++q) slot_of[st][q] = q;
      }
      unsigned char* dst = smem + size_t(st) * stage_bytes;
      unsigned char* bdst = dst + data_bytes;
      if constexpr (PARTS > 1) {
        // part 0 here, part p in the p-th stage after it
        const int64_t part_cols = C / PARTS;
        dev::mbar_arrive_expect_tx(&full[st], 2u * row_bytes);
        dev::bulk_g2s(dst, data + r0 * C, row_bytes, &full[st], pol_stream);
        dev::bulk_g2s(bdst, bias + b0 * C, row_bytes, &full[st], pol_keep);
        for (int p = 1; p < PARTS; ++p) {
          ++j;
          ring.next();
          const int sp = ring.st;
          if (j >= stages && !dev::mbar_wait(&empty[sp], ring.phase ^ 1u)) {
            for (int64_t k = j - stages; k < j; ++k)
              dev::mbar_wait(&full[k % stages], static_cast<uint32_t>((k / stages) & 1));
            clc.drain();
            return;
          }
          tile_of[sp] = tile;
          slot_of[sp][0] = 0;
          unsigned char* dp = smem + size_t(sp) * stage_bytes;
          dev::mbar_arrive_expect_tx(&full[sp], 2u * row_bytes);
          dev::bulk_g2s(dp, data + r0 * C + p * part_cols, row_bytes, &full[sp], pol_stream);
          dev::bulk_g2s(dp + data_bytes, bias + b0 * C + p * part_cols, row_bytes, &full[sp], pol_keep);
        }
      } else {
        // the arrive releases the slot_of writes above to the consumers
        dev::mbar_arrive_expect_tx(&full[st], uint32_t(nr) * row_bytes + uint32_t(n1 + n2) * row_bytes);
        dev::bulk_g2s(dst, data + r0 * C, uint32_t(nr) * row_bytes, &full[st], pol_stream);
        dev::bulk_g2s(bdst, bias + b0 * C, uint32_t(n1) * row_bytes, &full[st], pol_keep);
        if (n2 > 0) dev::bulk_g2s(bdst + n1 * row_bytes, bias, uint32_t(n2) * row_bytes, &full[st], pol_keep);
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
  const int g = tid / TPR;
  const int lane = tid % TPR;
  const int bar_id = 1 + g;
  const int gwarp0 = (g * TPR) >> 5;

  dev::Ring ring(stages);
  for (;; ring.next()) {
    const int st = ring.st;
    bool ok = dev::mbar_wait(&full[st], ring.phase);
    if constexpr (TPR > 32) ok = dev::named_barrier_and(bar_id, TPR, ok);
    else ok = __all_sync(0xffffffffu, ok);
    if (!ok) return;
    const int64_t tile = tile_of[st];  // the same for every consumer
    if (tile < 0) return;

    const int64_t r = tile * RT + g;
    const bool active = r < a.rows;
    float z[NV][VW];
    if constexpr (PARTS > 1) {
      // part p of the row (fragments [p PV, (p+1) PV)) is in the p-th stage
      constexpr int PV = NV / PARTS;
      const int part_cols = C / PARTS;
#pragma unroll
      for (int p = 0; p < PARTS; ++p) {
        if (p > 0) {
          ring.next();
          if (!dev::named_barrier_and(bar_id, TPR, dev::mbar_wait(&full[ring.st], ring.phase))) return;
        }
        const T* s_d = reinterpret_cast<const T*>(smem + size_t(ring.st) * stage_bytes);
        const T* s_b = reinterpret_cast<const T*>(smem + size_t(ring.st) * stage_bytes + data_bytes);
        // one row a tile (RT == 1): the tile's row always exists
#pragma unroll
        for (int v = p * PV; v < (p + 1) * PV; ++v) {
          const int c = (v * TPR + lane) * VW - p * part_cols;
          dev::lds_add(s_d + c, s_b + c, z[v]);
        }
        dev::release_stage(&empty[ring.st]);
      }
    } else {
      const unsigned char* stage = smem + size_t(st) * stage_bytes;
      const T* s_d = reinterpret_cast<const T*>(stage) + g * C;
      const T* s_b = reinterpret_cast<const T*>(stage + data_bytes) + (active ? slot_of[st][g] : 0) * C;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int c = (v * TPR + lane) * VW;
        if (active && (EXACT || c < C)) {
          dev::lds_add(s_d + c, s_b + c, z[v]);
        } else {
#pragma unroll
          for (int e = 0; e < VW; ++e) z[v][e] = -INFINITY;
        }
      }
      dev::release_stage(&empty[st]);
    }

    float m = z[0][0];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int e = 0; e < VW; e += 2) m = dev::max3(m, z[v][e], z[v][e + 1]);
    m = dev::group_max_named<TPR>(m, red_a, bar_id, gwarp0);
    float sum = 0.f;
    if constexpr (sizeof(T) == 2 && EP_SM_LEAN16) {
      // 16-bit results: the exponent z log2e - m log2e as one packed fused
      // multiply-add per pair (its extra rounding, a few float32 ulp of
      // |m log2e|, is far below a 16-bit result's spacing), and two sums
      float2 acc = make_float2(0.f, 0.f);
      const float2 l2 = make_float2(dev::kLog2e, dev::kLog2e);
      const float2 ml = make_float2(-m * dev::kLog2e, -m * dev::kLog2e);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int c = (v * TPR + lane) * VW;
#pragma unroll
        for (int e = 0; e < VW; e += 2) {
          const float2 t = __ffma2_rn(make_float2(z[v][e], z[v][e + 1]), l2, ml);
          float e0 = dev::ex2_approx(t.x), e1 = dev::ex2_approx(t.y);
          if (!EXACT && c >= C) e0 = e1 = 0.f;
          z[v][e] = e0;
          z[v][e + 1] = e1;
          acc = __fadd2_rn(acc, make_float2(e0, e1));
        }
      }
      sum = acc.x + acc.y;
    } else {
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int c = (v * TPR + lane) * VW;
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          float ev = dev::ex2_approx((z[v][e] - m) * dev::kLog2e);
          if (!EXACT && c >= C) ev = 0.f;
          z[v][e] = ev;
          sum += ev;
        }
      }
    }
    sum = dev::group_sum_named<TPR>(sum, red_b, bar_id, gwarp0);
    const float inv = 1.0f / sum;
    if (active) {
      T* orow = out + r * C;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int c = (v * TPR + lane) * VW;
        if (EXACT || c < C) {
          dev::scale_pairs(z[v], inv);
          dev::stg_pack_stream(orow + c, z[v]);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// split-row path.  A row is cut into chunks of kChunkBytes (4096 float32 or
// 8192 float16 columns); pass 1 writes each chunk's (max z, sum exp(z - max))
// to the workspace, pass 2 combines a row's chunk statistics into
// M = max m_b, S = sum s_b exp(m_b - M) and writes exp(z - M) / S.
// ---------------------------------------------------------------------------

constexpr int kSplitThreads = 256;
constexpr int64_t kChunkBytes = 16384;
template <typename T> constexpr int64_t chunk_cols() { return kChunkBytes / int64_t(sizeof(T)); }
template <typename T, int VW> struct SplitNV {
  static constexpr int value = int(chunk_cols<T>() / kSplitThreads / VW);
};

// Register path (any alignment): one 256-thread CTA per chunk.
// Loads the chunk's z = data + bias (columns beyond the row are -inf).
template <typename T, int VW, int NV = SplitNV<T, VW>::value>
__device__ __forceinline__ void load_chunk(const SmKernelArgs& a, int64_t r, int64_t c0,
                                           Frag<T, VW> (&z)[NV]) {
  const T* data = static_cast<const T*>(a.data);
  const T* bias = static_cast<const T*>(a.bias);
  const int64_t off = r * a.cols;
  const int64_t boff = bias_row(a, r) * a.cols;
  Frag<T, VW> b[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int64_t c = c0 + int64_t(v * kSplitThreads + threadIdx.x) * VW;
    if (c < a.cols) {
      z[v].load_stream(data + off + c);
      b[v].load_keep(bias + boff + c);
    }
  }
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int64_t c = c0 + int64_t(v * kSplitThreads + threadIdx.x) * VW;
#pragma unroll
    for (int e = 0; e < VW; ++e) z[v].v[e] = (c < a.cols) ? z[v].v[e] + b[v].v[e] : -INFINITY;
  }
}

template <typename T, int VW>
__global__ void __launch_bounds__(kSplitThreads)
k_softmax_chunk_stats(const SmKernelArgs a, int64_t row0, int64_t nrows, int64_t nchunks, float2* stats) {
  dev::pdl_wait();
  dev::pdl_trigger();
  __shared__ float red_a[kSplitThreads / 32];
  __shared__ float red_b[kSplitThreads / 32];
  const int64_t total = nrows * nchunks;
  for (int64_t blk = blockIdx.x; blk < total; blk += gridDim.x) {
    const int64_t r = row0 + blk / nchunks;
    const int64_t ch = blk % nchunks;
    constexpr int NV = SplitNV<T, VW>::value;
    Frag<T, VW> z[NV];
    load_chunk<T, VW>(a, r, ch * chunk_cols<T>(), z);
    float m = -INFINITY;
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int e = 0; e < VW; ++e) m = fmaxf(m, z[v].v[e]);
    m = dev::group_max<kSplitThreads>(m, red_a);
    float s = 0.f;
    if (m != -INFINITY) {
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int e = 0; e < VW; ++e) s += __expf(z[v].v[e] - m);
    }
    s = dev::group_sum<kSplitThreads>(s, red_b);
    if (threadIdx.x == 0) stats[r * nchunks + ch] = make_float2(m, s);
  }
}

template <typename T, int VW>
__global__ void __launch_bounds__(kSplitThreads)
k_softmax_chunk_normalize(const SmKernelArgs a, int64_t row0, int64_t nrows, int64_t nchunks,
                          const float2* stats) {
  dev::pdl_wait();
  dev::pdl_trigger();
  __shared__ float red_a[kSplitThreads / 32];
  __shared__ float red_b[kSplitThreads / 32];
  constexpr int NV = SplitNV<T, VW>::value;
  T* out = static_cast<T*>(a.output);
  const int64_t total = nrows * nchunks;
  for (int64_t blk = blockIdx.x; blk < total; blk += gridDim.x) {
    const int64_t r = row0 + blk / nchunks;
    const int64_t ch = blk % nchunks;
    // issue this chunk's loads first; the row combine below overlaps them
    Frag<T, VW> z[NV];
    load_chunk<T, VW>(a, r, ch * chunk_cols<T>(), z);
    const float2* st = stats + r * nchunks;
    float M = -INFINITY;
    for (int64_t j = threadIdx.x; j < nchunks; j += kSplitThreads) M = fmaxf(M, st[j].x);
    M = dev::group_max<kSplitThreads>(M, red_a);
    float S = 0.f;
    for (int64_t j = threadIdx.x; j < nchunks; j += kSplitThreads) {
      const float2 p = st[j];
      if (p.x != -INFINITY) S += p.y * __expf(p.x - M);
    }
    S = dev::group_sum<kSplitThreads>(S, red_b);
    const float inv = 1.0f / S;
    const int64_t off = r * a.cols;
    const int64_t c0 = ch * chunk_cols<T>();
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int64_t c = c0 + int64_t(v * kSplitThreads + threadIdx.x) * VW;
      if (c < a.cols) {
#pragma unroll
        for (int e = 0; e < VW; ++e) z[v].v[e] = __expf(z[v].v[e] - M) * inv;
        z[v].store_stream(out + off + c);
      }
    }
  }
}

// Staged path (16-byte-aligned rows): warp-specialised and persistent, each CTA
// owning a contiguous range of the window's chunks (so it meets few rows).  A
// chunk is streamed through shared memory as kSpTiles tiles; a stage holds one
// tile of data and the matching tile of its bias row, so many small stages keep
// enough bytes in flight per SM.  Each of the 8 consumer warps takes a 1/8 slice
// of every tile.  Pass 1 keeps running statistics per lane and combines the
// lanes and warps only where the CTA's part of a row ends; pass 2's producer
// warp combines a row's chunk statistics when the row changes and hands
// (M, 1/S) to the consumers in the stage header.

constexpr int kSpConsumers = 256;
constexpr int kSpThreads = kSpConsumers + 32;
constexpr int kSpWarps = kSpConsumers / 32;
constexpr int kSpMaxStages = 16;
constexpr int64_t kSpTileBytes = EP_SM_SPLIT_TILE_BYTES;
constexpr int64_t kSpTiles = kChunkBytes / kSpTileBytes;  // tiles per chunk
static_assert(kChunkBytes % kSpTileBytes == 0, "a chunk is a whole number of tiles");
static_assert(kSpTileBytes % (kSpConsumers * 16) == 0, "every consumer lane takes whole 16-byte fragments");
template <typename T> constexpr int sp_tile_cols() { return int(kSpTileBytes / int64_t(sizeof(T))); }

// Walks the tiles of a CTA's range in order: tile s of chunk kc of row r.
struct SplitCursor {
  int64_t r, kc;
  int s;
  __device__ __forceinline__ void start(int64_t row0, int64_t nchunks, int64_t chunk) {
    r = row0 + chunk / nchunks;
    kc = chunk % nchunks;
    s = 0;
  }
  __device__ __forceinline__ void next(int64_t nchunks) {
    if (++s == kSpTiles) {
      s = 0;
      if (++kc == nchunks) {
        kc = 0;
        ++r;
      }
    }
  }
  template <typename T> __device__ __forceinline__ int64_t col() const {
    return kc * chunk_cols<T>() + int64_t(s) * sp_tile_cols<T>();
  }
  // columns in this tile (<= 0 past the end of the row)
  template <typename T> __device__ __forceinline__ int width(int64_t cols) const {
    return static_cast<int>(min(int64_t(sp_tile_cols<T>()), cols - col<T>()));
  }
};

// Range [lo, hi) of the window's chunks owned by this CTA.
__device__ __forceinline__ void split_range(int64_t total, int64_t* lo, int64_t* hi) {
  const int64_t q = total / gridDim.x, rem = total % gridDim.x, b = blockIdx.x;
  *lo = b * q + min(b, rem);
  *hi = *lo + q + (b < rem ? 1 : 0);
}

// z = data + bias for one lane's fragments of a staged tile (columns c0 +
// v * 32 * VW); fragments at or past column `tw` are -inf unless WHOLE says the
// tile is full.
template <typename T, int NV, int VW, bool WHOLE>
__device__ __forceinline__ void split_load_z(const T* sd, const T* sb, int c0, int tw, float (&z)[NV][VW]) {
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int c = c0 + v * 32 * VW;
    if (WHOLE || c < tw) {
      dev::lds_add(sd + c, sb + c, z[v]);
    } else {
#pragma unroll
      for (int e = 0; e < VW; ++e) z[v][e] = -INFINITY;
    }
  }
}

// y = e^(z - M) / S for one lane's fragments, stored where they lie in the row.
template <typename T, int NV, int VW, bool WHOLE>
__device__ __forceinline__ void split_store_y(T* orow, int c0, int tw, const float (&z)[NV][VW], float2 h) {
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int c = c0 + v * 32 * VW;
    if (WHOLE || c < tw) {
      float y[VW];
      if constexpr (sizeof(T) == 2) {
        // 16-bit results: the exponent as one packed fused multiply-add per pair
        const float2 l2 = make_float2(dev::kLog2e, dev::kLog2e);
        const float2 ml = make_float2(-h.x * dev::kLog2e, -h.x * dev::kLog2e);
#pragma unroll
        for (int e = 0; e < VW; e += 2) {
          const float2 t = __ffma2_rn(make_float2(z[v][e], z[v][e + 1]), l2, ml);
          y[e] = dev::ex2_approx(t.x);
          y[e + 1] = dev::ex2_approx(t.y);
        }
        dev::scale_pairs(y, h.y);
      } else {
#pragma unroll
        for (int e = 0; e < VW; ++e) y[e] = dev::ex2_approx((z[v][e] - h.x) * dev::kLog2e) * h.y;
      }
      dev::stg_pack_stream(orow + c, y);
    }
  }
}

template <typename T, bool STATS>
__global__ void __launch_bounds__(kSpThreads)
k_softmax_split_tma(const SmKernelArgs a, int64_t row0, int64_t nrows, int64_t nchunks, float2* stats, int stages) {
  constexpr int VW = dev::Vec16<T>::N;
  constexpr int SLICE = sp_tile_cols<T>() / kSpWarps;  // columns per consumer warp
  constexpr int NV = SLICE / 32 / VW;                   // fragments per lane
  constexpr uint32_t kStageBytes = 2 * uint32_t(kSpTileBytes);
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[kSpMaxStages];
  __shared__ __align__(8) uint64_t empty[kSpMaxStages];
  __shared__ float2 hdr[kSpMaxStages];     // pass 2: (M, 1/S) of the stage's row
  __shared__ float2 part[2][kSpWarps];     // pass 1: per-warp statistics of a row segment
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  int64_t lo, hi;
  split_range(nrows * nchunks, &lo, &hi);
  const int64_t mine = (hi - lo) * kSpTiles;  // tiles in the range

  if (tid == 0) {
    for (int st = 0; st < stages; ++st) {
      // pass 2: the producer arrives twice per stage (copies armed; header written)
      dev::mbar_init(&full[st], STATS ? 1 : 2);
      dev::mbar_init(&empty[st], kSpWarps);
    }
    dev::mbar_init_fence();
  }
  __syncthreads();
  // pass 1 waits for the work before it, then lets the (programmatically
  // dependent) pass 2 be scheduled as its CTAs retire; pass 2's producer waits
  // for pass 1 below, before it reads the chunk statistics
  if (STATS) {
    dev::pdl_wait();
    dev::pdl_trigger();
  }
  if (mine <= 0) return;

  if (warp == kSpWarps) {
    // ---- producer warp: lane 0 copies; pass 2 also combines row statistics ----
    const T* data = static_cast<const T*>(a.data);
    const T* bias = static_cast<const T*>(a.bias);
    const uint64_t pol_data = STATS ? dev::policy_evict_last() : dev::policy_evict_first();
    const uint64_t pol_keep = dev::policy_evict_last();
    // lane 0: fill the next stage with tile n of the range (waiting for it to
    // be empty first); false if the consumers stopped.  A tile past the end of
    // its row completes its stage with no bytes.
    SplitCursor fc;  // the tile the next fill copies
    fc.start(row0, nchunks, lo);
    dev::Ring fring(stages);  // its stage
    auto fill = [&](int64_t n) -> bool {
      const int st = fring.st;
      if (n >= stages && !dev::mbar_wait(&empty[st], fring.phase ^ 1u)) {
        for (int64_t k = n - stages; k < n; ++k)
          dev::mbar_wait(&full[k % stages], static_cast<uint32_t>((k / stages) & 1));
        return false;
      }
      const int w = fc.width<T>(a.cols);
      unsigned char* dst = smem + size_t(st) * kStageBytes;
      const uint32_t bytes = w > 0 ? uint32_t(w) * uint32_t(sizeof(T)) : 0u;
      dev::mbar_arrive_expect_tx(&full[st], 2u * bytes);
      if (bytes) {
        const int64_t c = fc.col<T>();
        dev::bulk_g2s(dst, data + fc.r * a.cols + c, bytes, &full[st], pol_data);
        dev::bulk_g2s(dst + kSpTileBytes, bias + bias_row(a, fc.r) * a.cols + c, bytes, &full[st], pol_keep);
      }
      fc.next(nchunks);
      fring.next();
      return true;
    };
    const int64_t pre = min(int64_t(stages), mine);
    if (lane == 0)
      for (int64_t n = 0; n < pre; ++n) fill(n);
    if (STATS) {
      if (lane == 0)
        for (int64_t n = pre; n < mine; ++n)
          if (!fill(n)) break;
      return;
    }

    // pass 2: the statistics come from pass 1, which may still be finishing
    dev::pdl_wait();
    dev::pdl_trigger();
    int64_t cur_row = -1;
    float2 cur = make_float2(0.f, 0.f);
    SplitCursor hc;  // the tile whose header is written next
    hc.start(row0, nchunks, lo);
    dev::Ring hring(stages);
    for (int64_t n = 0; n < mine; ++n, hc.next(nchunks), hring.next()) {
      int stop = 0;
      if (n >= pre && lane == 0) stop = fill(n) ? 0 : 1;
      if (__shfl_sync(0xffffffffu, stop, 0)) break;  // the whole warp stops together
      const int64_t r = hc.r;
      if (r != cur_row) {
        // M = max m_b, S = sum s_b e^(m_b - M) over the row's chunks, 8 pairs per
        // lane in flight, merged online across blocks of 256 pairs
        const float2* sp = stats + r * nchunks;
        float M = -INFINITY, S = 0.f;
        for (int64_t q0 = 0; q0 < nchunks; q0 += 256) {
          float2 p[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int64_t q = q0 + k * 32 + lane;
            p[k] = q < nchunks ? sp[q] : make_float2(-INFINITY, 0.f);
          }
          float mb = p[0].x;
#pragma unroll
          for (int k = 1; k < 8; ++k) mb = fmaxf(mb, p[k].x);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
          float sb = 0.f;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (p[k].x != -INFINITY) sb += p[k].y * dev::ex2_approx((p[k].x - mb) * dev::kLog2e);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sb += __shfl_xor_sync(0xffffffffu, sb, o);
          const float Mn = fmaxf(M, mb);
          if (Mn != -INFINITY) {
            S = (M != -INFINITY ? S * dev::ex2_approx((M - Mn) * dev::kLog2e) : 0.f) +
                (mb != -INFINITY ? sb * dev::ex2_approx((mb - Mn) * dev::kLog2e) : 0.f);
          }
          M = Mn;
        }
        cur = make_float2(M, 1.0f / S);
        cur_row = r;
      }
      if (lane == 0) {
        const int st = hring.st;
        hdr[st] = cur;
        dev::mbar_arrive(&full[st]);  // releases the header with the second arrival
      }
    }
    return;
  }

  // ---- consumers ----
  float ml = -INFINITY, sl = 0.f;  // pass 1: this lane's running (max, sum e^(z - max))
  bool failed = false;             // this warp saw a wait run out: it reads no more stages
  int seg = 0;
  T* out = static_cast<T*>(a.output);
  SplitCursor t;
  t.start(row0, nchunks, lo);
  dev::Ring ring(stages);
  for (int64_t n = 0; n < mine; ++n, t.next(nchunks), ring.next()) {
    const int st = ring.st;
    const int tw = t.width<T>(a.cols);
    if (!failed) failed = !__all_sync(0xffffffffu, dev::mbar_wait(&full[st], ring.phase));
    if constexpr (!STATS) {
      if (failed) return;  // pass 2's consumers never meet at a barrier
    }
    if (!failed) {
      const T* sd = reinterpret_cast<const T*>(smem + size_t(st) * kStageBytes);
      const T* sb = reinterpret_cast<const T*>(smem + size_t(st) * kStageBytes + kSpTileBytes);
      const bool whole = tw == sp_tile_cols<T>();
      const int c0 = warp * SLICE + lane * VW;
      float z[NV][VW];
      if (whole) split_load_z<T, NV, VW, true>(sd, sb, c0, tw, z);
      else split_load_z<T, NV, VW, false>(sd, sb, c0, tw, z);
      float2 h = make_float2(0.f, 0.f);
      if (!STATS) h = hdr[st];
      dev::release_stage(&empty[st]);

      if constexpr (STATS) {
        float cm = -INFINITY;
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
          for (int e = 0; e < VW; e += 2) cm = dev::max3(cm, z[v][e], z[v][e + 1]);
        const float mn = fmaxf(ml, cm);
        if (mn != -INFINITY) {
          float acc0 = sl * dev::ex2_approx((ml - mn) * dev::kLog2e);  // ml = -inf gives 0
          float acc1 = 0.f;
          if constexpr (sizeof(T) == 2) {
            // 16-bit data: the exponent as one packed fused multiply-add per pair
            const float2 l2 = make_float2(dev::kLog2e, dev::kLog2e);
            const float2 nl = make_float2(-mn * dev::kLog2e, -mn * dev::kLog2e);
            float2 acc = make_float2(acc0, acc1);
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
              for (int e = 0; e < VW; e += 2) {
                const float2 t = __ffma2_rn(make_float2(z[v][e], z[v][e + 1]), l2, nl);
                acc = __fadd2_rn(acc, make_float2(dev::ex2_approx(t.x), dev::ex2_approx(t.y)));
              }
            acc0 = acc.x;
            acc1 = acc.y;
          } else {
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
              for (int e = 0; e < VW; e += 2) {
                acc0 += dev::ex2_approx((z[v][e] - mn) * dev::kLog2e);
                acc1 += dev::ex2_approx((z[v][e + 1] - mn) * dev::kLog2e);
              }
          }
          sl = acc0 + acc1;
          ml = mn;
        }
      } else {
        T* orow = out + t.r * a.cols + t.col<T>();
        if (whole) split_store_y<T, NV, VW, true>(orow, c0, tw, z, h);
        else split_store_y<T, NV, VW, false>(orow, c0, tw, z, h);
      }
    }

    if constexpr (STATS) {
      // Where a chunk ends: if the CTA's part of the row ends too, combine the
      // lanes and warps into the part's (max, sum) and store it as this chunk's
      // statistics; otherwise store (-inf, 0), which pass 2's combine skips.
      if (t.s != kSpTiles - 1) continue;
      const bool seg_end = n + 1 == mine || t.kc + 1 == nchunks;
      if (!seg_end) {
        if (tid == 0) stats[t.r * nchunks + t.kc] = make_float2(-INFINITY, 0.f);
        continue;
      }
      float M = ml;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      float S = (ml != -INFINITY) ? sl * dev::ex2_approx((ml - M) * dev::kLog2e) : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
      // double-buffered by segment parity: warp 0 has read part[seg & 1] before
      // it meets the next segment's barrier, which comes before any rewrite
      if (lane == 0) part[seg & 1][warp] = make_float2(M, S);
      // the consumers meet here only, and decide together whether to stop
      if (!dev::named_barrier_and(2, kSpConsumers, !failed)) return;
      if (warp == 0) {
        const float2 p = part[seg & 1][lane & (kSpWarps - 1)];
        float Mc = p.x;
#pragma unroll
        for (int o = kSpWarps / 2; o > 0; o >>= 1) Mc = fmaxf(Mc, __shfl_xor_sync(0xffffffffu, Mc, o));
        float Sc = (p.x != -INFINITY) ? p.y * dev::ex2_approx((p.x - Mc) * dev::kLog2e) : 0.f;
#pragma unroll
        for (int o = kSpWarps / 2; o > 0; o >>= 1) Sc += __shfl_xor_sync(0xffffffffu, Sc, o);
        if (lane == 0) stats[t.r * nchunks + t.kc] = make_float2(Mc, Sc);
      }
      ml = -INFINITY;
      sl = 0.f;
      ++seg;
    }
  }
}

// ---------------------------------------------------------------------------
// launch planning
// ---------------------------------------------------------------------------

using RowFn = void (*)(SmKernelArgs);

// Row-group shapes per (T, VW) in order of capacity; each keeps at most 32
// floats of the row per thread.  The largest holds kRowMax columns; longer rows
// take the split-row path.
constexpr int64_t kRowMax = 16384;

template <typename T, int VW>
RowFn pick_row_kernel(int64_t cols, int* tpr_out) {
  const int64_t nfrag = cols / VW;
#define EP_SM_CASE(TPR_, NV_)                        \
  if (nfrag <= int64_t(TPR_) * NV_) {                \
    *tpr_out = TPR_;                                 \
    return k_bias_softmax_rows<T, VW, TPR_, NV_>;    \
  }
  // Rows of 1-11 16-byte fragments: groups of 1, 2 or 4 threads holding 1-11
  // fragments each, exact (no column checks) but for float32 rows of 7, 9 and
  // 11 fragments.  Against groups of 4, 8 or 16 threads holding one fragment
  // this shares each row's reductions, reciprocal and index arithmetic among
  // more elements a thread: at 256 MB float16 rows of 32 and 64 columns went
  // from 0.58 to 0.98-0.99 of the copy bandwidth, float32 rows of 16 and 32
  // from 0.77 to 1.0 (groups of 4 threads with idle lanes measured slower).
#define EP_SM_SHORT_X(N_, TPR_, NV_, EX_) \
  case N_: *tpr_out = TPR_; return k_bias_softmax_rows<T, VW, TPR_, NV_, EX_>;
  if constexpr (VW > 1) {
    if (nfrag * VW == cols && nfrag >= 1 && nfrag <= 11) {
      switch (nfrag) {
        EP_SM_SHORT_X(1, 1, 1, true) EP_SM_SHORT_X(2, 1, 2, true) EP_SM_SHORT_X(3, 1, 3, true) EP_SM_SHORT_X(4, 2, 2, true)
        EP_SM_SHORT_X(5, 1, 5, true) EP_SM_SHORT_X(6, 2, 3, true)
        EP_SM_SHORT_X(8, 4, 2, true) EP_SM_SHORT_X(10, 2, 5, true)
        default: break;
      }
      // 7, 9 or 11 fragments: a thread holding the whole row (16-bit, 0.71-0.77
      // of the copy bandwidth against 0.59-0.67 on two threads with an idle
      // fragment); float32 rows, whose one-thread form holds 28-44 floats, run
      // better on two threads (0.74 / 0.64 / 0.69 against 0.71 / 0.61 / 0.62)
      if constexpr (VW == 4) {
        switch (nfrag) {
          EP_SM_SHORT_X(7, 2, 4, false) EP_SM_SHORT_X(9, 2, 5, false) EP_SM_SHORT_X(11, 2, 6, false)
          default: break;
        }
      } else {
        switch (nfrag) {
          EP_SM_SHORT_X(7, 1, 7, true) EP_SM_SHORT_X(9, 1, 9, true) EP_SM_SHORT_X(11, 1, 11, true)
          default: break;
        }
      }
    }
  }
#undef EP_SM_SHORT_X
  // (16-byte fragments: rows of up to 11 fragments never get here)
  if constexpr (VW == 8) {
    EP_SM_CASE(16, 1)
    EP_SM_CASE(32, 1) EP_SM_CASE(32, 2) EP_SM_CASE(32, 4) EP_SM_CASE(64, 4)
    EP_SM_CASE(128, 4) EP_SM_CASE(256, 4) EP_SM_CASE(512, 4)
  } else if constexpr (VW == 4) {
    EP_SM_CASE(16, 1)
    EP_SM_CASE(32, 1) EP_SM_CASE(32, 2) EP_SM_CASE(32, 4) EP_SM_CASE(32, 8)
    EP_SM_CASE(64, 8) EP_SM_CASE(128, 8) EP_SM_CASE(256, 8) EP_SM_CASE(512, 8)
  } else {
    EP_SM_CASE(32, 1) EP_SM_CASE(32, 2) EP_SM_CASE(32, 4) EP_SM_CASE(32, 8)
    EP_SM_CASE(64, 8) EP_SM_CASE(128, 8) EP_SM_CASE(256, 8) EP_SM_CASE(512, 8)
    EP_SM_CASE(512, 16) EP_SM_CASE(512, 32)
  }
#undef EP_SM_CASE
  return nullptr;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T>
bool vec_ok(const void* data, const void* bias, const void* out, int64_t cols) {
  return cols % dev::Vec16<T>::N == 0 && al16(data) && al16(bias) && al16(out);
}

template <typename T, int VW>
cudaError_t launch_split(const SmKernelArgs& k, const SoftmaxArgs& a, int sm_count, int l2_bytes,
                         cudaStream_t stream, int* launches) {
  const int64_t nchunks = (a.cols + chunk_cols<T>() - 1) / chunk_cols<T>();
  float2* stats = static_cast<float2*>(a.workspace);
  // rows per window: keep a window's data within a fraction of L2 so that the
  // second read (normalize) hits L2
  const int64_t row_bytes = a.cols * int64_t(sizeof(T));
  const int64_t budget = std::max<int64_t>(int64_t(l2_bytes) * EP_SM_SPLIT_WINDOW_QUARTERS / 4, 1);
  const int64_t win = std::max<int64_t>(1, budget / row_bytes);
  if constexpr (VW > 1) {
    if (EP_SM_TMA) {
      const int stages = std::min<int>(kSpMaxStages, std::max<int>(2, int(EP_SM_SPLIT_STAGE_BUDGET / (2 * kSpTileBytes))));
      const size_t smem = size_t(stages) * 2 * kSpTileBytes;
      int per1 = 1, per2 = 1;
      cudaError_t e = resident_ctas(reinterpret_cast<const void*>(k_softmax_split_tma<T, true>), kSpThreads, smem, &per1);
      if (e == cudaSuccess)
        e = resident_ctas(reinterpret_cast<const void*>(k_softmax_split_tma<T, false>), kSpThreads, smem, &per2);
      if (e != cudaSuccess) return e;
      for (int64_t r0 = 0; r0 < a.rows; r0 += win) {
        const int64_t nr = std::min(win, a.rows - r0);
        const int64_t total = nr * nchunks;
        const unsigned g1 = static_cast<unsigned>(std::min<int64_t>(total, int64_t(sm_count) * per1));
        const unsigned g2 = static_cast<unsigned>(std::min<int64_t>(total, int64_t(sm_count) * per2));
        cudaError_t el = launch(k_softmax_split_tma<T, true>, dim3(g1), dim3(kSpThreads), smem, stream, k, r0, nr,
                                nchunks, stats, stages);
        if (el != cudaSuccess) return el;
        // pass 2 may start while pass 1 drains; it waits for pass 1 (griddepcontrol.wait)
        // before reading the chunk statistics, and reads only data before that
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(g2);
        cfg.blockDim = dim3(kSpThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, k_softmax_split_tma<T, false>, k, r0, nr, nchunks, stats, stages);
        if (e != cudaSuccess) return e;
        *launches += 2;
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
      }
      return cudaSuccess;
    }
  }
  const int64_t cap = int64_t(sm_count) * 8 * 16;
  for (int64_t r0 = 0; r0 < a.rows; r0 += win) {
    const int64_t nr = std::min(win, a.rows - r0);
    const unsigned grid = static_cast<unsigned>(std::min(nr * nchunks, cap));
    cudaError_t e = launch(k_softmax_chunk_stats<T, VW>, dim3(grid), dim3(kSplitThreads), 0, stream, k, r0, nr,
                           nchunks, stats);
    if (e == cudaSuccess)
      e = launch(k_softmax_chunk_normalize<T, VW>, dim3(grid), dim3(kSplitThreads), 0, stream, k, r0, nr, nchunks,
                 static_cast<const float2*>(stats));
    if (e != cudaSuccess) return e;
    *launches += 2;
  }
  return cudaSuccess;
}

using TmaRowFn = void (*)(SmKernelArgs, int, int, int64_t);
constexpr uint32_t kTmaTileBytes = EP_SM_TMA_TILE_BYTES;
constexpr uint32_t kTmaStageBudget = EP_SM_TMA_STAGE_BUDGET;

// Row shapes: a row of nfrag = cols/VW 16-byte fragments is split over TPR
// threads (a power of two, 4 to 256) holding NV fragments each; a tile is
// RT = 256/TPR rows.  Measured on GB300 (128-256 MB of data, row lengths 32 to
// 16384, bias broadcast either way), a shape that covers the row exactly beats
// a ragged one by 10 to 30 %, and among exact shapes NV = 4 to 6 is best
// (NV = 3 loses up to 5 %: the stage also carries bias rows, so fewer, fuller
// threads per row pay off).  So the exact shape with the smallest NV >= 4,
// then NV = 3, then NV = 2.  Short rows take 4 or 8 threads a row: 96-192
// columns of float16 went from 0.43-0.56 of the copy bandwidth on the register
// kernel to 0.8-0.93; rows under 12 fragments stay on the register kernel (a
// 4-thread row of 1 or 2 fragments measured slower).  Rows with no exact shape
// and at least 32 fragments take the first TPR whose NV <= 8 fragments hold
// the row and whose data tile is at most kTmaTileBytes.
inline int exact_tpr(int64_t nfrag, int nv) {
  if (nfrag % nv != 0) return 0;
  const int64_t t = nfrag / nv;
  return (t >= 4 && t <= 256 && (t & (t - 1)) == 0) ? static_cast<int>(t) : 0;
}

// Rows of 16385-32768 columns that 512 threads cover exactly and that the
// shapes below do not take (16-bit rows of 32768, and of 20480-28672 when those
// are switched off; float32 rows of every multiple of 2048): one row a tile on
// 512 consumer threads holding NV fragments each (40-64 floats), staged with
// its bias row in NV/2 parts of 16 KB (NV odd: NV parts of 8 KB); the CTA runs
// alone on its SM and takes as many stages as fit.
constexpr int kWideTpr = 512;
template <typename T, int NV>
TmaRowFn wide_row_kernel() {
  return k_bias_softmax_rows_tma<T, kWideTpr, NV, true, (NV % 2 == 0 ? NV / 2 : NV), kWideTpr>;
}

// 16-bit rows of 28672 and 30720 columns (and, without EP_SM_WIDE_2CTA, every
// multiple of 2048 from 18432): 4 fragments a thread on nfrag / 4 consumer
// threads (576-960, whole warps), the row staged in halves.  Against 512
// threads holding 5-7 fragments each, the extra warps hide more of each row's
// reductions: 0.50-0.62 of the copy bandwidth became 0.65-0.73 (rows of 24576
// and 32768, which 512 threads cover with 6 and 8 fragments, measured the same
// either way; four parts a row measured slower).
template <typename T, int TPR>
TmaRowFn wide4_row_kernel() {
  return k_bias_softmax_rows_tma<T, TPR, 4, true, 2, TPR>;
}

// 16-bit rows of 18432-26624 columns (multiples of 2048): 8 fragments a
// thread on nfrag / 8 threads (288-416), two CTAs an SM, the row staged in
// quarters: one CTA's reductions and exponent phase overlap the other's, which
// one row at a time on one CTA could not hide (0.76-0.79 -> 0.83-0.88 of the
// copy bandwidth against nfrag/4 threads of 4 fragments).  Wider rows would
// need more than 80 registers a thread at two CTAs an SM, and spilled
// (28672-30720: 0.51-0.55).
template <typename T, int TPR>
TmaRowFn wide8_row_kernel() {
  return k_bias_softmax_rows_tma<T, TPR, 8, true, 4, TPR>;
}

template <typename T>
TmaRowFn pick_wide4_row_kernel(int64_t nfrag, int* parts, int* consumers) {
  if (nfrag % 256 != 0) return nullptr;
  if (EP_SM_WIDE_2CTA) {
    *parts = 4;
    *consumers = static_cast<int>(nfrag / 8);
    switch (nfrag / 8) {
      case 288: return wide8_row_kernel<T, 288>();
      case 320: return wide8_row_kernel<T, 320>();
      case 352: return wide8_row_kernel<T, 352>();
      case 384: return wide8_row_kernel<T, 384>();
      case 416: return wide8_row_kernel<T, 416>();
      default: break;
    }
  }
  *parts = 2;
  *consumers = static_cast<int>(nfrag / 4);
  switch (nfrag / 4) {
    case 576: return wide4_row_kernel<T, 576>();
    case 640: return wide4_row_kernel<T, 640>();
    case 704: return wide4_row_kernel<T, 704>();
    case 768: return wide4_row_kernel<T, 768>();
    case 832: return wide4_row_kernel<T, 832>();
    case 896: return wide4_row_kernel<T, 896>();
    case 960: return wide4_row_kernel<T, 960>();
    default: return nullptr;
  }
}

template <typename T>
TmaRowFn pick_wide_row_kernel(int64_t nfrag, int* parts) {
  constexpr int VW = dev::Vec16<T>::N;
  if (nfrag % kWideTpr != 0) return nullptr;
  const int64_t nv = nfrag / kWideTpr;
  *parts = static_cast<int>(nv % 2 == 0 ? nv / 2 : nv);
  if constexpr (VW == 8) {
    switch (nv) {
      case 5: return wide_row_kernel<T, 5>();
      case 6: return wide_row_kernel<T, 6>();
      case 7: return wide_row_kernel<T, 7>();
      case 8: return wide_row_kernel<T, 8>();
      default: return nullptr;
    }
  } else {
    switch (nv) {
      case 9: return wide_row_kernel<T, 9>();
      case 10: return wide_row_kernel<T, 10>();
      case 11: return wide_row_kernel<T, 11>();
      case 12: return wide_row_kernel<T, 12>();
      case 13: return wide_row_kernel<T, 13>();
      case 14: return wide_row_kernel<T, 14>();
      case 15: return wide_row_kernel<T, 15>();
      case 16: return wide_row_kernel<T, 16>();
      default: return nullptr;
    }
  }
}

template <typename T>
TmaRowFn pick_tma_row_kernel(int64_t cols, int* rows_per_tile, int* parts, int* consumers) {
  *parts = 1;
  *consumers = kWsConsumers;
  constexpr int VW = dev::Vec16<T>::N;
  const int64_t nfrag = cols / VW;
  const int64_t row_bytes = cols * int64_t(sizeof(T));
  if (nfrag < 12) return nullptr;
  if (cols > kRowMax) {
    if (!EP_SM_WIDE) return nullptr;
    *rows_per_tile = 1;
    if constexpr (VW == 8) {
      if (EP_SM_WIDE_NV4)
        if (TmaRowFn f = pick_wide4_row_kernel<T>(nfrag, parts, consumers)) return f;
    }
    *consumers = kWideTpr;
    return pick_wide_row_kernel<T>(nfrag, parts);
  }
  // exact shapes; the compiled set is every (TPR, NV) this search can return
  for (int nv : {4, 5, 6, 7, 8, 3, 12, 16}) {
    const int tpr = exact_tpr(nfrag, nv);
    if (tpr == 0 || tpr < EP_SM_TMA_MIN_TPR) continue;
    *rows_per_tile = kWsConsumers / tpr;
#define EP_SM_TMA_EXACT(TPR_, NV_) \
    if (tpr == TPR_ && nv == NV_) return k_bias_softmax_rows_tma<T, TPR_, NV_, true>;
    EP_SM_TMA_EXACT(4, 4) EP_SM_TMA_EXACT(8, 4) EP_SM_TMA_EXACT(16, 4) EP_SM_TMA_EXACT(32, 4)
    EP_SM_TMA_EXACT(64, 4) EP_SM_TMA_EXACT(128, 4) EP_SM_TMA_EXACT(256, 4)
    EP_SM_TMA_EXACT(4, 5) EP_SM_TMA_EXACT(8, 5) EP_SM_TMA_EXACT(16, 5) EP_SM_TMA_EXACT(32, 5)
    EP_SM_TMA_EXACT(64, 5) EP_SM_TMA_EXACT(128, 5) EP_SM_TMA_EXACT(256, 5)
    EP_SM_TMA_EXACT(4, 6) EP_SM_TMA_EXACT(8, 6) EP_SM_TMA_EXACT(16, 6) EP_SM_TMA_EXACT(32, 6)
    EP_SM_TMA_EXACT(64, 6) EP_SM_TMA_EXACT(128, 6) EP_SM_TMA_EXACT(256, 6)
    EP_SM_TMA_EXACT(4, 7) EP_SM_TMA_EXACT(8, 7) EP_SM_TMA_EXACT(16, 7) EP_SM_TMA_EXACT(32, 7)
    EP_SM_TMA_EXACT(64, 7) EP_SM_TMA_EXACT(128, 7) EP_SM_TMA_EXACT(256, 7)
    // NV = 8 below TPR = 256 is NV = 4 at twice the TPR.  A 256x8 row is 32 KB:
    // staged in halves, so that two CTAs (three stages each) fit on an SM
    if (tpr == 256 && nv == 8) {
      *parts = 2;
      return k_bias_softmax_rows_tma<T, 256, 8, true, 2>;
    }
    if constexpr (VW == 4) {
      // float32 rows of 12288 and 16384: 48 and 64 floats a thread, staged in
      // 16 KB parts
      if (tpr == 256 && nv == 12) {
        *parts = 3;
        return k_bias_softmax_rows_tma<T, 256, 12, true, 3>;
      }
      if (tpr == 256 && nv == 16) {
        *parts = 4;
        return k_bias_softmax_rows_tma<T, 256, 16, true, 4>;
      }
    }
    EP_SM_TMA_EXACT(4, 3)     // NV = 3 above TPR = 4 is NV = 6 at half the TPR; NV = 2 is never
                              // reached (nfrag = 2 TPR is NV = 4 at TPR / 2, or under 12 fragments)
#undef EP_SM_TMA_EXACT
    return nullptr;
  }
  if (nfrag < 32) return nullptr;
  for (int tpr : {16, 32, 64, 128, 256}) {
    const int64_t nv = (nfrag + tpr - 1) / tpr;
    if (nv > 8 || tpr < EP_SM_TMA_MIN_TPR) continue;
    const int rt = kWsConsumers / tpr;
    if (rt * row_bytes > kTmaTileBytes && tpr != 256) continue;
    *rows_per_tile = rt;
#define EP_SM_TMA_RAGGED(TPR_, NV_) \
    if (tpr == TPR_ && nv <= NV_) return k_bias_softmax_rows_tma<T, TPR_, NV_, false>;
    EP_SM_TMA_RAGGED(16, 4) EP_SM_TMA_RAGGED(32, 4) EP_SM_TMA_RAGGED(64, 4) EP_SM_TMA_RAGGED(128, 4)
    EP_SM_TMA_RAGGED(256, 4) EP_SM_TMA_RAGGED(256, 8)
#undef EP_SM_TMA_RAGGED
    return nullptr;
  }
  return nullptr;
}

template <typename T>
bool launch_tma_rows(const SmKernelArgs& k, const SoftmaxArgs& a, int sm_count, cudaStream_t stream,
                     int* launches, cudaError_t* err) {
  int rt = 0;
  int parts = 1;
  int consumers = kWsConsumers;
  TmaRowFn f = pick_tma_row_kernel<T>(a.cols, &rt, &parts, &consumers);
  if (f == nullptr) return false;
  // a stage holds a tile (or one part of a row) and its bias rows
  const uint32_t row_bytes = uint32_t(a.cols * int64_t(sizeof(T))) / uint32_t(parts);
  const int64_t slots = parts > 1 ? 1
                      : a.inner ? std::min<int64_t>(rt, (rt - 1) / a.inner_repeat + 2)
                                : std::min<int64_t>(rt, a.bias_rows);
  const uint32_t stage_bytes = uint32_t(rt + slots) * row_bytes;
  if (2 * stage_bytes > 2 * kTmaStageBudget) return false;
  int stages = std::min<int>(kTmaMaxStages, std::max<int>(parts > 1 ? 3 : 2, kTmaStageBudget / stage_bytes));
  // wide-row CTAs (more than 256 consumers) run alone on their SM, or two to
  // an SM up to kWide2Max consumers: as many stages as fit in their share
  if (consumers > kWsConsumers)
    stages = std::min<int>(kTmaMaxStages, int((consumers <= kWide2Max ? 112u * 1024u : 224u * 1024u) / stage_bytes));
  const size_t smem = size_t(stages) * stage_bytes;
  const int threads = consumers + 32;
  int per_sm = 1;
  *err = resident_ctas(reinterpret_cast<const void*>(f), threads, smem, &per_sm);
  if (*err != cudaSuccess) return true;
  const int64_t ntiles = (a.rows + rt - 1) / rt;
  // one CTA per tile under launch control, else a persistent grid
  const bool clc = EP_SM_CLC && ntiles <= int64_t(INT32_MAX);
  const unsigned grid = static_cast<unsigned>(clc ? ntiles : std::min<int64_t>(ntiles, int64_t(sm_count) * per_sm));
  *err = launch(f, dim3(grid), dim3(threads), smem, stream, k, stages, int(slots), ntiles);
  if (*err == cudaSuccess) *launches += 1;
  return true;
}

template <typename T>
cudaError_t launch_t(const SoftmaxArgs& a, int sm_count, int l2_bytes, cudaStream_t stream, int* launches) {
  constexpr int VW = dev::Vec16<T>::N;
  SmKernelArgs k{a.data, a.bias, a.output, a.rows, a.cols, a.bias_rows, a.inner_repeat, a.inner};
  const bool vec = vec_ok<T>(a.data, a.bias, a.output, a.cols);
  // aligned rows of exactly 8 elements (one 16-bit fragment, or two float32
  // ones) take the register kernel's one-thread rows: 0.23 -> 0.74 (float16)
  // and 0.34 -> 0.99 (float32) of the copy bandwidth; float32 rows of 4 stay
  // here (0.69 against 0.59)
  if (a.cols <= kPackedMax && !(vec && EP_SM_SHORT_VEC && a.cols == kPackedMax)) {
    const int64_t blocks = (a.rows + 255) / 256;
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(blocks, int64_t(sm_count) * 32));
    cudaError_t el = launch(k_bias_softmax_packed<T>, dim3(grid), dim3(256), 0, stream, k);
    if (el != cudaSuccess) return el;
    *launches += 1;
    return cudaGetLastError();
  }
  if (vec && EP_SM_TMA) {
    cudaError_t e = cudaSuccess;
    if (launch_tma_rows<T>(k, a, sm_count, stream, launches, &e)) return e;
  }
  if (a.cols <= kRowMax) {
    int tpr = 0;
    RowFn fn = vec ? pick_row_kernel<T, VW>(a.cols, &tpr) : pick_row_kernel<T, 1>(a.cols, &tpr);
    const int bs = std::max(tpr, 256);
    const int rpc = bs / tpr;
    const int64_t need = (a.rows + rpc - 1) / rpc;
    const int64_t cap = int64_t(sm_count) * 64 * (2048 / bs);
    cudaError_t el = launch(fn, dim3(static_cast<unsigned>(std::min(need, cap))), dim3(bs), 0, stream, k);
    if (el != cudaSuccess) return el;
    *launches += 1;
    return cudaGetLastError();
  }
  return vec ? launch_split<T, VW>(k, a, sm_count, l2_bytes, stream, launches)
             : launch_split<T, 1>(k, a, sm_count, l2_bytes, stream, launches);
}

}  // namespace

size_t softmax_workspace_bytes(DType t, int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= kRowMax) return 0;
  const int64_t chunk = kChunkBytes / dtype_size(t);
  const int64_t nchunks = (cols + chunk - 1) / chunk;
  return static_cast<size_t>(rows * nchunks) * sizeof(float2);
}

cudaError_t launch_bias_softmax(const SoftmaxArgs& a, int sm_count, int l2_bytes, cudaStream_t stream,
                                int* launches) {
  switch (a.t) {
    case DType::F32: return launch_t<float>(a, sm_count, l2_bytes, stream, launches);
    case DType::F16: return launch_t<__half>(a, sm_count, l2_bytes, stream, launches);
    default: return launch_t<__nv_bfloat16>(a, sm_count, l2_bytes, stream, launches);
  }
}


// ---------------------------------------------------------------------------
// Fixed scratch for ep_bias_softmax_noalloc: split-row chunk statistics in a
// file-scope device array instead of a caller-provided workspace.  Every
// device that loads the library holds these kStaticScratchBytes until the
// process exits.  The array's name in host code is only a stand-in, so the
// host looks up its device address once per device (with that device current)
// and passes that address to the kernels like any workspace.
// ---------------------------------------------------------------------------

constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 131072 (max, sum) pairs
static __device__ __align__(256) unsigned char g_softmax_static_scratch[kStaticScratchBytes];

namespace {
constexpr int kScratchDevices = 64;
std::atomic<void*> g_softmax_static_scratch_addr[kScratchDevices];
}  // namespace

size_t static_softmax_scratch_bytes() { return kStaticScratchBytes; }

cudaError_t static_softmax_scratch(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kScratchDevices) {
    void* p = g_softmax_static_scratch_addr[dev].load(std::memory_order_acquire);
    if (p != nullptr) {
      *addr = p;
      return cudaSuccess;
    }
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_softmax_static_scratch);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kScratchDevices) g_softmax_static_scratch_addr[dev].store(p, std::memory_order_release);
  *addr = p;
  return cudaSuccess;
}

cudaError_t softmax_pipe_timeouts(unsigned int* count, bool clear) { return read_pipe_timeouts(count, clear); }

}  // namespace ep
