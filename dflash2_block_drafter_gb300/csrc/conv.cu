// The two-tap dynamic grouped depthwise conv around each drafter sublayer:
//   Conv_side(y)[t, c] = sum_tau (base[side, tau, c] + D[t, side, tau, c / gs]) * y[t - tau, c],
// t block-local, y[-1] = 0 (dflash2.ts header "layer" paragraph, #coefficients, #conv; MAX
// DFlash2GroupedConv). D = kernel_projection(n) comes from the tensor-core GEMM (gemm.cu) as
// fp32 split-K partials; the coefficient broadcast (base + per-group delta) is fused into the
// apply passes and never materialised at channel width.
//
// Apply passes: a thread owns one 8-channel strip of a few consecutive rows of one block: it loads
// the base kernel once, the row before its first row, and then per row the 16-byte input vector
// and the row's group deltas (all independent loads, issued before any arithmetic), and writes one
// vector per row, carrying the row as the next row's t-1 input. A CTA holds every row of a block
// for its channels, so no read crosses a block boundary. RMSNorm is a pass of a few rows per CTA.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {
namespace {

constexpr int kApplyMaxThreads = 256;  // threads per apply CTA: G rows x (256 / G) vectors
constexpr int kNormThreads = 1024;     // at most one thread per 8 channels of a row (H <= 8192)

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float (&f)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store8(float* p, const float (&f)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
__device__ __forceinline__ void store1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void store1(float* p, float v) { *p = v; }
__device__ __forceinline__ float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float load1(const float* p) { return *p; }

// 16 consecutive elements as 8 float pairs (bf16 widens exactly: its bits are the top half of
// the float's), for the packed fp32 arithmetic of the streamed passes.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ void load16(const __nv_bfloat16* p, float2 (&f)[8]) {
  const uint4 a = reinterpret_cast<const uint4*>(p)[0];
  const uint4 b = reinterpret_cast<const uint4*>(p)[1];
  f[0] = bf16x2_to_float2(a.x);
  f[1] = bf16x2_to_float2(a.y);
  f[2] = bf16x2_to_float2(a.z);
  f[3] = bf16x2_to_float2(a.w);
  f[4] = bf16x2_to_float2(b.x);
  f[5] = bf16x2_to_float2(b.y);
  f[6] = bf16x2_to_float2(b.z);
  f[7] = bf16x2_to_float2(b.w);
}
__device__ __forceinline__ void load16(const float* p, float2 (&f)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 v = reinterpret_cast<const float4*>(p)[i];
    f[2 * i] = make_float2(v.x, v.y);
    f[2 * i + 1] = make_float2(v.z, v.w);
  }
}
__device__ __forceinline__ void store16(__nv_bfloat16* p, const float2 (&f)[8]) {
  uint4 u[2];
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(u);
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = __float22bfloat162_rn(f[i]);
  reinterpret_cast<uint4*>(p)[0] = u[0];
  reinterpret_cast<uint4*>(p)[1] = u[1];
}
__device__ __forceinline__ void store16(float* p, const float2 (&f)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) reinterpret_cast<float4*>(p)[i] = make_float4(f[2 * i].x, f[2 * i].y, f[2 * i + 1].x, f[2 * i + 1].y);
}


// Rows per thread of the apply passes: a thread walks RPT consecutive rows of one 8-channel strip,
// loading the base kernel once and taking each row's t-1 input from the previous iteration.
#ifndef DFL_APPLY_RPT
#define DFL_APPLY_RPT 2
#endif
constexpr int kRpt = DFL_APPLY_RPT;

// Vectors (of 8 channels) per apply CTA for blocks of G rows, kRpt rows per thread.
__host__ __device__ inline int row_groups(int G) { return (G + kRpt - 1) / kRpt; }
__host__ __device__ inline int vectors_per_cta(int G) {
  return row_groups(G) >= kApplyMaxThreads ? 1 : kApplyMaxThreads / row_groups(G);
}

// RMSNorm of selected rows, kNormRows output rows per CTA (dflash2.ts #rms):
//   n[b, t - row0, :] = x[b, t, :] * rsqrt(mean(x[b, t, :]^2) + eps) * w   for t in [row0, G).
// Thread i owns channels 8i..8i+7 of each of the CTA's rows; the rows' vectors and the weight
// vector are loaded before the reduction (all independent), and held in registers until scaled.
#ifndef DFL_NORM_ROWS
#define DFL_NORM_ROWS 1
#endif
constexpr int kNormRows = DFL_NORM_ROWS;

// Output rows of block b: rows_out dense rows at b * rows_out, or (row_off given) the
// row_off[b + 1] - row_off[b] rows at row_off[b] of an output of m_out rows. A span that is not
// inside [0, m_out), or that holds more rows than the block, records DFLASH2_ERR_INVALID_ARG (when
// err is given) and writes nothing.
struct RowSpan {
  size_t first;
  int n;
};
__device__ __forceinline__ RowSpan out_rows(const int32_t* row_off, int b, int rows_out, int m_out, int* err) {
  if (row_off == nullptr) return RowSpan{static_cast<size_t>(b) * rows_out, rows_out};
  const int lo = row_off[b];
  const int n = row_off[b + 1] - lo;
  if (lo < 0 || n < 0 || n > rows_out || lo > m_out - n) {
    if (err != nullptr) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_INVALID_ARG));
    return RowSpan{0, 0};
  }
  return RowSpan{static_cast<size_t>(lo), n};
}

template <typename T>
__global__ void __launch_bounds__(kNormThreads)
    rms_rows_kernel(const T* __restrict__ x, const T* __restrict__ w, float eps, T* __restrict__ n, int G, int row0,
                    int H, int total_rows, const int32_t* __restrict__ row_off, int m_out, int* err) {
  __shared__ float warp_ss[kNormRows][32];
  __shared__ float row_r[kNormRows];
  pdl_trigger();
  pdl_wait();
  const int rows_out = G - row0;
  const int c = threadIdx.x * 8;
  const bool active = c < H;
  float f[kNormRows][8];
  float g[8];
  float ss[kNormRows];
  if (active) load8(w + c, g);
#pragma unroll
  for (int k = 0; k < kNormRows; ++k) {
    const int o = blockIdx.x * kNormRows + k;  // output row
    ss[k] = 0.f;
    if (active && o < total_rows) {
      const int b = o / rows_out;
      const int t = row0 + o % rows_out;
      load8(x + (static_cast<size_t>(b) * G + t) * H + c, f[k]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[k][i] = 0.f;
    }
  }
#pragma unroll
  for (int k = 0; k < kNormRows; ++k) {
#pragma unroll
    for (int i = 0; i < 8; ++i) ss[k] = fmaf(f[k][i], f[k][i], ss[k]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss[k] += __shfl_xor_sync(0xffffffffu, ss[k], o);
    if ((threadIdx.x & 31) == 0) warp_ss[k][threadIdx.x >> 5] = ss[k];
  }
  __syncthreads();
  if (threadIdx.x < 32) {
#pragma unroll
    for (int k = 0; k < kNormRows; ++k) {
      float v = threadIdx.x < (blockDim.x >> 5) ? warp_ss[k][threadIdx.x] : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (threadIdx.x == 0) row_r[k] = rsqrtf(v / static_cast<float>(H) + eps);
    }
  }
  __syncthreads();
  if (!active) return;
#pragma unroll
  for (int k = 0; k < kNormRows; ++k) {
    const int o = blockIdx.x * kNormRows + k;
    if (o >= total_rows) break;
    const int b = o / rows_out;
    const int i = o % rows_out;
    const RowSpan span = out_rows(row_off, b, rows_out, m_out, (threadIdx.x == 0 && i == 0) ? err : nullptr);
    if (i >= span.n) continue;
    const float r = row_r[k];
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = f[k][j] * r * g[j];
    store8(n + (span.first + i) * H + c, v);
  }
}

// prepare's apply pass: out = side-0 conv of n; coef1 = side 1's deltas (no base); d_full = D.
// part: [k_splits][B*G][4*groups] fp32 split-K partial sums of D, column (side*2+tap)*groups + g.
// Thread (tg, v): rows tg*RPT .. tg*RPT+RPT-1 of block blockIdx.y, channels
// 8*(blockIdx.x*vpc + v) .. +8. The thread that starts a group also writes that group's side-1
// deltas (and D when asked).
template <typename T, int RPT>
__global__ void __launch_bounds__(kApplyMaxThreads)
    conv_side0_kernel(const T* __restrict__ n, const float* __restrict__ part, int k_splits,
                      const float* __restrict__ base, T* __restrict__ out, T* __restrict__ coef1,
                      float* __restrict__ d_full, int B, int G, int H, int gs, int groups, int vpc) {
  pdl_trigger();
  pdl_wait();
  const int t0 = (threadIdx.x / vpc) * RPT;
  const int c = (blockIdx.x * vpc + threadIdx.x % vpc) * 8;
  if (t0 >= G || c >= H) return;
  const size_t row0 = static_cast<size_t>(blockIdx.y) * G + t0;
  const int g = c / gs;
  const int N = 4 * groups;
  const size_t MN = static_cast<size_t>(B) * G * N;
  const bool leader = (c % gs) == 0;
  float b0[8], b1[8], prev[8];
  load8(base + c, b0);      // base[0][0][c..]
  load8(base + H + c, b1);  // base[0][1][c..]
  if (t0 > 0) {
    load8(n + (row0 - 1) * H + c, prev);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) prev[i] = 0.f;
  }
  float cur[RPT][8];
  float d0[RPT], d1[RPT], d2[RPT], d3[RPT];
#pragma unroll
  for (int k = 0; k < RPT; ++k) {
    d0[k] = d1[k] = d2[k] = d3[k] = 0.f;
    if (t0 + k >= G) continue;
    load8(n + (row0 + k) * H + c, cur[k]);
    const float* pr = part + (row0 + k) * N + g;
    for (int s = 0; s < k_splits; ++s) {
      d0[k] += __ldg(pr + s * MN);
      d1[k] += __ldg(pr + s * MN + groups);
    }
    if (leader) {
      for (int s = 0; s < k_splits; ++s) {
        d2[k] += __ldg(pr + s * MN + 2 * groups);
        d3[k] += __ldg(pr + s * MN + 3 * groups);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < RPT; ++k) {
    if (t0 + k >= G) break;
    const size_t row = row0 + k;
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = (b0[i] + d0[k]) * cur[k][i] + (b1[i] + d1[k]) * prev[i];
    store8(out + row * H + c, o);
#pragma unroll
    for (int i = 0; i < 8; ++i) prev[i] = cur[k][i];
    if (leader) {
      store1(coef1 + (row * 2 + 0) * groups + g, d2[k]);
      store1(coef1 + (row * 2 + 1) * groups + g, d3[k]);
      if (d_full != nullptr) {
        float* df = d_full + row * N + g;
        df[0] = d0[k];
        df[groups] = d1[k];
        df[2 * groups] = d2[k];
        df[3 * groups] = d3[k];
      }
    }
  }
}

// finish's apply pass: out = residual + side-1 conv of y (fp32 add, one rounding). `out` may be
// `residual` (in place): every thread reads and then writes only its own rows and channels.
template <typename T, int RPT>
__global__ void __launch_bounds__(kApplyMaxThreads)
    conv_side1_kernel(const T* __restrict__ y, const T* __restrict__ coef1, const float* __restrict__ base,
                      const T* residual, T* out, int G, int H, int gs, int groups, int vpc) {
  pdl_trigger();
  pdl_wait();
  const int t0 = (threadIdx.x / vpc) * RPT;
  const int c = (blockIdx.x * vpc + threadIdx.x % vpc) * 8;
  if (t0 >= G || c >= H) return;
  const size_t row0 = static_cast<size_t>(blockIdx.y) * G + t0;
  const int g = c / gs;
  float b0[8], b1[8], prev[8];
  load8(base + 2 * H + c, b0);  // base[1][0][c..]
  load8(base + 3 * H + c, b1);  // base[1][1][c..]
  if (t0 > 0) {
    load8(y + (row0 - 1) * H + c, prev);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) prev[i] = 0.f;
  }
  float cur[RPT][8], res[RPT][8], d0[RPT], d1[RPT];
#pragma unroll
  for (int k = 0; k < RPT; ++k) {
    if (t0 + k >= G) continue;
    const size_t row = row0 + k;
    load8(y + row * H + c, cur[k]);
    if (residual != nullptr) {
      load8(residual + row * H + c, res[k]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) res[k][i] = 0.f;
    }
    d0[k] = load1(coef1 + (row * 2 + 0) * groups + g);
    d1[k] = load1(coef1 + (row * 2 + 1) * groups + g);
  }
#pragma unroll
  for (int k = 0; k < RPT; ++k) {
    if (t0 + k >= G) break;
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = (b0[i] + d0[k]) * cur[k][i] + (b1[i] + d1[k]) * prev[i] + res[k][i];
    store8(out + (row0 + k) * H + c, o);
#pragma unroll
    for (int i = 0; i < 8; ++i) prev[i] = cur[k][i];
  }
}

// ------------------------------------------------------------------ streamed apply passes
// Persistent CTAs over items (block b, 256-channel strip j). Warp kStreamConsumers (one lane)
// streams each item's tiles into a shared-memory ring with TMA; the consumer warps compute from
// shared memory and store 16-byte vectors. A CTA's items are all in flight as soon as it starts
// (ring depth >= items per CTA at the drafter's shape), and the bytes in flight cost no registers.
constexpr int kStreamSW = 256;        // channels per strip
#ifndef DFL_STREAM_WARPS
#define DFL_STREAM_WARPS 8
#endif
constexpr int kStreamConsumers = DFL_STREAM_WARPS;  // consumer warps (8 measured faster than 16)
constexpr int kStreamThreads = 32 * (kStreamConsumers + 1);
constexpr int kSsRows = (32 + kStreamConsumers - 1) / kStreamConsumers;  // rows per warp, G <= 32
constexpr int kStreamMaxStages = 4;

#ifndef DFL_STREAM
#define DFL_STREAM 1
#endif

__device__ __forceinline__ void stream_abort(volatile int* abort_flag, int* err) {
  *abort_flag = 1;
  if (err != nullptr) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_TIMEOUT));
}

// Producer side of the ring: waits for the last fills still in flight after an abort.
__device__ __forceinline__ void stream_drain(uint64_t* full, int stage, uint32_t phase, int issued, int n_stages) {
  const int n = min(issued, n_stages);
  for (int i = 0; i < n; ++i) {
    if (stage == 0) {
      stage = n_stages - 1;
      phase ^= 1u;
    } else {
      --stage;
    }
    mbar_wait_bounded(smem_u32(&full[stage]), phase, nullptr, 100000000ull);
  }
}

// finish's apply pass, streamed: out = residual + side-1 conv of y. Per item the ring stage holds
// y[b, :, strip] (G x 256), residual[b, :, strip] and coef1[b, :, :, strip groups] (2G x 256/gs).
template <typename T>
__global__ void __launch_bounds__(kStreamThreads, 2)
    conv_side1_stream_kernel(const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmR,
                             const __grid_constant__ CUtensorMap tmC, const float* __restrict__ base, T* out, int G,
                             int H, int gs, int n_items, int strips, int has_res, int n_stages, int stage_bytes,
                             int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int tileY = G * kStreamSW * static_cast<int>(sizeof(T));
  const int cgrp = kStreamSW / gs;  // groups per strip
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + n_stages * stage_bytes);
  uint64_t* empty = full + n_stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + n_stages);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < n_stages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kStreamConsumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmY);
    if (has_res) prefetch_tmap(&tmR);
    prefetch_tmap(&tmC);
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();  // no global memory is touched above this line
  const uint32_t tx = static_cast<uint32_t>((has_res ? 2 : 1) * tileY + 2 * G * cgrp * static_cast<int>(sizeof(T)));

  if (warp == kStreamConsumers) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_normal();
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int b = it / strips;
        const int j = it - b * strips;
        if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&full[stage]);
        mbar_arrive_expect_tx(fb, tx);
        uint8_t* st = smem + stage * stage_bytes;
        tma_load_2d(smem_u32(st), &tmY, fb, j * kStreamSW, b * G, pol);
        if (has_res) tma_load_2d(smem_u32(st + tileY), &tmR, fb, j * kStreamSW, b * G, pol);
        tma_load_2d(smem_u32(st + 2 * tileY), &tmC, fb, j * cgrp, b * G * 2, pol);
        ++issued;
        if (++stage == n_stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        stream_abort(abort_flag, err);
        stream_drain(full, stage, phase, issued, n_stages);
      }
    }
    return;
  }
  // The grid is a multiple of `strips`, so a CTA's items share one strip and each consumer thread
  // one 8-channel vector of it (lane = vector): its base-kernel values are loaded once, here.
  const int j = blockIdx.x % strips;
  const int v = lane;
  const int c = j * kStreamSW + v * 8;
  const int gl = (v * 8) / gs;
  float b0[8], b1[8];
  load8(base + 2 * H + c, b0);  // base[1][0][c..]
  load8(base + 3 * H + c, b1);  // base[1][1][c..]
  int stage = 0;
  uint32_t phase = 0;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int b = it / strips;
    if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
      if (lane == 0) stream_abort(abort_flag, err);
      break;
    }
    const uint8_t* st = smem + stage * stage_bytes;
    const T* sy = reinterpret_cast<const T*>(st);
    const T* sr = reinterpret_cast<const T*>(st + tileY);
    const T* sc = reinterpret_cast<const T*>(st + 2 * tileY);
    for (int t = warp; t < G; t += kStreamConsumers) {
      float cur[8], prev[8], res[8];
      load8(sy + t * kStreamSW + v * 8, cur);
      if (t > 0) {
        load8(sy + (t - 1) * kStreamSW + v * 8, prev);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) prev[i] = 0.f;
      }
      if (has_res) {
        load8(sr + t * kStreamSW + v * 8, res);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) res[i] = 0.f;
      }
      const float d0 = load1(sc + (t * 2 + 0) * cgrp + gl);
      const float d1 = load1(sc + (t * 2 + 1) * cgrp + gl);
      float o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = (b0[i] + d0) * cur[i] + (b1[i] + d1) * prev[i] + res[i];
      store8(out + (static_cast<size_t>(b) * G + t) * H + c, o);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
    if (++stage == n_stages) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

__host__ __device__ constexpr int round128(int b) { return (b + 127) & ~127; }

// The value a float becomes when stored as T.
template <typename T>
__device__ __forceinline__ float round_as(float v);
template <>
__device__ __forceinline__ float round_as<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float round_as<__nv_bfloat16>(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// finish fused with the next RMSNorm. A cluster of C CTAs owns block b; CTA r of the cluster owns
// the channels [r*SPC*256, (r+1)*SPC*256) of all G rows, one resident shared-memory stage per
// 256-channel strip (y, residual, coefficient, base-kernel and norm-weight tiles, all loaded by TMA
// at the start). Pass 1 writes x = residual + side-1 conv of y (rounded to T, to memory and over
// the residual tile) and each row's partial sum of squares; each row belongs to one warp, so a
// warp reduction gives the CTA's partial. The C partials of every row are exchanged through
// distributed shared memory across a cluster barrier; pass 2 writes n = x * rsqrt(mean + eps) * w
// for rows next_row0..G-1 (compact when next_row0 = 1: the head's h).
template <typename T>
__global__ void __launch_bounds__(kStreamThreads, 2)
    conv_finish_norm_kernel(const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmR,
                            const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmW, T* out, T* next_n, float eps, int G, int H,
                            int gs, int spc, int csize, int has_res, int next_row0, int stage_bytes,
                            const int32_t* __restrict__ row_off, int m_out, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int es = static_cast<int>(sizeof(T));
  const int tileY = G * kStreamSW * es;
  const int cgrp = kStreamSW / gs;
  const int offR = round128(tileY);
  const int offC = offR + round128(tileY);
  const int offB = offC + round128(2 * G * cgrp * es);
  const int offW = offB + 2 * kStreamSW * 4;
  float* ss_all = reinterpret_cast<float*>(smem + spc * stage_bytes);  // [csize][G]
  uint64_t* full = reinterpret_cast<uint64_t*>(ss_all + 8 * 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + spc);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int b = static_cast<int>(blockIdx.x) / csize;
  const int strip0 = static_cast<int>(rank) * spc;
  if (threadIdx.x == 0) {
    for (int s = 0; s < spc; ++s) mbar_init(smem_u32(&full[s]), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmY);
    if (has_res) prefetch_tmap(&tmR);
    prefetch_tmap(&tmC);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmW);
  }
  __syncthreads();
  cluster_arrive_relaxed();  // every CTA of the cluster has started once the matching wait returns
  pdl_trigger();
  pdl_wait();  // no global memory is touched above this line

  if (warp == kStreamConsumers) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_normal();
      const uint32_t tx = static_cast<uint32_t>((has_res ? 2 : 1) * tileY + 2 * G * cgrp * es + 2 * kStreamSW * 4 +
                                                kStreamSW * es);
      for (int s = 0; s < spc; ++s) {
        const uint32_t fb = smem_u32(&full[s]);
        const int x0 = (strip0 + s) * kStreamSW;
        uint8_t* st = smem + s * stage_bytes;
        mbar_arrive_expect_tx(fb, tx);
        tma_load_2d(smem_u32(st), &tmY, fb, x0, b * G, pol);
        if (has_res) tma_load_2d(smem_u32(st + offR), &tmR, fb, x0, b * G, pol);
        tma_load_2d(smem_u32(st + offC), &tmC, fb, (strip0 + s) * cgrp, b * G * 2, pol);
        tma_load_2d(smem_u32(st + offB), &tmB, fb, x0, 2, pol);  // base[1][0..1][strip]
        tma_load_2d(smem_u32(st + offW), &tmW, fb, x0, 0, pol);
      }
    }
    __syncwarp();
  } else {
    // ---- pass 1: x and the rows' partial sums of squares (lane = 8-channel vector of a strip)
    const int v = lane;
    const int gl = (v * 8) / gs;
    float ss[kSsRows] = {};  // rows warp + k * kStreamConsumers (G <= 32)
    bool ok = true;
    for (int s = 0; s < spc && ok; ++s) {
      if (!mbar_wait_bounded(smem_u32(&full[s]), 0, abort_flag, kWaitLimitNs)) {
        if (lane == 0) stream_abort(abort_flag, err);
        ok = false;
        break;
      }
      uint8_t* st = smem + s * stage_bytes;
      const T* sy = reinterpret_cast<const T*>(st);
      T* sr = reinterpret_cast<T*>(st + offR);
      const T* sc = reinterpret_cast<const T*>(st + offC);
      const float* sb = reinterpret_cast<const float*>(st + offB);
      const int c = (strip0 + s) * kStreamSW + v * 8;
      float b0[8], b1[8];
      load8(sb + v * 8, b0);              // base[1][0][c..]
      load8(sb + kStreamSW + v * 8, b1);  // base[1][1][c..]
#pragma unroll
      for (int k = 0; k < kSsRows; ++k) {
        const int t = warp + k * kStreamConsumers;
        if (t >= G) break;
        float cur[8], prev[8], res[8];
        load8(sy + t * kStreamSW + v * 8, cur);
        if (t > 0) {
          load8(sy + (t - 1) * kStreamSW + v * 8, prev);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) prev[i] = 0.f;
        }
        if (has_res) {
          load8(sr + t * kStreamSW + v * 8, res);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) res[i] = 0.f;
        }
        const float d0 = load1(sc + (t * 2 + 0) * cgrp + gl);
        const float d1 = load1(sc + (t * 2 + 1) * cgrp + gl);
        // packed fp32 pairs: x = ((base + D0) * y[t] + (base' + D1) * y[t-1]) + residual
        const float2 d0p = make_float2(d0, d0), d1p = make_float2(d1, d1);
        float o[8];
        float2 sq = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 k0 = __fadd2_rn(make_float2(b0[2 * i], b0[2 * i + 1]), d0p);
          const float2 k1 = __fadd2_rn(make_float2(b1[2 * i], b1[2 * i + 1]), d1p);
          const float2 pv = __fmul2_rn(k1, make_float2(prev[2 * i], prev[2 * i + 1]));
          const float2 x = __fadd2_rn(__ffma2_rn(k0, make_float2(cur[2 * i], cur[2 * i + 1]), pv),
                                      make_float2(res[2 * i], res[2 * i + 1]));
          const float2 xr = make_float2(round_as<T>(x.x), round_as<T>(x.y));
          o[2 * i] = xr.x;
          o[2 * i + 1] = xr.y;
          sq = __ffma2_rn(xr, xr, sq);
        }
        store8(out + (static_cast<size_t>(b) * G + t) * H + c, o);
        store8(sr + t * kStreamSW + v * 8, o);  // x as stored, for pass 2
        ss[k] += sq.x + sq.y;
      }
    }
    // the CTA's partial of each of this warp's rows, to every CTA of the cluster
    cluster_wait();
#pragma unroll
    for (int k = 0; k < kSsRows; ++k) {
      const int t = warp + k * kStreamConsumers;
      if (t >= G) break;
      float q = ss[k];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
      if (lane < csize) st_shared_cluster_f32(mapa_shared(smem_u32(&ss_all[rank * G + t]), lane), q);
    }
  }
  if (warp == kStreamConsumers) cluster_wait();
  cluster_sync_all();  // every partial has arrived in every CTA

  if (warp < kStreamConsumers && *abort_flag == 0) {
    // ---- pass 2: n = x * r * w for rows next_row0 .. G-1 (with row_off: the first
    // row_off[b + 1] - row_off[b] of them, at rows row_off[b] + ...)
    const int v = lane;
    const int rows_out = G - next_row0;
    const RowSpan span = out_rows(row_off, b, rows_out, m_out, warp == 0 && lane == 0 && rank == 0 ? err : nullptr);
    for (int t = warp; t < G; t += kStreamConsumers) {
      if (t < next_row0 || t - next_row0 >= span.n) continue;
      float tot = 0.f;
      for (int q = 0; q < csize; ++q) tot += ss_all[q * G + t];
      const float r = rsqrtf(tot / static_cast<float>(H) + eps);
      for (int s = 0; s < spc; ++s) {
        const uint8_t* st = smem + s * stage_bytes;
        const T* sr = reinterpret_cast<const T*>(st + offR);
        const T* sw = reinterpret_cast<const T*>(st + offW);
        float x8[8], w8[8], o[8];
        load8(sr + t * kStreamSW + v * 8, x8);
        load8(sw + v * 8, w8);
        const float2 r2 = make_float2(r, r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // (x * r) * w in packed pairs
          const float2 y2 = __fmul2_rn(__fmul2_rn(make_float2(x8[2 * i], x8[2 * i + 1]), r2),
                                       make_float2(w8[2 * i], w8[2 * i + 1]));
          o[2 * i] = y2.x;
          o[2 * i + 1] = y2.y;
        }
        store8(next_n + (span.first + (t - next_row0)) * H + (strip0 + s) * kStreamSW + v * 8, o);
      }
    }
  }
}

// finish (+ the next RMSNorm) for a few rows: one CTA per row, thread i owning channels
// 8i .. 8i + 7, so that a small batch spreads over as many SMs as it has rows instead of the few
// clusters of the strip-resident kernel. Same arithmetic as that kernel:
//   x = residual + (base[1][0] + D10) y[t] + (base[1][1] + D11) y[t - 1]   (rounded to T)
//   n = (x * rsqrt(mean(x^2) + eps)) * w   for rows t >= next_row0 (next_w given)
template <typename T>
__global__ void __launch_bounds__(kNormThreads)
    conv_finish_rows_kernel(const T* __restrict__ y, const T* __restrict__ coef1, const float* __restrict__ base,
                            const T* __restrict__ residual, T* __restrict__ out, const T* __restrict__ next_w,
                            float eps, T* __restrict__ next_n, int G, int H, int gs, int groups, int next_row0,
                            const int32_t* __restrict__ row_off, int m_out, int* err) {
  __shared__ float warp_ss[32];
  __shared__ float row_r;
  pdl_trigger();
  pdl_wait();
  const int o = blockIdx.x;  // row b * G + t
  const int b = o / G;
  const int t = o - b * G;
  const int c = threadIdx.x * 8;
  const bool active = c < H;
  float xr[8];
  float ss = 0.f;
  if (active) {
    float cur[8], prev[8], res[8], b0[8], b1[8];
    load8(y + static_cast<size_t>(o) * H + c, cur);
    if (t > 0) {
      load8(y + static_cast<size_t>(o - 1) * H + c, prev);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) prev[i] = 0.f;
    }
    if (residual != nullptr) {
      load8(residual + static_cast<size_t>(o) * H + c, res);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) res[i] = 0.f;
    }
    load8(base + 2 * static_cast<size_t>(H) + c, b0);  // base[1][0]
    load8(base + 3 * static_cast<size_t>(H) + c, b1);  // base[1][1]
    const int g = c / gs;
    const float d0 = load1(coef1 + (static_cast<size_t>(o) * 2 + 0) * groups + g);
    const float d1 = load1(coef1 + (static_cast<size_t>(o) * 2 + 1) * groups + g);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float x = fmaf(b0[i] + d0, cur[i], (b1[i] + d1) * prev[i]) + res[i];
      xr[i] = round_as<T>(x);
      ss = fmaf(xr[i], xr[i], ss);
    }
    store8(out + static_cast<size_t>(o) * H + c, xr);
  }
  if (next_n == nullptr) return;
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
  if ((threadIdx.x & 31) == 0) warp_ss[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? warp_ss[threadIdx.x] : 0.f;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) v += __shfl_xor_sync(0xffffffffu, v, s);
    if (threadIdx.x == 0) row_r = rsqrtf(v / static_cast<float>(H) + eps);
  }
  __syncthreads();
  if (!active || t < next_row0) return;
  const int rows_out = G - next_row0;
  const int i = t - next_row0;
  const RowSpan span = out_rows(row_off, b, rows_out, m_out, (threadIdx.x == 0 && i == 0) ? err : nullptr);
  if (i >= span.n) return;
  const float r = row_r;
  float w8[8], v[8];
  load8(next_w + c, w8);
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = (xr[j] * r) * w8[j];
  store8(next_n + (span.first + i) * H + c, v);
}

// D of one row and group (and of the next group when `two`) summed over KS split-K partial tiles
// in split order; pa points at split 0's (side, tap) 0 tile, pstride floats apart.
template <int KS>
__device__ __forceinline__ void sum_splits(const float* pa, int pstride, bool two, float (&da)[4], float (&db)[4]) {
  float va[KS][4], vb[KS][4];
#pragma unroll
  for (int s = 0; s < KS; ++s)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      va[s][q] = pa[(s * 4 + q) * pstride];
      vb[s][q] = two ? pa[(s * 4 + q) * pstride + 1] : 0.f;
    }
#pragma unroll
  for (int s = 0; s < KS; ++s)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      da[q] += va[s][q];
      db[q] += vb[s][q];
    }
}

// prepare's apply pass, streamed: out = side-0 conv of n, coef1 = side 1's deltas, d_full = D.
// Per item (block b, strip j) the ring stage holds n[b, :, strip] (G x 256) and, for every K split
// s and (side, tap) st, the G x (256/gs) tile of the fp32 partial sums of D for the strip's groups.
// The grid is a multiple of `strips`, so each CTA keeps one strip and its base kernel in registers.
template <typename T>
__global__ void __launch_bounds__(kStreamThreads, 2)
    conv_side0_stream_kernel(const __grid_constant__ CUtensorMap tmN, const __grid_constant__ CUtensorMap tmP,
                             const float* __restrict__ base, T* out, T* coef1, float* d_full, int G, int H, int gs,
                             int groups, int k_splits, int M, int n_items, int strips, int n_stages, int stage_bytes,
                             int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int es = static_cast<int>(sizeof(T));
  const int cgrp = kStreamSW / gs;
  const int tileN = round128(G * kStreamSW * es);
  const int tileP = round128(G * cgrp * 4);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + n_stages * stage_bytes);
  uint64_t* empty = full + n_stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + n_stages);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < n_stages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kStreamConsumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmN);
    prefetch_tmap(&tmP);
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();  // no global memory is touched above this line
  const uint32_t tx = static_cast<uint32_t>(G * kStreamSW * es + 4 * k_splits * G * cgrp * 4);

  if (warp == kStreamConsumers) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_normal();
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int b = it / strips;
        const int j = it - b * strips;
        if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&full[stage]);
        mbar_arrive_expect_tx(fb, tx);
        uint8_t* st = smem + stage * stage_bytes;
        tma_load_2d(smem_u32(st), &tmN, fb, j * kStreamSW, b * G, pol);
        for (int s = 0; s < k_splits; ++s)
          for (int q = 0; q < 4; ++q)
            tma_load_2d(smem_u32(st + tileN + (s * 4 + q) * tileP), &tmP, fb, q * groups + j * cgrp, s * M + b * G,
                        pol);
        ++issued;
        if (++stage == n_stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        stream_abort(abort_flag, err);
        stream_drain(full, stage, phase, issued, n_stages);
      }
    }
    return;
  }
  // Half-warp h of consumer warp w takes rows 2w + h (+ 16 k); lane l of the half owns the 16
  // channels [16 l, 16 l + 16) of the strip: one group (or two, at group size 8), whose summed
  // partials serve all 16 channels. Arithmetic in packed fp32 pairs, in the order
  // (base[0][0] + D0) * n[t] + ((base[0][1] + D1) * n[t-1]).
  const int j = blockIdx.x % strips;
  const int h = lane >> 4;
  const int cl = (lane & 15) * 16;    // first channel within the strip
  const int c = j * kStreamSW + cl;
  const int gla = cl / gs;            // strip-local group of channels cl .. cl+7
  const int glb = (cl + 8) / gs;      // and of cl+8 .. cl+15
  const bool lead_a = (cl % gs) == 0;
  const bool lead_b = glb != gla;     // group size 8: the second vector starts its own group
  const int N = 4 * groups;
  float2 b0[8], b1[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 x = reinterpret_cast<const float4*>(base + c)[i];      // base[0][0][c..]
    const float4 y = reinterpret_cast<const float4*>(base + H + c)[i];  // base[0][1][c..]
    b0[2 * i] = make_float2(x.x, x.y);
    b0[2 * i + 1] = make_float2(x.z, x.w);
    b1[2 * i] = make_float2(y.x, y.y);
    b1[2 * i + 1] = make_float2(y.z, y.w);
  }
  int stage = 0;
  uint32_t phase = 0;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int b = it / strips;
    if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
      if (lane == 0) stream_abort(abort_flag, err);
      break;
    }
    const uint8_t* st = smem + stage * stage_bytes;
    const T* sn = reinterpret_cast<const T*>(st);
    const float* sp = reinterpret_cast<const float*>(st + tileN);
    const int pstride = tileP / 4;  // floats between consecutive (split, side-tap) tiles
    for (int t = 2 * warp + h; t < G; t += 2 * kStreamConsumers) {
      float da[4] = {0.f, 0.f, 0.f, 0.f}, db[4] = {0.f, 0.f, 0.f, 0.f};
      const float* pa = sp + t * cgrp + gla;
      switch (k_splits) {  // the common split counts unrolled: every load issued before the sums
        case 1: sum_splits<1>(pa, pstride, lead_b, da, db); break;
        case 2: sum_splits<2>(pa, pstride, lead_b, da, db); break;
        case 3: sum_splits<3>(pa, pstride, lead_b, da, db); break;
        default:
          for (int s = 0; s < k_splits; ++s, pa += 4 * pstride) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              da[q] += pa[q * pstride];
              if (lead_b) db[q] += pa[q * pstride + 1];
            }
          }
      }
      if (!lead_b) {
#pragma unroll
        for (int q = 0; q < 4; ++q) db[q] = da[q];
      }
      float2 cur[8], prev[8];
      load16(sn + t * kStreamSW + cl, cur);
      if (t > 0) {
        load16(sn + (t - 1) * kStreamSW + cl, prev);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) prev[i] = make_float2(0.f, 0.f);
      }
      const float2 d0a = make_float2(da[0], da[0]), d1a = make_float2(da[1], da[1]);
      const float2 d0b = make_float2(db[0], db[0]), d1b = make_float2(db[1], db[1]);
      float2 o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 k0 = __fadd2_rn(b0[i], i < 4 ? d0a : d0b);
        const float2 k1 = __fadd2_rn(b1[i], i < 4 ? d1a : d1b);
        o[i] = __ffma2_rn(k0, cur[i], __fmul2_rn(k1, prev[i]));
      }
      const size_t row = static_cast<size_t>(b) * G + t;
      store16(out + row * H + c, o);
      if (lead_a) {
        const int g = j * cgrp + gla;
        store1(coef1 + (row * 2 + 0) * groups + g, da[2]);
        store1(coef1 + (row * 2 + 1) * groups + g, da[3]);
        if (d_full != nullptr) {
          float* df = d_full + row * N + g;
          df[0] = da[0];
          df[groups] = da[1];
          df[2 * groups] = da[2];
          df[3 * groups] = da[3];
        }
      }
      if (lead_b) {
        const int g = j * cgrp + glb;
        store1(coef1 + (row * 2 + 0) * groups + g, db[2]);
        store1(coef1 + (row * 2 + 1) * groups + g, db[3]);
        if (d_full != nullptr) {
          float* df = d_full + row * N + g;
          df[0] = db[0];
          df[groups] = db[1];
          df[2 * groups] = db[2];
          df[3 * groups] = db[3];
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
    if (++stage == n_stages) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

}  // namespace

// Split-K plan of kernel_projection, picked by a small cost model over the M tiles per CTA (1 or
// 2 x 128 rows), the N tile (64, 128 or 256 columns) and the number of K splits:
//   issue:   k-blocks per CTA x MMAs per k-block x ~145 cycles (a tcgen05.mma of any N up to 256
//            takes about that long, so wide tiles do more work per instruction)
//   ingest:  bytes each CTA pulls through TMA at ~100 GB/s per SM (measured: with a ~200 KB stage
//            ring the bytes in flight, not L2 bandwidth, cap what one SM can pull)
//   stream:  weight bytes / (CTAs x ~40 GB/s per SM)   (small M: spread the weight over the SMs)
//   output:  each CTA's fp32 tile leaves at ~16 GB/s per SM (measured), and with K splits the
//            partials are read back by the side-0 pass (~5 TB/s)
// cost = max(issue, ingest, stream) + output.
// CTA-pair plans (above 128 rows): 256-row pair tiles, each SM ingesting its 128 rows and half of
// the tile's weight rows, partials leaving by TMA store (~50 GB/s per SM assumed).
#ifndef DFL_KP_PAIR
#define DFL_KP_PAIR 1
#endif
GemmPlan kp_plan(const ConvShape& s, int sms) {
  const int M = s.rows();
  const int N = 4 * s.groups;
  const int bk = 64;  // elements of K per pipeline stage at most (fewer with 64-byte rows)
  const int k_blocks = (s.H + bk - 1) / bk;
  const double w_bytes = 2.0 * N * s.H;
  GemmPlan best{};
  double best_cost = 1e30;
  for (int mt = 1; mt <= (M > 128 ? 2 : 1); ++mt) {
    for (int tile_chunks = 4; tile_chunks >= 1; tile_chunks /= 2) {
      GemmPlan p{};
      p.mt = mt;
      p.m_groups = (M + 128 * mt - 1) / (128 * mt);
      p.n_chunks = (N + 63) / 64;
      p.n_splits = (p.n_chunks + tile_chunks - 1) / tile_chunks;
      const int units = p.m_groups * p.n_splits;
      p.k_splits = std::max(1, std::min(std::min(k_blocks, 32), sms / std::max(1, units)));
      const int ctas = units * p.k_splits;
      const int waves = (ctas + sms - 1) / sms;
      const double kb_per_cta = static_cast<double>(k_blocks) / p.k_splits;
      const double cols = 64.0 * tile_chunks;
      const double rows = std::min(M, 128 * mt);
      const double t_issue = waves * kb_per_cta * 4.0 * mt * 145.0 / 1.9e9;
      const double t_ingest = waves * kb_per_cta * (mt * 16384.0 + tile_chunks * 8192.0) / 100e9;
      const double t_stream = w_bytes / (std::min(ctas, sms) * 40e9);
      const double t_out = waves * rows * cols * 4.0 / 16e9 +
                           (p.k_splits > 1 ? p.k_splits * static_cast<double>(M) * N * 8.0 / 5e12 : 0.0);
      const double cost = std::max(std::max(t_issue, t_ingest), t_stream) + t_out;
      if (cost < best_cost) {
        best_cost = cost;
        best = p;
      }
    }
  }
  const int pairs = (DFL_KP_PAIR && M > 128 && N % 4 == 0) ? std::min(gemm_pair_capacity(), sms / 2) : 0;
  for (int tile_units = 2; pairs > 0 && tile_units >= 1; --tile_units) {
    GemmPlan p{};
    p.pair = 1;
    p.mt = 2;
    p.m_groups = (M + 255) / 256;
    p.n_chunks = (N + 127) / 128;  // 128-column units
    p.n_splits = (p.n_chunks + tile_units - 1) / tile_units;
    const int tiles = p.m_groups * p.n_splits;
    p.k_splits = std::max(1, std::min(std::min(k_blocks, 32), pairs / std::max(1, tiles)));
    const int used = tiles * p.k_splits;
    const int waves = (used + pairs - 1) / pairs;
    const int units_per_pair = (p.n_chunks + p.n_splits - 1) / p.n_splits;
    const int tiles_per_pair = (units_per_pair + 1) / 2;
    const double kb_per_cta = static_cast<double>(k_blocks) / p.k_splits * tiles_per_pair;
    const double t_issue = waves * kb_per_cta * 4.0 * 145.0 / 1.9e9;
    const double t_ingest = waves * kb_per_cta * (16384.0 + std::min(units_per_pair, 2) * 8192.0) / 100e9;
    const double t_stream = w_bytes / (std::min(2 * used, sms) * 40e9);
    const double t_out = waves * 128.0 * 128.0 * units_per_pair * 4.0 / 50e9 +
                         (p.k_splits > 1 ? p.k_splits * static_cast<double>(M) * N * 8.0 / 5e12 : 0.0);
    const double cost = std::max(std::max(t_issue, t_ingest), t_stream) + t_out;
    if (cost < best_cost) {
      best_cost = cost;
      best = p;
    }
  }
  return best;
}

size_t conv_prepare_workspace(const ConvShape& s, int sms) {
  const GemmPlan p = kp_plan(s, sms);
  const size_t es = s.dtype == DFLASH2_F32 ? 4 : 2;
  size_t n_bytes = static_cast<size_t>(s.rows()) * s.H * es;
  n_bytes = (n_bytes + 255) & ~static_cast<size_t>(255);
  const size_t part = static_cast<size_t>(p.k_splits) * s.rows() * 4 * s.groups * sizeof(float);
  return n_bytes + part + 256;
}

template <typename T>
static int rms_rows_typed(const void* x, const void* w, float eps, void* n, int B, int G, int row0, int H,
                          cudaStream_t st, const int32_t* row_off, int m_out) {
  const int threads = std::min(kNormThreads, ((H / 8 + 31) / 32) * 32);
  const int total = B * (G - row0);
  const cudaError_t e = launch_pdl(rms_rows_kernel<T>, dim3((total + kNormRows - 1) / kNormRows), dim3(threads), 0,
                                   st, nullptr, 0, static_cast<const T*>(x), static_cast<const T*>(w), eps,
                                   static_cast<T*>(n), G, row0, H, total, row_off, m_out, device_error_word());
  return e == cudaSuccess ? DFLASH2_OK : fail(DFLASH2_ERR_CUDA, "rmsnorm launch failed: %s", cudaGetErrorString(e));
}

int launch_rmsnorm_rows(const void* x, const void* w, float eps, void* n, int B, int G, int row0, int H, int dtype,
                        cudaStream_t st, const int32_t* row_off, int m_out) {
  if (dtype == DFLASH2_F32) return rms_rows_typed<float>(x, w, eps, n, B, G, row0, H, st, row_off, m_out);
  return rms_rows_typed<__nv_bfloat16>(x, w, eps, n, B, G, row0, H, st, row_off, m_out);
}

int launch_rmsnorm(const void* x, const void* w, float eps, void* n, int rows, int H, int dtype, cudaStream_t st) {
  return launch_rmsnorm_rows(x, w, eps, n, rows, 1, 0, H, dtype, st, nullptr, 0);
}

#ifndef DFL_STREAM0
#define DFL_STREAM0 1
#endif

static int side0_stage_bytes(const ConvShape& s, int k_splits) {
  const int es = s.dtype == DFLASH2_F32 ? 4 : 2;
  const int b = round128(s.G * kStreamSW * es) + 4 * k_splits * round128(s.G * (kStreamSW / s.gs) * 4);
  return (b + 1023) & ~1023;
}

// The streamed side-0 pass needs whole 256-channel strips, partial-sum tiles TMA can address
// (16-byte rows: 256/gs groups a multiple of 4, groups a multiple of 4) and a two-stage ring.
static bool side0_streamable(const ConvShape& s, int k_splits) {
  if (!(DFL_STREAM && DFL_STREAM0 && s.H % kStreamSW == 0 && kStreamSW % s.gs == 0 && (kStreamSW / s.gs) % 4 == 0 &&
        s.groups % 4 == 0 && s.G <= 256))
    return false;
  return 1024 + 2 * side0_stage_bytes(s, k_splits) + 128 <= 232448;
}

template <typename T>
static int launch_side0_stream(const ConvShape& s, const void* n, const float* part, int k_splits, const float* base,
                               void* out, void* coef1, float* d_full, cudaStream_t st) {
  const int es = static_cast<int>(sizeof(T));
  const uint64_t rows = static_cast<uint64_t>(s.B) * s.G;
  const int N = 4 * s.groups;
  CUtensorMap mN, mP;
  const uint64_t dn[2] = {static_cast<uint64_t>(s.H), rows};
  const uint64_t sn[1] = {static_cast<uint64_t>(s.H) * es};
  const uint32_t bn[2] = {static_cast<uint32_t>(kStreamSW), static_cast<uint32_t>(s.G)};
  const uint64_t dp[2] = {static_cast<uint64_t>(N), rows * k_splits};
  const uint64_t sp[1] = {static_cast<uint64_t>(N) * 4};
  const uint32_t bp[2] = {static_cast<uint32_t>(kStreamSW / s.gs), static_cast<uint32_t>(s.G)};
  if (!make_tmap_plain(&mN, n, s.dtype, 2, dn, sn, bn) || !make_tmap_plain(&mP, part, DFLASH2_F32, 2, dp, sp, bp))
    return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (side-0 stream)");
  const int stage_bytes = side0_stage_bytes(s, k_splits);
  const int n_stages = std::max(2, std::min(kStreamMaxStages, (160 * 1024) / stage_bytes));
  const int smem = 1024 + n_stages * stage_bytes + 128;
  const int per_sm = std::max(1, std::min(3, 232448 / smem));
  const int strips = s.H / kStreamSW;
  const int n_items = s.B * strips;
  const int grid = std::min(n_items, std::max(1, sm_count() * per_sm / strips) * strips);
  static unsigned done = 0;
  if (!ensure_smem_attr(conv_side0_stream_kernel<T>, 232448, &done))
    return fail(DFLASH2_ERR_CUDA, "cudaFuncSetAttribute failed (side-0 stream)");
  const cudaError_t e = launch_pdl(conv_side0_stream_kernel<T>, dim3(grid), dim3(kStreamThreads), smem, st, nullptr, 0,
                                   mN, mP, base, static_cast<T*>(out), static_cast<T*>(coef1), d_full, s.G, s.H, s.gs,
                                   s.groups, k_splits, static_cast<int>(rows), n_items, strips, n_stages, stage_bytes,
                                   device_error_word());
  return e == cudaSuccess ? DFLASH2_OK : fail(DFLASH2_ERR_CUDA, "side-0 stream launch failed: %s", cudaGetErrorString(e));
}

int launch_conv_side0(const ConvShape& s, const void* n, const float* part, int k_splits, const float* base,
                      void* out, void* coef1, float* d_full, cudaStream_t st) {
  if (side0_streamable(s, k_splits))
    return s.dtype == DFLASH2_F32
               ? launch_side0_stream<float>(s, n, part, k_splits, base, out, coef1, d_full, st)
               : launch_side0_stream<__nv_bfloat16>(s, n, part, k_splits, base, out, coef1, d_full, st);
  const int vpc = vectors_per_cta(s.G);
  const dim3 grid((s.H / 8 + vpc - 1) / vpc, s.B);
  const dim3 threads(row_groups(s.G) * vpc);
  cudaError_t e;
  if (s.dtype == DFLASH2_F32)
    e = launch_pdl(conv_side0_kernel<float, kRpt>, grid, threads, 0, st, nullptr, 0, static_cast<const float*>(n), part,
                   k_splits, base, static_cast<float*>(out), static_cast<float*>(coef1), d_full, s.B, s.G, s.H, s.gs,
                   s.groups, vpc);
  else
    e = launch_pdl(conv_side0_kernel<__nv_bfloat16, kRpt>, grid, threads, 0, st, nullptr, 0,
                   static_cast<const __nv_bfloat16*>(n), part, k_splits, base, static_cast<__nv_bfloat16*>(out),
                   static_cast<__nv_bfloat16*>(coef1), d_full, s.B, s.G, s.H, s.gs, s.groups, vpc);
  return e == cudaSuccess ? DFLASH2_OK : fail(DFLASH2_ERR_CUDA, "conv side0 launch failed: %s", cudaGetErrorString(e));
}

// The streamed side-1 pass needs tiles TMA can express: whole 256-channel strips, 16-byte rows of
// the coefficient tile and of coef1 itself, and at most 128 rows per block.
static bool side1_streamable(const ConvShape& s) {
  const int es = s.dtype == DFLASH2_F32 ? 4 : 2;
  if (!(DFL_STREAM && s.H % kStreamSW == 0 && kStreamSW % s.gs == 0 && ((kStreamSW / s.gs) * es) % 16 == 0 &&
        (s.groups * es) % 16 == 0 && 2 * s.G <= 256))
    return false;
  const int stage_bytes = ((2 * s.G * kStreamSW * es + 2 * s.G * (kStreamSW / s.gs) * es) + 1023) & ~1023;
  return 1024 + 2 * stage_bytes + 128 <= 232448;  // a two-stage ring fits
}

template <typename T>
static int launch_side1_stream(const ConvShape& s, const void* y, const void* coef1, const float* base,
                               const void* residual, void* out, cudaStream_t st) {
  const int dt = s.dtype;
  const int es = static_cast<int>(sizeof(T));
  const uint64_t rows = static_cast<uint64_t>(s.B) * s.G;
  CUtensorMap mY, mR, mC;
  const uint64_t dy[2] = {static_cast<uint64_t>(s.H), rows};
  const uint64_t sy[1] = {static_cast<uint64_t>(s.H) * es};
  const uint32_t by[2] = {static_cast<uint32_t>(kStreamSW), static_cast<uint32_t>(s.G)};
  const uint64_t dc[2] = {static_cast<uint64_t>(s.groups), rows * 2};
  const uint64_t sc[1] = {static_cast<uint64_t>(s.groups) * es};
  const uint32_t bc[2] = {static_cast<uint32_t>(kStreamSW / s.gs), static_cast<uint32_t>(2 * s.G)};
  if (!make_tmap_plain(&mY, y, dt, 2, dy, sy, by) || !make_tmap_plain(&mC, coef1, dt, 2, dc, sc, bc) ||
      (residual != nullptr && !make_tmap_plain(&mR, residual, dt, 2, dy, sy, by)))
    return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (side-1 stream)");
  if (residual == nullptr) mR = mY;
  const int tileY = s.G * kStreamSW * es;
  const int stage_bytes = ((2 * tileY + 2 * s.G * (kStreamSW / s.gs) * es) + 1023) & ~1023;
  const int n_stages = std::max(2, std::min(kStreamMaxStages, (200 * 1024) / stage_bytes));
  const int smem = 1024 + n_stages * stage_bytes + 128;
  const int per_sm = std::max(1, std::min(3, 232448 / smem));
  const int strips = s.H / kStreamSW;
  const int n_items = s.B * strips;
  // a multiple of `strips` (each CTA keeps one strip), at most one wave
  const int grid = std::min(n_items, std::max(1, sm_count() * per_sm / strips) * strips);
  static unsigned done = 0;
  if (!ensure_smem_attr(conv_side1_stream_kernel<T>, 232448, &done))  // once, for every shape's ring
    return fail(DFLASH2_ERR_CUDA, "cudaFuncSetAttribute failed (side-1 stream)");
  const cudaError_t e = launch_pdl(conv_side1_stream_kernel<T>, dim3(grid), dim3(kStreamThreads), smem, st, nullptr, 0,
                                   mY, mR, mC, base, static_cast<T*>(out), s.G, s.H, s.gs, n_items, strips,
                                   residual != nullptr ? 1 : 0, n_stages, stage_bytes, device_error_word());
  return e == cudaSuccess ? DFLASH2_OK : fail(DFLASH2_ERR_CUDA, "side-1 stream launch failed: %s", cudaGetErrorString(e));
}

// finish + next RMSNorm in one kernel: a cluster of csize CTAs per block, spc resident strips per
// CTA. Returns the cluster size (0: not eligible). Prefers the largest cluster that keeps the grid
// in one wave with two CTAs per SM.
static int finish_norm_stage_bytes(const ConvShape& s) {  // matches the kernel's tile offsets
  const int es = s.dtype == DFLASH2_F32 ? 4 : 2;
  const int b = 2 * round128(s.G * kStreamSW * es) + round128(2 * s.G * (kStreamSW / s.gs) * es) + 2 * kStreamSW * 4 +
                kStreamSW * es;
  return (b + 1023) & ~1023;
}
static size_t finish_norm_smem(const ConvShape& s, int spc) {
  return 1024 + static_cast<size_t>(spc) * finish_norm_stage_bytes(s) + 8 * 64 * 4 + 8 * spc + 64;
}
static int finish_norm_cluster(const ConvShape& s) {
  if (!side1_streamable(s) || s.G > 32) return 0;
  const int strips = s.H / kStreamSW;
  int any = 0;
  for (int c = 8; c >= 1; --c) {
    if (strips % c != 0) continue;
    const size_t sm = finish_norm_smem(s, strips / c);
    if (sm > 232448) continue;
    const int per_sm = static_cast<int>(std::min<size_t>(2, 232448 / sm));
    if (s.B * c <= sm_count() * per_sm) return c;
    if (any == 0) any = c;
  }
  return any;
}

template <typename T>
static int launch_finish_norm(const ConvShape& s, int csize, const void* y, const void* coef1, const float* base,
                              const void* residual, void* out, const void* next_w, float eps, void* next_n,
                              int next_row0, cudaStream_t st, const int32_t* row_off, int m_out) {
  const int dt = s.dtype;
  const int es = static_cast<int>(sizeof(T));
  const uint64_t rows = static_cast<uint64_t>(s.B) * s.G;
  CUtensorMap mY, mR, mC, mB, mW;
  const uint64_t dy[2] = {static_cast<uint64_t>(s.H), rows};
  const uint64_t sy[1] = {static_cast<uint64_t>(s.H) * es};
  const uint32_t by[2] = {static_cast<uint32_t>(kStreamSW), static_cast<uint32_t>(s.G)};
  const uint64_t dc[2] = {static_cast<uint64_t>(s.groups), rows * 2};
  const uint64_t sc[1] = {static_cast<uint64_t>(s.groups) * es};
  const uint32_t bc[2] = {static_cast<uint32_t>(kStreamSW / s.gs), static_cast<uint32_t>(2 * s.G)};
  const uint64_t db[2] = {static_cast<uint64_t>(s.H), 4};
  const uint64_t sb[1] = {static_cast<uint64_t>(s.H) * 4};
  const uint32_t bb[2] = {static_cast<uint32_t>(kStreamSW), 2};
  const uint64_t dw[2] = {static_cast<uint64_t>(s.H), 1};
  const uint64_t sw[1] = {static_cast<uint64_t>(s.H) * es};
  const uint32_t bw[2] = {static_cast<uint32_t>(kStreamSW), 1};
  if (!make_tmap_plain(&mY, y, dt, 2, dy, sy, by) || !make_tmap_plain(&mC, coef1, dt, 2, dc, sc, bc) ||
      !make_tmap_plain(&mB, base, DFLASH2_F32, 2, db, sb, bb) || !make_tmap_plain(&mW, next_w, dt, 2, dw, sw, bw) ||
      (residual != nullptr && !make_tmap_plain(&mR, residual, dt, 2, dy, sy, by)))
    return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (finish + norm)");
  if (residual == nullptr) mR = mY;
  const int spc = (s.H / kStreamSW) / csize;
  const int smem = static_cast<int>(finish_norm_smem(s, spc));
  static unsigned done = 0;
  if (!ensure_smem_attr(conv_finish_norm_kernel<T>, 232448, &done))
    return fail(DFLASH2_ERR_CUDA, "cudaFuncSetAttribute failed (finish + norm)");
  cudaLaunchAttribute cl[1];
  cl[0].id = cudaLaunchAttributeClusterDimension;
  cl[0].val.clusterDim.x = static_cast<unsigned>(csize);
  cl[0].val.clusterDim.y = 1;
  cl[0].val.clusterDim.z = 1;
  const cudaError_t e = launch_pdl(conv_finish_norm_kernel<T>, dim3(s.B * csize), dim3(kStreamThreads), smem, st, cl, 1,
                                   mY, mR, mC, mB, mW, static_cast<T*>(out), static_cast<T*>(next_n), eps, s.G, s.H,
                                   s.gs, spc, csize, residual != nullptr ? 1 : 0, next_row0,
                                   finish_norm_stage_bytes(s), row_off, m_out, device_error_word());
  return e == cudaSuccess ? DFLASH2_OK
                          : fail(DFLASH2_ERR_CUDA, "finish + norm launch failed: %s", cudaGetErrorString(e));
}

#ifndef DFL_FINISH_NORM
#define DFL_FINISH_NORM 1
#endif

// The row-per-CTA finish takes batches of at most this many rows (a CTA per row, all resident at once).
#ifndef DFL_FINISH_ROWS_MAX
#define DFL_FINISH_ROWS_MAX 256
#endif
static bool finish_rows_eligible(const ConvShape& s) {
  return s.rows() <= DFL_FINISH_ROWS_MAX && s.H % 8 == 0 && s.H / 8 <= kNormThreads && s.gs % 8 == 0;
}

template <typename T>
static int launch_finish_rows(const ConvShape& s, const void* y, const void* coef1, const float* base,
                              const void* residual, void* out, const void* next_w, float eps, void* next_n,
                              int next_row0, cudaStream_t st, const int32_t* row_off, int m_out) {
  const int threads = ((s.H / 8 + 31) / 32) * 32;
  const cudaError_t e = launch_pdl(conv_finish_rows_kernel<T>, dim3(s.rows()), dim3(threads), 0, st, nullptr, 0,
                                   static_cast<const T*>(y), static_cast<const T*>(coef1), base,
                                   static_cast<const T*>(residual), static_cast<T*>(out),
                                   static_cast<const T*>(next_w), eps, static_cast<T*>(next_n), s.G, s.H, s.gs,
                                   s.groups, next_row0, row_off, m_out, device_error_word());
  return e == cudaSuccess ? DFLASH2_OK : fail(DFLASH2_ERR_CUDA, "finish rows launch failed: %s", cudaGetErrorString(e));
}

int launch_conv_side1(const ConvShape& s, const void* y, const void* coef1, const float* base, const void* residual,
                      void* out, const void* next_w, float eps, void* next_n, int next_row0, cudaStream_t st,
                      const int32_t* row_off, int m_out) {
  if (finish_rows_eligible(s))
    return s.dtype == DFLASH2_F32
               ? launch_finish_rows<float>(s, y, coef1, base, residual, out, next_w, eps, next_n, next_row0, st,
                                           row_off, m_out)
               : launch_finish_rows<__nv_bfloat16>(s, y, coef1, base, residual, out, next_w, eps, next_n, next_row0,
                                                   st, row_off, m_out);
  const int csize = (DFL_FINISH_NORM && next_n != nullptr) ? finish_norm_cluster(s) : 0;
  if (csize > 0)
    return s.dtype == DFLASH2_F32
               ? launch_finish_norm<float>(s, csize, y, coef1, base, residual, out, next_w, eps, next_n, next_row0, st,
                                           row_off, m_out)
               : launch_finish_norm<__nv_bfloat16>(s, csize, y, coef1, base, residual, out, next_w, eps, next_n,
                                                   next_row0, st, row_off, m_out);
  if (side1_streamable(s)) {
    const int rc = s.dtype == DFLASH2_F32 ? launch_side1_stream<float>(s, y, coef1, base, residual, out, st)
                                          : launch_side1_stream<__nv_bfloat16>(s, y, coef1, base, residual, out, st);
    if (rc != DFLASH2_OK) return rc;
    if (next_n == nullptr) return DFLASH2_OK;
    return launch_rmsnorm_rows(out, next_w, eps, next_n, s.B, s.G, next_row0, s.H, s.dtype, st, row_off, m_out);
  }
  const int vpc = vectors_per_cta(s.G);
  const dim3 grid((s.H / 8 + vpc - 1) / vpc, s.B);
  const dim3 threads(row_groups(s.G) * vpc);
  cudaError_t e;
  if (s.dtype == DFLASH2_F32)
    e = launch_pdl(conv_side1_kernel<float, kRpt>, grid, threads, 0, st, nullptr, 0, static_cast<const float*>(y),
                   static_cast<const float*>(coef1), base, static_cast<const float*>(residual),
                   static_cast<float*>(out), s.G, s.H, s.gs, s.groups, vpc);
  else
    e = launch_pdl(conv_side1_kernel<__nv_bfloat16, kRpt>, grid, threads, 0, st, nullptr, 0,
                   static_cast<const __nv_bfloat16*>(y), static_cast<const __nv_bfloat16*>(coef1), base,
                   static_cast<const __nv_bfloat16*>(residual), static_cast<__nv_bfloat16*>(out), s.G, s.H, s.gs,
                   s.groups, vpc);
  if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "conv side1 launch failed: %s", cudaGetErrorString(e));
  if (next_n == nullptr) return DFLASH2_OK;
  // The next RMSNorm as its own row-per-CTA pass: measured faster than fusing it into the
  // apply pass, whose row-per-CTA layout loses the L1 reuse of the previous row.
  return launch_rmsnorm_rows(out, next_w, eps, next_n, s.B, s.G, next_row0, s.H, s.dtype, st, row_off, m_out);
}

int conv_prepare_kernels(const ConvShape& s, bool with_norm) {
  // [RMSNorm] + kernel_projection + side-0 pass, or the two in one kernel for a few rows
  return (with_norm ? 1 : 0) + (kp_small_eligible(s, sm_count()) ? 1 : 2);
}

int conv_finish_kernels(const ConvShape& s, bool with_next_norm) {
  if (!with_next_norm || finish_rows_eligible(s)) return 1;
  return (DFL_FINISH_NORM && finish_norm_cluster(s) > 0) ? 1 : 2;
}

}  // namespace dfl
