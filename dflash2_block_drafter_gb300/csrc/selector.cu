// Edge scores and the greedy walk of the candidate-path selector:
//   S[b, l, p, c] = unary[b, l, c] + sum_r pred_book[pid(b,l,p), r] * z[b, l, r] * succ_book[cand[b, l, c], r],
//   pid(b, 0, p) = anchor[b], pid(b, l, p) = cand[b, l-1, p]
// (MAX DFlash2CandidateSelector, score_edges; dflash2.ts #select), then
//   c_0 = argmax_c S[b, 0, 0, c],  c_l = argmax_c S[b, l, c_{l-1}, c],  path[b, l] = cand[b, l, c_l]
// with ties to the lowest position (MAX select_path: one greedy pass, no beam, no Viterbi).
//
// One CTA per block. All codebook rows a block needs (K successor rows and K predecessor rows per
// slot) are gathered up front with 16-byte loads into shared memory, so the gathers form no
// dependent chain; S is built there in fp32 and the 'steps'-long walk runs from shared memory.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"
#include "warp_keys.cuh"

namespace dfl {
namespace {

constexpr int kThreads = 256;
constexpr int kSmemBudget = 200 * 1024;

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

// Warp argmax over lanes [0, K) (value desc, position asc); every lane gets the winner. Two warp
// reductions: the largest value key, then the lowest lane holding it.
__device__ __forceinline__ int warp_argmax(float v, int K) {
  const int lane = threadIdx.x & 31;
  uint32_t kmax, imin;
  warp_max_min_index(float_key(v), lane < K, static_cast<uint32_t>(lane), kmax, imin);
  return static_cast<int>(imin);
}

// Draft length of block b: all `steps` slots without a depths array; else the tokens a block
// asked to draft depths[b] drafts, min(steps, max(1, depths[b])) (dflash2.ts blockColumns: the
// anchor and max(1, depth) mask rows, at most the block; MAX supports_zero_draft_rows is False).
// Every value is accepted, as blockColumns accepts it.
__device__ __forceinline__ int block_depth(const int32_t* depths, int b, int steps) {
  if (depths == nullptr) return steps;
  return min(steps, max(1, static_cast<int>(depths[b])));
}

// Slots are processed in chunks of `lchunk` (all of them at once at the drafter's shape).
template <typename T>
__global__ void __launch_bounds__(kThreads)
    score_edges_kernel(const int32_t* __restrict__ cand, const float* __restrict__ unary, const float* __restrict__ z,
                       const int32_t* __restrict__ anchors, const T* __restrict__ pred, const T* __restrict__ succ,
                       int steps, int K, int R, int V, int lchunk, float* __restrict__ S, int32_t* __restrict__ path,
                       const int32_t* __restrict__ depths, int* err) {
  extern __shared__ float sm[];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int RP = R + 1;  // padded row: the K successor rows of a slot fall in distinct banks
  int* sid = reinterpret_cast<int*>(sm);               // [steps*K] candidate ids
  float* sS = sm + steps * K;                          // [steps*K*K] scores (for the walk)
  float* sw = sS + steps * K * K;                      // [lchunk*K][RP] pred row * z
  float* sc = sw + lchunk * K * RP;                    // [lchunk*K][RP] succ row
  const int tid = threadIdx.x;
  const int anchor = anchors[b];

  for (int i = tid; i < steps * K; i += kThreads) sid[i] = cand[static_cast<size_t>(b) * steps * K + i];
  __syncthreads();

  const int segs = R / 8;
  for (int l0 = 0; l0 < steps; l0 += lchunk) {
    const int nl = min(lchunk, steps - l0);
    // gather: one 16-byte segment of one row per thread-iteration
    for (int u = tid; u < nl * K * segs; u += kThreads) {
      const int i = u / segs;            // local row index (l - l0) * K + k
      const int sg = u - i * segs;
      const int l = l0 + i / K;
      const int k = i % K;
      const int cid = sid[l * K + k];
      const int pid = (l == 0) ? anchor : sid[(l - 1) * K + k];
      const bool okc = cid >= 0 && cid < V;
      const bool okp = pid >= 0 && pid < V;
      if ((!okc || !okp) && err != nullptr) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_BAD_INDEX));
      float cs[8], ps[8], zs[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cs[j] = 0.f;
        ps[j] = 0.f;
      }
      if (okc) load8(succ + static_cast<size_t>(cid) * R + sg * 8, cs);
      if (okp) load8(pred + static_cast<size_t>(pid) * R + sg * 8, ps);
      load8(z + (static_cast<size_t>(b) * steps + l) * R + sg * 8, zs);
      float* wr = sw + i * RP + sg * 8;
      float* cr = sc + i * RP + sg * 8;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        wr[j] = ps[j] * zs[j];
        cr[j] = cs[j];
      }
    }
    __syncthreads();
    // scores: one (l, p, c) entry per thread-iteration, c fastest
    for (int e = tid; e < nl * K * K; e += kThreads) {
      const int li = e / (K * K);
      const int p = (e / K) % K;
      const int c = e % K;
      const float* wr = sw + (li * K + p) * RP;
      const float* cr = sc + (li * K + c) * RP;
      float acc = 0.f;
      for (int r = 0; r < R; ++r) acc = fmaf(wr[r], cr[r], acc);
      const int l = l0 + li;
      const float s = unary[(static_cast<size_t>(b) * steps + l) * K + c] + acc;
      sS[(l * K + p) * K + c] = s;
      if (S != nullptr) S[((static_cast<size_t>(b) * steps + l) * K + p) * K + c] = s;
    }
    __syncthreads();
  }
  if (path != nullptr && tid < 32) {
    const int d = block_depth(depths, b, steps);
    int p = 0;
    for (int l = 0; l < d; ++l) {
      const float v = tid < K ? sS[(l * K + p) * K + tid] : -INFINITY;
      const int c = warp_argmax(v, K);
      if (tid == 0) path[static_cast<size_t>(b) * steps + l] = sid[l * K + c];
      p = c;
    }
    for (int l = d + tid; l < steps; l += 32) path[static_cast<size_t>(b) * steps + l] = -1;
  }
}

// The walk alone over a given S: one warp per block.
__global__ void __launch_bounds__(128) select_path_kernel(const float* __restrict__ S, const int32_t* __restrict__ cand,
                                                          int B, int steps, int K, int32_t* __restrict__ path,
                                                          const int32_t* __restrict__ depths, int* err) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const int d = block_depth(depths, b, steps);
  for (int l = d + lane; l < steps; l += 32) path[static_cast<size_t>(b) * steps + l] = -1;
  int p = 0;
  for (int l = 0; l < d; ++l) {
    const size_t rowoff = ((static_cast<size_t>(b) * steps + l) * K + p) * K;
    const float v = lane < K ? S[rowoff + lane] : -INFINITY;
    const int c = warp_argmax(v, K);
    if (lane == 0) path[static_cast<size_t>(b) * steps + l] = cand[(static_cast<size_t>(b) * steps + l) * K + c];
    p = c;
  }
}

// Warp-per-slot variant (the drafter's shapes): warp w of block b's CTA handles slots w, w + nw, ...
// It issues every 16-byte segment load of the slot's 2K codebook rows before using any of them
// (one latency round per slot instead of one per loop iteration), keeps pred*z and succ rows in its
// own padded shared-memory rows, and computes the K x K scores with float4 reads (the lanes of a
// quarter-warp read different succ rows at a 4-bank offset: no conflicts). Then warp 0 walks.
constexpr int kEdgeWarpsMax = 16;

__device__ __forceinline__ uint4 ldg16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ void unpack16(const uint4& u, const __nv_bfloat16*, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}
__device__ __forceinline__ void unpack16(const uint4& u, const float*, float* f) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}

template <typename T>
__global__ void __launch_bounds__(32 * kEdgeWarpsMax)
    score_edges_warp_kernel(const int32_t* __restrict__ cand, const float* __restrict__ unary,
                            const float* __restrict__ z, const int32_t* __restrict__ anchors,
                            const T* __restrict__ pred, const T* __restrict__ succ, int steps, int K, int R, int V,
                            float* __restrict__ S, int32_t* __restrict__ path, const int32_t* __restrict__ depths,
                            int tiled, int* err) {
  extern __shared__ float sm[];
  pdl_trigger();
  pdl_wait();
  constexpr int E = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte segment
  const int b = blockIdx.x;
  const int nw = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int RP = R + 4;  // padded row in floats (16-byte aligned, 4-bank offset between rows)
  float* sS = sm;        // [steps][K][K]
  float* rows = sm + ((steps * K * K + 3) & ~3) + warp * (2 * K * RP);  // [K] pred*z rows, [K] succ rows
  const int anchor = anchors[b];
  const int segs = R / E;
  const int items = 2 * K * segs;
  for (int l = warp; l < steps; l += nw) {
    const size_t slot = static_cast<size_t>(b) * steps + l;
    const float* zl = z + slot * R;
    // K = 16: this lane's four unary values, loaded before the gathers (no dependence on them)
    const float4 un4 = tiled ? __ldg(reinterpret_cast<const float4*>(unary + slot * K) + (lane & 3))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    // When 32 is a multiple of segs every item of this lane has the same segment: its z values
    // are loaded here, alongside the gathers rather than after them.
    const bool fixed_sg = (32 % segs) == 0;
    float zf[E];
#pragma unroll
    for (int e = 0; e < E; ++e) zf[e] = fixed_sg ? __ldg(zl + (lane % segs) * E + e) : 0.f;
    for (int q0 = 0; q0 < items; q0 += 32 * 8) {
      // Branch-free in two rounds: every candidate id of this lane's 8 items first, then every row
      // segment (an invalid id or an item past the end reads row 0 and is zeroed afterwards), so
      // the compiler can keep all 8 loads of each round in flight at once.
      int ids[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = min(q0 + i * 32 + lane, items - 1);
        const int row = q / segs;
        const bool from_anchor = row < K && l == 0;  // slot 0's predecessor is the anchor
        const size_t src = from_anchor ? 0 : (row < K ? (slot - 1) * K + row : slot * K + row - K);
        ids[i] = from_anchor ? anchor : __ldg(cand + src);
      }
      uint4 buf[8];
      bool bad = false;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = min(q0 + i * 32 + lane, items - 1);
        const int row = q / segs;
        const int sg = q - row * segs;
        const bool ok = ids[i] >= 0 && ids[i] < V;
        bad |= !ok && (q0 + i * 32 + lane < items);
        buf[i] = ldg16((row < K ? pred : succ) + static_cast<size_t>(ok ? ids[i] : 0) * R + sg * E);
        if (!ok) buf[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (bad && err != nullptr) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_BAD_INDEX));
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = q0 + i * 32 + lane;
        if (q < items) {
          const int row = q / segs;
          const int sg = q - row * segs;
          float f[E];
          unpack16(buf[i], static_cast<const T*>(nullptr), f);
          float* dst = rows + row * RP + sg * E;
          if (row < K) {
#pragma unroll
            for (int e = 0; e < E; ++e) dst[e] = f[e] * (fixed_sg ? zf[e] : __ldg(zl + sg * E + e));
          } else {
#pragma unroll
            for (int e = 0; e < E; ++e) dst[e] = f[e];
          }
        }
      }
    }
    __syncwarp();
    if (tiled) {
      // K = 16 (unary and S 16-byte aligned): 2 x 4 register tile per lane: rows p0, p0+1 of pred*z against succ rows c0..c0+3, so each
      // 4-wide step of r reads 6 float4 for 32 multiply-adds (same order of r as the plain loop)
      const int p0 = 2 * (lane >> 2);
      const int c0 = 4 * (lane & 3);
      float acc[2][4] = {};
      for (int r = 0; r < R; r += 4) {
        float4 a4[2], c4[4];
#pragma unroll
        for (int i = 0; i < 2; ++i) a4[i] = *reinterpret_cast<const float4*>(rows + (p0 + i) * RP + r);
#pragma unroll
        for (int j = 0; j < 4; ++j) c4[j] = *reinterpret_cast<const float4*>(rows + (K + c0 + j) * RP + r);
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[i][j] = fmaf(a4[i].x, c4[j].x, acc[i][j]);
            acc[i][j] = fmaf(a4[i].y, c4[j].y, acc[i][j]);
            acc[i][j] = fmaf(a4[i].z, c4[j].z, acc[i][j]);
            acc[i][j] = fmaf(a4[i].w, c4[j].w, acc[i][j]);
          }
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float4 o;
        o.x = un4.x + acc[i][0];
        o.y = un4.y + acc[i][1];
        o.z = un4.z + acc[i][2];
        o.w = un4.w + acc[i][3];
        *reinterpret_cast<float4*>(sS + (l * K + p0 + i) * K + c0) = o;
        if (S != nullptr) *reinterpret_cast<float4*>(S + (slot * K + p0 + i) * K + c0) = o;
      }
    } else {
      for (int e = lane; e < K * K; e += 32) {
        const int p = e / K;
        const int c = e - p * K;
        const float* wr = rows + p * RP;
        const float* cr = rows + (K + c) * RP;
        float acc = 0.f;
        for (int r = 0; r < R; r += 4) {
          const float4 a4 = *reinterpret_cast<const float4*>(wr + r);
          const float4 c4 = *reinterpret_cast<const float4*>(cr + r);
          acc = fmaf(a4.x, c4.x, acc);
          acc = fmaf(a4.y, c4.y, acc);
          acc = fmaf(a4.z, c4.z, acc);
          acc = fmaf(a4.w, c4.w, acc);
        }
        const float s = __ldg(unary + slot * K + c) + acc;
        sS[(l * K + p) * K + c] = s;
        if (S != nullptr) S[(slot * K + p) * K + c] = s;
      }
    }
    __syncwarp();  // the next slot overwrites this warp's rows
  }
  __syncthreads();
  if (path != nullptr && warp == 0) {
    // The walk touches only shared memory: lane l keeps the position chosen at slot l (lane l - 32
    // for slots 32..63), and the candidate ids are looked up afterwards in one parallel round.
    const int d = block_depth(depths, b, steps);
    int p = 0, pos_lo = 0, pos_hi = 0;
    for (int l = 0; l < d; ++l) {
      const float v = lane < K ? sS[(l * K + p) * K + lane] : -INFINITY;
      const int c = warp_argmax(v, K);
      if (lane == l) pos_lo = c;
      if (lane + 32 == l) pos_hi = c;
      p = c;
    }
    const size_t base_slot = static_cast<size_t>(b) * steps;
    for (int h = 0; h < 2; ++h) {
      const int l = lane + 32 * h;
      if (l >= steps) break;
      path[base_slot + l] = l < d ? cand[(base_slot + l) * K + (h == 0 ? pos_lo : pos_hi)] : -1;
    }
  }
}

size_t edges_smem(int steps, int K, int R, int lchunk) {
  return sizeof(float) * (static_cast<size_t>(steps) * K + static_cast<size_t>(steps) * K * K +
                          2 * static_cast<size_t>(lchunk) * K * (R + 1));
}

}  // namespace

#ifndef DFL_EDGE_WARP
#define DFL_EDGE_WARP 1
#endif

int launch_score_edges(const int32_t* cand, const float* unary, const float* z, const int32_t* anchors,
                       const void* pred, const void* succ, int B, int steps, int K, int R, int V, int dtype,
                       float* S, int32_t* path, cudaStream_t st, const int32_t* depths) {
  {
    // warp-per-slot kernel when its scores and at least a few warps' rows fit in shared memory
    const size_t s_floats = (static_cast<size_t>(steps) * K * K + 3) & ~static_cast<size_t>(3);
    const size_t per_warp = 2 * static_cast<size_t>(K) * (R + 4);
    const size_t budget = kSmemBudget / sizeof(float);
    const int nw = s_floats + per_warp <= budget
                       ? static_cast<int>(std::min<size_t>({static_cast<size_t>(kEdgeWarpsMax),
                                                            static_cast<size_t>(steps), (budget - s_floats) / per_warp}))
                       : 0;
    if (DFL_EDGE_WARP && nw >= 4) {
      const size_t smem = sizeof(float) * (s_floats + nw * per_warp);
      const int tiled = K == 16 && reinterpret_cast<uintptr_t>(unary) % 16 == 0 &&
                        reinterpret_cast<uintptr_t>(S) % 16 == 0;  // float4 unary loads and S stores
      static unsigned dw_f32 = 0, dw_bf16 = 0;
      cudaError_t e = cudaSuccess;
      if (dtype == DFLASH2_F32) {
        if (!ensure_smem_attr(score_edges_warp_kernel<float>, kSmemBudget, &dw_f32)) e = cudaErrorInvalidValue;
        if (e == cudaSuccess)
          e = launch_pdl(score_edges_warp_kernel<float>, dim3(B), dim3(32 * nw), smem, st, nullptr, 0, cand, unary, z,
                         anchors, static_cast<const float*>(pred), static_cast<const float*>(succ), steps, K, R, V, S,
                         path, depths, tiled, device_error_word());
      } else {
        if (!ensure_smem_attr(score_edges_warp_kernel<__nv_bfloat16>, kSmemBudget, &dw_bf16)) e = cudaErrorInvalidValue;
        if (e == cudaSuccess)
          e = launch_pdl(score_edges_warp_kernel<__nv_bfloat16>, dim3(B), dim3(32 * nw), smem, st, nullptr, 0, cand,
                         unary, z, anchors, static_cast<const __nv_bfloat16*>(pred),
                         static_cast<const __nv_bfloat16*>(succ), steps, K, R, V, S, path, depths, tiled,
                         device_error_word());
      }
      return e == cudaSuccess ? DFLASH2_OK
                              : fail(DFLASH2_ERR_CUDA, "score_edges launch failed: %s", cudaGetErrorString(e));
    }
  }
  int lchunk = steps;
  while (lchunk > 1 && edges_smem(steps, K, R, lchunk) > static_cast<size_t>(kSmemBudget)) --lchunk;
  const size_t smem = edges_smem(steps, K, R, lchunk);
  if (smem > static_cast<size_t>(kSmemBudget))
    return fail(DFLASH2_ERR_INVALID_ARG, "score_edges: steps*K*K too large for shared memory");
  static unsigned done_f32 = 0, done_bf16 = 0;
  cudaError_t e = cudaSuccess;
  if (dtype == DFLASH2_F32) {
    if (!ensure_smem_attr(score_edges_kernel<float>, kSmemBudget, &done_f32)) e = cudaErrorInvalidValue;
    if (e == cudaSuccess)
      e = launch_pdl(score_edges_kernel<float>, dim3(B), dim3(kThreads), smem, st, nullptr, 0, cand, unary, z, anchors,
                     static_cast<const float*>(pred), static_cast<const float*>(succ), steps, K, R, V, lchunk, S, path,
                     depths, device_error_word());
  } else {
    if (!ensure_smem_attr(score_edges_kernel<__nv_bfloat16>, kSmemBudget, &done_bf16)) e = cudaErrorInvalidValue;
    if (e == cudaSuccess)
      e = launch_pdl(score_edges_kernel<__nv_bfloat16>, dim3(B), dim3(kThreads), smem, st, nullptr, 0, cand, unary, z,
                     anchors, static_cast<const __nv_bfloat16*>(pred), static_cast<const __nv_bfloat16*>(succ), steps,
                     K, R, V, lchunk, S, path, depths, device_error_word());
  }
  return e == cudaSuccess ? DFLASH2_OK : fail(DFLASH2_ERR_CUDA, "score_edges launch failed: %s", cudaGetErrorString(e));
}

int launch_select_path(const float* S, const int32_t* cand, int B, int steps, int K, int32_t* path,
                       cudaStream_t st, const int32_t* depths) {
  const cudaError_t e = launch_pdl(select_path_kernel, dim3((B + 3) / 4), dim3(128), 0, st, nullptr, 0, S, cand, B,
                                   steps, K, path, depths, device_error_word());
  return e == cudaSuccess ? DFLASH2_OK : fail(DFLASH2_ERR_CUDA, "select_path launch failed: %s", cudaGetErrorString(e));
}

}  // namespace dfl
