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

// Rows of block b: `steps` slots at b * steps, or (row_off given, a ragged batch) the
// row_off[b + 1] - row_off[b] slots at row_off[b] of an m_rows-row input. A block whose span is not
// inside [0, m_rows) or holds outside [1, steps] slots records DFLASH2_ERR_INVALID_ARG (when err is
// given) and is skipped (its path is all -1).
struct SlotSpan {
  size_t first;
  int n;
};
__device__ __forceinline__ SlotSpan block_slots(const int32_t* row_off, int b, int steps, int m_rows, int* err) {
  if (row_off == nullptr) return SlotSpan{static_cast<size_t>(b) * steps, steps};
  const int lo = row_off[b];
  const int n = row_off[b + 1] - lo;
  if (lo < 0 || n < 1 || n > steps || lo > m_rows - n) {
    if (err != nullptr) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_INVALID_ARG));
    return SlotSpan{0, 0};
  }
  return SlotSpan{static_cast<size_t>(lo), n};
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

// K = 16 kernel (the drafter's top-16): a CTA per block, W warps taking slots w, w + W, ...
// Lane (c = lane & 15, half = lane >> 4) keeps successor row cand[c]'s half of r in registers
// (fp32), the warp's 16 predecessor rows times z go to a padded shared-memory tile, and every
// lane accumulates the 16 scores S[p][c] over its half of r with packed fp32 FMAs, reading the
// tile as float4 broadcasts (the two halves sit 4 banks apart). One shuffle adds the halves.
// The gathers of the warp's next slot are issued before the current slot is computed, and the
// candidate ids two slots ahead before that, so each warp keeps a slot's rows in flight while it
// computes. Every slot's 16 x 16 scores go to shared memory for the walk (warp 0, after the CTA
// barrier) and, when requested, to S.
template <typename T, int R>
struct K16Slot {
  static constexpr int E = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte segment
  static constexpr int NS = R / E;                             // segments per codebook row
  static constexpr int PS = NS / 2;                            // segments per lane (pred and succ)
  static constexpr int HR = R / 2;                             // r values per half
  static constexpr int WS = R + 8;                             // floats per pred*z row (2 halves + pad)
  static_assert(NS >= 2 && NS <= 32 && (32 % NS) == 0, "row segments must tile a warp");
};

template <typename T, int R>
__device__ __forceinline__ void k16_ids(const int32_t* __restrict__ cand, int anchor, size_t slot, int l, int lane,
                                        int& cid, int (&pid)[K16Slot<T, R>::PS]) {
  using P = K16Slot<T, R>;
  cid = __ldg(cand + slot * 16 + (lane & 15));
#pragma unroll
  for (int i = 0; i < P::PS; ++i) {
    const int p = lane / P::NS + i * (32 / P::NS);
    pid[i] = l == 0 ? anchor : __ldg(cand + (slot - 1) * 16 + p);
  }
}

template <typename T, int R>
__device__ __forceinline__ bool k16_rows(const T* __restrict__ pred, const T* __restrict__ succ, int V, int lane,
                                         int cid, const int (&pid)[K16Slot<T, R>::PS], uint4 (&rs)[K16Slot<T, R>::PS],
                                         uint4 (&rp)[K16Slot<T, R>::PS]) {
  using P = K16Slot<T, R>;
  const int half = lane >> 4;
  const int sg = lane % P::NS;
  const bool okc = cid >= 0 && cid < V;
  bool bad = !okc;
  const T* srow = succ + static_cast<size_t>(okc ? cid : 0) * R + half * P::HR;
#pragma unroll
  for (int j = 0; j < P::PS; ++j) rs[j] = ldg16(srow + j * P::E);
  if (!okc)
#pragma unroll
    for (int j = 0; j < P::PS; ++j) rs[j] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int i = 0; i < P::PS; ++i) {
    const bool ok = pid[i] >= 0 && pid[i] < V;
    bad |= !ok;
    rp[i] = ldg16(pred + static_cast<size_t>(ok ? pid[i] : 0) * R + sg * P::E);
    if (!ok) rp[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  return bad;
}

template <typename T, int R>
__global__ void __launch_bounds__(512)
    score_edges_k16_kernel(const int32_t* __restrict__ cand, const float* __restrict__ unary,
                           const float* __restrict__ z, const int32_t* __restrict__ anchors,
                           const T* __restrict__ pred, const T* __restrict__ succ, int steps, int V,
                           float* __restrict__ S, int32_t* __restrict__ path, const int32_t* __restrict__ depths,
                           const int32_t* __restrict__ row_off, int m_rows, int* err) {
  using P = K16Slot<T, R>;
  constexpr int PS = P::PS, E = P::E, NS = P::NS, HR = P::HR, WS = P::WS;
  extern __shared__ float sm[];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int W = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = lane & 15;
  const int half = lane >> 4;
  const int sg = lane % NS;  // this lane's segment of each predecessor row it gathers
  float* sS = sm;            // [steps][16][16]
  float* wt = sm + steps * 256 + warp * 16 * WS;  // [16][2 halves][HR + 4] pred rows * z
  const int anchor = __ldg(anchors + b);
  const SlotSpan span = block_slots(row_off, b, steps, m_rows, threadIdx.x == 0 ? err : nullptr);
  const size_t slot0 = span.first;
  const int nst = span.n;
  bool bad = false;

  int l = warp;
  int cid = 0, pid[PS] = {};
  uint4 rs[PS], rp[PS];
  float zc[E];
  float un = 0.f;
  if (l < nst) {
    k16_ids<T, R>(cand, anchor, slot0 + l, l, lane, cid, pid);
    bad |= k16_rows<T, R>(pred, succ, V, lane, cid, pid, rs, rp);
#pragma unroll
    for (int e = 0; e < E; e += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(z + (slot0 + l) * R + sg * E + e));
      zc[e] = v.x; zc[e + 1] = v.y; zc[e + 2] = v.z; zc[e + 3] = v.w;
    }
    un = __ldg(unary + (slot0 + l) * 16 + c);
  }
  int cidn = 0, pidn[PS] = {};
  if (l + W < nst) k16_ids<T, R>(cand, anchor, slot0 + l + W, l + W, lane, cidn, pidn);

  for (; l < nst; l += W) {
    const int ln = l + W;
    // next slot's rows, z and unary; the ids one slot further
    uint4 rsn[PS], rpn[PS];
    float zn[E];
    float unn = 0.f;
    if (ln < nst) {
      bad |= k16_rows<T, R>(pred, succ, V, lane, cidn, pidn, rsn, rpn);
#pragma unroll
      for (int e = 0; e < E; e += 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(z + (slot0 + ln) * R + sg * E + e));
        zn[e] = v.x; zn[e + 1] = v.y; zn[e + 2] = v.z; zn[e + 3] = v.w;
      }
      unn = __ldg(unary + (slot0 + ln) * 16 + c);
      if (ln + W < nst) k16_ids<T, R>(cand, anchor, slot0 + ln + W, ln + W, lane, cidn, pidn);
    }
    // predecessor rows times z into the warp's tile
#pragma unroll
    for (int i = 0; i < PS; ++i) {
      const int p = lane / NS + i * (32 / NS);
      float f[E];
      unpack16(rp[i], static_cast<const T*>(nullptr), f);
      const int r0 = sg * E;
      float* dst = wt + p * WS + (r0 >= HR ? HR + 4 : 0) + (r0 % HR);
#pragma unroll
      for (int e = 0; e < E; e += 4)
        *reinterpret_cast<float4*>(dst + e) =
            make_float4(f[e] * zc[e], f[e + 1] * zc[e + 1], f[e + 2] * zc[e + 2], f[e + 3] * zc[e + 3]);
    }
    // this lane's successor half-row in registers
    float sv[HR];
#pragma unroll
    for (int j = 0; j < PS; ++j) unpack16(rs[j], static_cast<const T*>(nullptr), sv + j * E);
    __syncwarp();
    float2 acc[16];
#pragma unroll
    for (int p = 0; p < 16; ++p) acc[p] = make_float2(0.f, 0.f);
    const float* wr = wt + half * (HR + 4);
#pragma unroll
    for (int j = 0; j < HR; j += 4) {
#pragma unroll
      for (int p = 0; p < 16; ++p) {
        const float4 w4 = *reinterpret_cast<const float4*>(wr + p * WS + j);
        acc[p] = __ffma2_rn(make_float2(w4.x, w4.y), make_float2(sv[j], sv[j + 1]), acc[p]);
        acc[p] = __ffma2_rn(make_float2(w4.z, w4.w), make_float2(sv[j + 2], sv[j + 3]), acc[p]);
      }
    }
    __syncwarp();  // the tile is rewritten for the next slot
    const size_t slot = slot0 + l;
#pragma unroll
    for (int pp = 0; pp < 8; ++pp) {
      float v0 = acc[2 * pp].x + acc[2 * pp].y;
      float v1 = acc[2 * pp + 1].x + acc[2 * pp + 1].y;
      v0 += __shfl_xor_sync(0xffffffffu, v0, 16);
      v1 += __shfl_xor_sync(0xffffffffu, v1, 16);
      const int p = 2 * pp + half;
      const float v = un + (half ? v1 : v0);
      sS[(l * 16 + p) * 16 + c] = v;
      if (S != nullptr) S[(slot * 16 + p) * 16 + c] = v;
    }
    // rotate the pipeline
#pragma unroll
    for (int j = 0; j < PS; ++j) {
      rs[j] = rsn[j];
      rp[j] = rpn[j];
    }
#pragma unroll
    for (int e = 0; e < E; ++e) zc[e] = zn[e];
    un = unn;
  }
  if (bad && err != nullptr) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_BAD_INDEX));
  __syncthreads();
  if (path != nullptr && warp == 0) {
    const int d = row_off != nullptr ? nst : block_depth(depths, b, steps);
    int p = 0, pos_lo = 0, pos_hi = 0;
    for (int t = 0; t < d; ++t) {
      const float v = lane < 16 ? sS[(t * 16 + p) * 16 + lane] : -INFINITY;
      const int cc = warp_argmax(v, 16);
      if (lane == t) pos_lo = cc;
      if (lane + 32 == t) pos_hi = cc;
      p = cc;
    }
    for (int h2 = 0; h2 < 2; ++h2) {
      const int t = lane + 32 * h2;
      if (t >= steps) break;
      path[static_cast<size_t>(b) * steps + t] = t < d ? __ldg(cand + (slot0 + t) * 16 + (h2 == 0 ? pos_lo : pos_hi)) : -1;
    }
  }
}

size_t edges_smem(int steps, int K, int R, int lchunk) {
  return sizeof(float) * (static_cast<size_t>(steps) * K + static_cast<size_t>(steps) * K * K +
                          2 * static_cast<size_t>(lchunk) * K * (R + 1));
}

}  // namespace

// bf16 codebooks, K = 16: each slot's edge term is a 16 x 16 x R product of the predecessor rows
// times z (fp32) and the successor rows (bf16), done on the tensor cores with warp-level
// mma.sync m16n8k8 tf32, straight from registers. The operand fragments are gathered directly:
// the reduction index k of each MMA is mapped to r so that lane t (= lane & 3) owns the
// contiguous chunk r in [t R/4, (t + 1) R/4) of its rows, which it loads as 16-byte vectors
// (g = lane >> 2 gives the rows g and g + 8). Successor values are bf16, so exact in tf32; the
// product w = pred * z is split into w_big = tf32(w) and w_small = w - w_big and both are
// multiplied, so every product keeps about 21 bits (the error is below 2^-21 |w succ| per term),
// with fp32 accumulation. One CTA per block: warp w takes slots w, w + W, ... . For every slot the
// warp also reduces each predecessor row p to its best successor position (largest score, lowest
// position on a tie) in shared memory, so that the walk after the CTA barrier is a chain of
// table lookups, c_l = best[l][c_{l-1}], run by one thread.
__device__ __forceinline__ void mma_16x8x8_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

template <int R>
__global__ void __launch_bounds__(512, 2)
    score_edges_mma_kernel(const int32_t* __restrict__ cand, const float* __restrict__ unary,
                           const float* __restrict__ z, const int32_t* __restrict__ anchors,
                           const __nv_bfloat16* __restrict__ pred, const __nv_bfloat16* __restrict__ succ, int steps,
                           int V, float* __restrict__ S, int32_t* __restrict__ path,
                           const int32_t* __restrict__ depths, const int32_t* __restrict__ row_off, int m_rows,
                           int* err) {
  constexpr int Q = R / 4;   // r values per lane and row
  constexpr int NV = Q / 8;  // 16-byte vectors per lane and row
  constexpr int KS = R / 8;  // MMA k-steps
  static_assert(NV >= 1 && Q % 8 == 0, "R must be a multiple of 32");
  extern __shared__ float sm[];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int W = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  int* sId = reinterpret_cast<int*>(sm);                       // [steps][16] candidate ids, then [steps] path
  uint8_t* sBest = reinterpret_cast<uint8_t*>(sId + steps * 17);  // [steps][16] best successor of each row
  const int anchor = __ldg(anchors + b);
  const SlotSpan span = block_slots(row_off, b, steps, m_rows, threadIdx.x == 0 ? err : nullptr);
  const size_t slot0 = span.first;
  const int nst = span.n;
  bool bad = false;
  for (int l = warp; l < nst; l += W) {
    const size_t slot = slot0 + l;
    // this lane's rows: successors g and g + 8 of the slot, predecessors g and g + 8
    int cs[2], ps[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      cs[h] = __ldg(cand + slot * 16 + g + 8 * h);
      ps[h] = l == 0 ? anchor : __ldg(cand + (slot - 1) * 16 + g + 8 * h);
    }
    // z and unary do not depend on the ids: in flight with them, before the row gathers
    float zc[Q];
#pragma unroll
    for (int e = 0; e < Q; e += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(z + slot * R + Q * t + e));
      zc[e] = v.x; zc[e + 1] = v.y; zc[e + 2] = v.z; zc[e + 3] = v.w;
    }
    float u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = __ldg(unary + slot * 16 + 2 * t + (i & 1) + 8 * (i >> 1));
    uint4 sv[2][NV], pv[2][NV];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const bool okc = cs[h] >= 0 && cs[h] < V;
      const bool okp = ps[h] >= 0 && ps[h] < V;
      bad |= !okc || !okp;
      const __nv_bfloat16* srow = succ + static_cast<size_t>(okc ? cs[h] : 0) * R + Q * t;
      const __nv_bfloat16* prow = pred + static_cast<size_t>(okp ? ps[h] : 0) * R + Q * t;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        sv[h][v] = okc ? ldg16(srow + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
        pv[h][v] = okp ? ldg16(prow + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float acc[2][4] = {};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int v = ks / 4, wi = ks % 4;
      const uint32_t p0 = word_of(pv[0][v], wi), p1 = word_of(pv[1][v], wi);
      const float w0 = __uint_as_float(p0 << 16) * zc[2 * ks];              // row g,     r = Qt + 2ks
      const float w1 = __uint_as_float(p1 << 16) * zc[2 * ks];              // row g + 8, r = Qt + 2ks
      const float w2 = __uint_as_float(p0 & 0xffff0000u) * zc[2 * ks + 1];  // row g,     r = Qt + 2ks + 1
      const float w3 = __uint_as_float(p1 & 0xffff0000u) * zc[2 * ks + 1];  // row g + 8, r = Qt + 2ks + 1
      const uint32_t h0 = tf32_rna(w0), h1 = tf32_rna(w1), h2 = tf32_rna(w2), h3 = tf32_rna(w3);
      const uint32_t l0 = __float_as_uint(w0 - __uint_as_float(h0)), l1 = __float_as_uint(w1 - __uint_as_float(h1));
      const uint32_t l2 = __float_as_uint(w2 - __uint_as_float(h2)), l3 = __float_as_uint(w3 - __uint_as_float(h3));
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        const uint32_t sw = word_of(sv[n][v], wi);  // successor row g + 8n: r = Qt + 2ks (lo), + 1 (hi)
        mma_16x8x8_tf32(acc[n], h0, h1, h2, h3, sw << 16, sw & 0xffff0000u);
        mma_16x8x8_tf32(acc[n], l0, l1, l2, l3, sw << 16, sw & 0xffff0000u);
      }
    }
    // acc[n] = S[g][8n + 2t], S[g][8n + 2t + 1], S[g + 8][8n + 2t], S[g + 8][8n + 2t + 1] (edge terms)
    uint32_t bk[2] = {0u, 0u};
    int bc[2] = {0, 0};
#pragma unroll
    for (int n = 0; n < 2; ++n) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int hr = i >> 1;  // row g + 8 hr
        const int c = 8 * n + 2 * t + (i & 1);
        const float val = u[2 * n + (i & 1)] + acc[n][i];
        if (S != nullptr) S[(slot * 16 + g + 8 * hr) * 16 + c] = val;
        // best successor of each predecessor row: largest score, lowest position on a tie
        const uint32_t k = float_key(val);
        if ((n == 0 && (i & 1) == 0) || k > bk[hr] || (k == bk[hr] && c < bc[hr])) {
          bk[hr] = k;
          bc[hr] = c;
        }
      }
    }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const uint32_t ok = __shfl_xor_sync(0xffffffffu, bk[hr], m);
        const int oc = __shfl_xor_sync(0xffffffffu, bc[hr], m);
        if (ok > bk[hr] || (ok == bk[hr] && oc < bc[hr])) {
          bk[hr] = ok;
          bc[hr] = oc;
        }
      }
    }
    if (t == 0) {
      sBest[l * 16 + g] = static_cast<uint8_t>(bc[0]);
      sBest[l * 16 + g + 8] = static_cast<uint8_t>(bc[1]);
      sId[l * 16 + g] = cs[0];
      sId[l * 16 + g + 8] = cs[1];
    }
  }
  if (bad && err != nullptr) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_BAD_INDEX));
  __syncthreads();
  if (path != nullptr && warp == 0) {
    // the walk follows the best-successor table: c_l = best[l][c_{l-1}], c_{-1} = 0
    int* sPath = sId + steps * 16;
    if (lane == 0) {
      const int d = row_off != nullptr ? nst : block_depth(depths, b, steps);
      int p = 0;
      for (int tt = 0; tt < steps; ++tt) {
        if (tt < d) {
          p = sBest[tt * 16 + p];
          sPath[tt] = sId[tt * 16 + p];
        } else {
          sPath[tt] = -1;
        }
      }
    }
    __syncwarp();
    for (int tt = lane; tt < steps; tt += 32) path[static_cast<size_t>(b) * steps + tt] = sPath[tt];
  }
}

template <int R>
cudaError_t launch_mma_t(const int32_t* cand, const float* unary, const float* z, const int32_t* anchors,
                         const void* pred, const void* succ, int B, int steps, int V, float* S, int32_t* path,
                         cudaStream_t st, const int32_t* depths, const int32_t* row_off, int m_rows, int W,
                         size_t smem) {
  static unsigned done = 0;
  if (!ensure_smem_attr(score_edges_mma_kernel<R>, kSmemBudget, &done)) return cudaErrorInvalidValue;
  return launch_pdl(score_edges_mma_kernel<R>, dim3(B), dim3(32 * W), smem, st, nullptr, 0, cand, unary, z, anchors,
                    static_cast<const __nv_bfloat16*>(pred), static_cast<const __nv_bfloat16*>(succ), steps, V, S,
                    path, depths, row_off, m_rows, device_error_word());
}

template <typename T, int R>
cudaError_t launch_k16_t(const int32_t* cand, const float* unary, const float* z, const int32_t* anchors,
                         const void* pred, const void* succ, int B, int steps, int V, float* S, int32_t* path,
                         cudaStream_t st, const int32_t* depths, const int32_t* row_off, int m_rows, int W,
                         size_t smem) {
  static unsigned done = 0;
  if (!ensure_smem_attr(score_edges_k16_kernel<T, R>, kSmemBudget, &done)) return cudaErrorInvalidValue;
  return launch_pdl(score_edges_k16_kernel<T, R>, dim3(B), dim3(32 * W), smem, st, nullptr, 0, cand, unary, z,
                    anchors, static_cast<const T*>(pred), static_cast<const T*>(succ), steps, V, S, path, depths,
                    row_off, m_rows, device_error_word());
}

int launch_k16(const int32_t* cand, const float* unary, const float* z, const int32_t* anchors, const void* pred,
               const void* succ, int B, int steps, int R, int V, int dtype, float* S, int32_t* path,
               cudaStream_t st, const int32_t* depths, const int32_t* row_off, int m_rows, int W, size_t smem) {
  if (smem > static_cast<size_t>(kSmemBudget))
    return fail(DFLASH2_ERR_INVALID_ARG, "score_edges: steps=%d needs %zu bytes of shared memory", steps, smem);
  cudaError_t e = cudaErrorInvalidValue;
#define DFL_K16(TT, RR)                                                                                      \
  e = launch_k16_t<TT, RR>(cand, unary, z, anchors, pred, succ, B, steps, V, S, path, st, depths, row_off, m_rows, W, \
                           smem)
  if (dtype == DFLASH2_F32) {
    if (R == 16) DFL_K16(float, 16); else DFL_K16(float, 32);
  } else {
    DFL_K16(__nv_bfloat16, 16);
  }
#undef DFL_K16
  return e == cudaSuccess ? DFLASH2_OK : fail(DFLASH2_ERR_CUDA, "score_edges launch failed: %s", cudaGetErrorString(e));
}

#ifndef DFL_EDGE_WARP
#define DFL_EDGE_WARP 1
#endif

int launch_score_edges(const int32_t* cand, const float* unary, const float* z, const int32_t* anchors,
                       const void* pred, const void* succ, int B, int steps, int K, int R, int V, int dtype,
                       float* S, int32_t* path, cudaStream_t st, const int32_t* depths, const int32_t* row_off,
                       int m_rows) {
  if (K == 16 && dtype == DFLASH2_BF16 && (R == 32 || R == 64)) {
    // tensor-core edge terms; W warps per block: every CTA resident at once at 32 warps per SM
    // where B allows (a slot per warp at small B), down to 4 warps at large B
    const int sms = sm_count();
    int W = 16;
    while (W > 4 && static_cast<long long>(B) * W > 32LL * sms) W >>= 1;
    W = std::max(1, std::min(W, steps));
    const size_t smem = static_cast<size_t>(steps) * (17 * sizeof(int) + 16);
    const cudaError_t e =
        R == 32 ? launch_mma_t<32>(cand, unary, z, anchors, pred, succ, B, steps, V, S, path, st, depths, row_off,
                                   m_rows, W, smem)
                : launch_mma_t<64>(cand, unary, z, anchors, pred, succ, B, steps, V, S, path, st, depths, row_off,
                                   m_rows, W, smem);
    return e == cudaSuccess ? DFLASH2_OK
                            : fail(DFLASH2_ERR_CUDA, "score_edges launch failed: %s", cudaGetErrorString(e));
  }
  // the register-tiled FMA kernel for the other K = 16 shapes whose registers fit (f32 rows up to
  // R = 32, bf16 rows of R = 16)
  if (K == 16 && (R == 16 || (R == 32 && dtype == DFLASH2_F32))) {
    // W warps per block: as many as keep every CTA resident in one wave at 16 warps per SM (a
    // slot per warp at small B, for latency), down to 2 at large B (pipelined slots per warp)
    const int sms = sm_count();
    int W = 16;
    while (W > 2 && static_cast<long long>(B) * W > 16LL * sms) W >>= 1;
    W = std::max(1, std::min(W, steps));
    const size_t smem = sizeof(float) * (static_cast<size_t>(steps) * 256 + static_cast<size_t>(W) * 16 * (R + 8));
    return launch_k16(cand, unary, z, anchors, pred, succ, B, steps, R, V, dtype, S, path, st, depths, row_off,
                      m_rows, W, smem);
  }
  if (row_off != nullptr)
    return fail(DFLASH2_ERR_UNSUPPORTED,
                "ragged rows need K = 16 and R in {16, 32, 64} (bf16) or {16, 32} (f32); got K=%d, R=%d", K, R);
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
