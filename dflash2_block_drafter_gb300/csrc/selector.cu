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

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

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

// Warp argmax over lanes [0, K) (value desc, position asc); every lane gets the winner.
__device__ __forceinline__ int warp_argmax(float v, int K) {
  const int lane = threadIdx.x & 31;
  float bv = lane < K ? v : -INFINITY;
  int bi = lane < K ? lane : 0x7fffffff;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
    if (ov > bv || (ov == bv && oi < bi)) {
      bv = ov;
      bi = oi;
    }
  }
  return bi;
}

// Draft length of block b: depths[b] slots (the rest of the block's rows are padding of a
// mixed-depth batch; dflash2.ts blockColumns), all `steps` without a depths array. A value
// outside [0, steps] records DFLASH2_ERR_INVALID_ARG in the error word and is clamped.
__device__ __forceinline__ int block_depth(const int32_t* depths, int b, int steps, int* err) {
  if (depths == nullptr) return steps;
  const int d = depths[b];
  if (d < 0 || d > steps) {
    if (err != nullptr) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_INVALID_ARG));
    return d < 0 ? 0 : steps;
  }
  return d;
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
    const int d = block_depth(depths, b, steps, err);
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
  const int d = block_depth(depths, b, steps, err);
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

size_t edges_smem(int steps, int K, int R, int lchunk) {
  return sizeof(float) * (static_cast<size_t>(steps) * K + static_cast<size_t>(steps) * K * K +
                          2 * static_cast<size_t>(lchunk) * K * (R + 1));
}

}  // namespace

int launch_score_edges(const int32_t* cand, const float* unary, const float* z, const int32_t* anchors,
                       const void* pred, const void* succ, int B, int steps, int K, int R, int V, int dtype,
                       float* S, int32_t* path, cudaStream_t st, const int32_t* depths) {
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
