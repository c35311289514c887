// The two-tap dynamic grouped depthwise conv around each drafter sublayer:
//   Conv_side(y)[t, c] = sum_tau (base[side, tau, c] + D[t, side, tau, c / gs]) * y[t - tau, c],
// t block-local, y[-1] = 0 (dflash2.ts header "layer" paragraph, #coefficients, #conv; MAX
// DFlash2GroupedConv). D = kernel_projection(n) comes from the tensor-core GEMM (gemm.cu) as
// fp32 split-K partials; the coefficient broadcast (base + per-group delta) is fused into the
// apply passes and never materialised at channel width.
//
// Apply passes: one thread owns 8 consecutive channels (one 16-byte bf16 vector) of one block
// and walks the block's G rows in order, carrying row t-1 in registers, so each input element
// is read once and each output written once. The finish pass can also emit the next RMSNorm:
// the row reduction spans the block's channels across one thread-block cluster (DSMEM).
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "internal.h"

namespace cg = cooperative_groups;

namespace dfl {
namespace {

constexpr int kApplyThreads = 128;            // threads per apply CTA (8 channels each)
constexpr int kSlabCh = kApplyThreads * 8;    // channels per prepare CTA
constexpr int kRowChunk = 4;                  // rows loaded ahead of the arithmetic

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
// Round to the storage type and back (what a reader of the stored value sees).
__device__ __forceinline__ float stored(float v, const __nv_bfloat16*) { return __bfloat162float(__float2bfloat16_rn(v)); }
__device__ __forceinline__ float stored(float v, const float*) { return v; }
__device__ __forceinline__ void store1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void store1(float* p, float v) { *p = v; }
__device__ __forceinline__ float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float load1(const float* p) { return *p; }

// RMSNorm, one warp per row: n = x * rsqrt(mean(x^2) + eps) * w (dflash2.ts #rms).
template <typename T>
__global__ void __launch_bounds__(128) rmsnorm_kernel(const T* __restrict__ x, const T* __restrict__ w, float eps,
                                                      T* __restrict__ n, int rows, int H) {
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const T* xr = x + static_cast<size_t>(row) * H;
  float ss = 0.f;
  for (int c = lane * 8; c < H; c += 256) {
    float f[8];
    load8(xr + c, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float r = rsqrtf(ss / static_cast<float>(H) + eps);
  T* nr = n + static_cast<size_t>(row) * H;
  for (int c = lane * 8; c < H; c += 256) {
    float f[8], g[8];
    load8(xr + c, f);
    load8(w + c, g);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = f[i] * r * g[i];
    store8(nr + c, f);
  }
}

// prepare's apply pass: out = side-0 conv of n; coef1 = side 1's deltas (no base); d_full = D.
// part: [k_splits][B*G][4*groups] fp32 split-K partial sums of D, column (side*2+tap)*groups + g.
// One CTA per (block, slab of 1024 channels). The block's D values for the slab's groups are
// summed over the splits into shared memory first (coalesced along the group axis); then each
// thread walks the block's rows for its 8 channels, loading four rows ahead of the arithmetic.
template <typename T>
__global__ void __launch_bounds__(kApplyThreads)
    conv_side0_kernel(const T* __restrict__ n, const float* __restrict__ part, int k_splits,
                      const float* __restrict__ base, T* __restrict__ out, T* __restrict__ coef1,
                      float* __restrict__ d_full, int B, int G, int H, int gs, int groups) {
  extern __shared__ float sD[];  // [G][4][gsl]
  const int b = blockIdx.y;
  const int c0 = blockIdx.x * kSlabCh;
  const int cend = min(H, c0 + kSlabCh);
  const int g0 = c0 / gs;
  const int gsl = (cend - 1) / gs + 1 - g0;
  const int N = 4 * groups;
  const size_t MN = static_cast<size_t>(B) * G * N;
  const size_t row0 = static_cast<size_t>(b) * G;
  for (int i = threadIdx.x; i < G * 4 * gsl; i += kApplyThreads) {
    const int g = i % gsl;
    const int tk = i / gsl;
    const float* p = part + (row0 + (tk >> 2)) * N + (tk & 3) * groups + g0 + g;
    float acc = 0.f;
    for (int s = 0; s < k_splits; ++s) acc += __ldg(p + s * MN);
    sD[i] = acc;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * 2 * gsl; i += kApplyThreads) {
    const int g = i % gsl;
    const int tt = i / gsl;  // t*2 + tap
    store1(coef1 + (row0 * 2 + tt) * groups + g0 + g, sD[((tt >> 1) * 4 + 2 + (tt & 1)) * gsl + g]);
  }
  if (d_full != nullptr) {
    for (int i = threadIdx.x; i < G * 4 * gsl; i += kApplyThreads) {
      const int g = i % gsl;
      const int tk = i / gsl;
      d_full[(row0 + (tk >> 2)) * N + (tk & 3) * groups + g0 + g] = sD[i];
    }
  }
  const int c = c0 + threadIdx.x * 8;
  if (c >= H) return;
  const int gl = c / gs - g0;
  float b0[8], b1[8], prev[8];
  load8(base + c, b0);      // base[0][0][c..]
  load8(base + H + c, b1);  // base[0][1][c..]
#pragma unroll
  for (int i = 0; i < 8; ++i) prev[i] = 0.f;
  const T* np = n + row0 * H + c;
  T* op = out + row0 * H + c;
  for (int t0 = 0; t0 < G; t0 += kRowChunk) {
    float cur[kRowChunk][8];
#pragma unroll
    for (int j = 0; j < kRowChunk; ++j)
      if (t0 + j < G) load8(np + static_cast<size_t>(t0 + j) * H, cur[j]);
#pragma unroll
    for (int j = 0; j < kRowChunk; ++j) {
      const int t = t0 + j;
      if (t < G) {
        const float d0 = sD[(t * 4 + 0) * gsl + gl];
        const float d1 = sD[(t * 4 + 1) * gsl + gl];
        float o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          o[i] = (b0[i] + d0) * cur[j][i] + (b1[i] + d1) * prev[i];
          prev[i] = cur[j][i];
        }
        store8(op + static_cast<size_t>(t) * H, o);
      }
    }
  }
}

// finish's apply pass: out = residual + side-1 conv of y (fp32 add, one rounding); optionally
// next_n = rms(out) * next_w over rows [next_row0, G). The block's side-1 deltas for the CTA's
// groups are staged in shared memory first; rows are processed four at a time, loads first. With
// NORM the grid is one cluster per block (cluster = gridDim.x CTAs) and the per-row sums of
// squares meet through distributed shared memory.
template <typename T, bool NORM>
__global__ void __launch_bounds__(kApplyThreads)
    conv_side1_kernel(const T* __restrict__ y, const T* __restrict__ coef1, const float* __restrict__ base,
                      const T* residual, T* out, const T* __restrict__ next_w, float eps, T* __restrict__ next_n,
                      int next_row0, int G, int H, int gs, int groups) {
  extern __shared__ float sC[];  // [G][2][gsl]
  __shared__ float row_ss[64];
  __shared__ float row_r[64];
  const int b = blockIdx.y;
  const int c0 = blockIdx.x * blockDim.x * 8;
  const int cend = min(H, c0 + static_cast<int>(blockDim.x) * 8);
  const int g0 = c0 / gs;
  const int gsl = (cend - 1) / gs + 1 - g0;
  const size_t row0 = static_cast<size_t>(b) * G;
  const int c = c0 + threadIdx.x * 8;
  const bool active = c < H;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < G * 2 * gsl; i += blockDim.x) {
    const int g = i % gsl;
    const int tt = i / gsl;  // t*2 + tap
    sC[i] = load1(coef1 + (row0 * 2 + tt) * groups + g0 + g);
  }
  if (NORM)
    for (int i = threadIdx.x; i < 64; i += blockDim.x) row_ss[i] = 0.f;
  __syncthreads();
  const int gl = active ? c / gs - g0 : 0;
  float b0[8], b1[8], prev[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    b0[i] = 0.f;
    b1[i] = 0.f;
    prev[i] = 0.f;
  }
  if (active) {
    load8(base + 2 * H + c, b0);  // base[1][0][c..]
    load8(base + 3 * H + c, b1);  // base[1][1][c..]
  }
  for (int t0 = 0; t0 < G; t0 += kRowChunk) {
    float cur[kRowChunk][8], res[kRowChunk][8];
    if (active) {
#pragma unroll
      for (int j = 0; j < kRowChunk; ++j) {
        if (t0 + j < G) {
          load8(y + (row0 + t0 + j) * H + c, cur[j]);
          if (residual != nullptr) load8(residual + (row0 + t0 + j) * H + c, res[j]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kRowChunk; ++j) {
      const int t = t0 + j;
      if (t >= G) break;
      float ss = 0.f;
      if (active) {
        const float d0 = sC[(t * 2 + 0) * gsl + gl];
        const float d1 = sC[(t * 2 + 1) * gsl + gl];
        float o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          o[i] = (b0[i] + d0) * cur[j][i] + (b1[i] + d1) * prev[i];
          prev[i] = cur[j][i];
          if (residual != nullptr) o[i] += res[j][i];
        }
        store8(out + (row0 + t) * H + c, o);
        if (NORM) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float sv = stored(o[i], out);
            ss = fmaf(sv, sv, ss);
          }
        }
      }
      if (NORM && t >= next_row0) {  // every thread of the CTA takes part (inactive ones add 0)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (lane == 0) atomicAdd(&row_ss[t], ss);
      }
    }
  }
  if (!NORM) return;
  cg::cluster_group cluster = cg::this_cluster();
  __syncthreads();
  cluster.sync();
  const int ranks = static_cast<int>(cluster.num_blocks());
  for (int t = threadIdx.x; t < G; t += blockDim.x) {
    float tot = 0.f;
    for (int rk = 0; rk < ranks; ++rk) tot += cluster.map_shared_rank(row_ss, rk)[t];
    row_r[t] = rsqrtf(tot / static_cast<float>(H) + eps);
  }
  __syncthreads();
  cluster.sync();  // no CTA leaves while a peer may still read its row sums
  if (!active) return;
  float w[8];
  load8(next_w + c, w);
  const int rows_out = G - next_row0;
  for (int t0 = next_row0; t0 < G; t0 += kRowChunk) {
    float o[kRowChunk][8];
#pragma unroll
    for (int j = 0; j < kRowChunk; ++j)
      if (t0 + j < G) load8(out + (row0 + t0 + j) * H + c, o[j]);
#pragma unroll
    for (int j = 0; j < kRowChunk; ++j) {
      const int t = t0 + j;
      if (t < G) {
        const float r = row_r[t];
#pragma unroll
        for (int i = 0; i < 8; ++i) o[j][i] = o[j][i] * r * w[i];
        store8(next_n + (static_cast<size_t>(b) * rows_out + (t - next_row0)) * H + c, o[j]);
      }
    }
  }
}

// Threads per CTA and CTAs per block for the apply passes: H/8 vector lanes per block row.
void apply_geometry(int H, int* threads, int* ctas) {
  const int lanes = H / 8;
  const int n = std::max(1, (lanes + 127) / 128);
  const int per = (lanes + n - 1) / n;
  *threads = ((per + 31) / 32) * 32;
  *ctas = n;
}

}  // namespace

GemmPlan kp_plan(const ConvShape& s, int sms) {
  const int M = s.rows();
  const int N = 4 * s.groups;
  const int bk = s.dtype == DFLASH2_F32 ? 32 : 64;
  const int k_blocks = (s.H + bk - 1) / bk;
  GemmPlan p{};
  p.mt = M > 128 ? 2 : 1;
  p.m_groups = (M + 128 * p.mt - 1) / (128 * p.mt);
  p.n_chunks = (N + 63) / 64;
  const int tiles256 = (p.n_chunks + 3) / 4;
  p.n_splits = (p.m_groups * tiles256 >= std::max(1, sms / 8)) ? tiles256 : p.n_chunks;
  const int units = p.m_groups * p.n_splits;
  p.k_splits = std::max(1, std::min(std::min(k_blocks, 16), sms / std::max(1, units)));
  return p;
}

size_t conv_prepare_workspace(const ConvShape& s, int sms) {
  const GemmPlan p = kp_plan(s, sms);
  const size_t es = s.dtype == DFLASH2_F32 ? 4 : 2;
  size_t n_bytes = static_cast<size_t>(s.rows()) * s.H * es;
  n_bytes = (n_bytes + 255) & ~static_cast<size_t>(255);
  const size_t part = static_cast<size_t>(p.k_splits) * s.rows() * 4 * s.groups * sizeof(float);
  return n_bytes + part + 256;
}

int launch_rmsnorm(const void* x, const void* w, float eps, void* n, int rows, int H, int dtype, cudaStream_t st) {
  const int grid = (rows + 3) / 4;
  if (dtype == DFLASH2_F32)
    rmsnorm_kernel<float><<<grid, 128, 0, st>>>(static_cast<const float*>(x), static_cast<const float*>(w), eps,
                                                static_cast<float*>(n), rows, H);
  else
    rmsnorm_kernel<__nv_bfloat16><<<grid, 128, 0, st>>>(static_cast<const __nv_bfloat16*>(x),
                                                        static_cast<const __nv_bfloat16*>(w), eps,
                                                        static_cast<__nv_bfloat16*>(n), rows, H);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DFLASH2_OK : fail(DFLASH2_ERR_CUDA, "rmsnorm launch failed: %s", cudaGetErrorString(e));
}

// Largest number of groups one slab of `slab_ch` channels touches.
static int slab_groups(int H, int gs, int slab_ch) {
  int best = 0;
  for (int c0 = 0; c0 < H; c0 += slab_ch) {
    const int cend = std::min(H, c0 + slab_ch);
    best = std::max(best, (cend - 1) / gs + 1 - c0 / gs);
  }
  return best;
}

// Upper bound of the apply passes' dynamic shared memory: G <= 64 rows x 4 deltas x 129 groups.
constexpr int kApplySmemMax = 64 * 4 * 129 * 4;

int launch_conv_side0(const ConvShape& s, const void* n, const float* part, int k_splits, const float* base,
                      void* out, void* coef1, float* d_full, cudaStream_t st) {
  const dim3 grid((s.H + kSlabCh - 1) / kSlabCh, s.B);
  const size_t smem = sizeof(float) * s.G * 4 * slab_groups(s.H, s.gs, kSlabCh);
  static unsigned done_f32 = 0, done_bf16 = 0;
  if (s.dtype == DFLASH2_F32) {
    if (!ensure_smem_attr(conv_side0_kernel<float>, kApplySmemMax, &done_f32))
      return fail(DFLASH2_ERR_CUDA, "cudaFuncSetAttribute failed (side0)");
    conv_side0_kernel<float><<<grid, kApplyThreads, smem, st>>>(static_cast<const float*>(n), part, k_splits, base,
                                                                static_cast<float*>(out), static_cast<float*>(coef1),
                                                                d_full, s.B, s.G, s.H, s.gs, s.groups);
  } else {
    if (!ensure_smem_attr(conv_side0_kernel<__nv_bfloat16>, kApplySmemMax, &done_bf16))
      return fail(DFLASH2_ERR_CUDA, "cudaFuncSetAttribute failed (side0)");
    conv_side0_kernel<__nv_bfloat16><<<grid, kApplyThreads, smem, st>>>(
        static_cast<const __nv_bfloat16*>(n), part, k_splits, base, static_cast<__nv_bfloat16*>(out),
        static_cast<__nv_bfloat16*>(coef1), d_full, s.B, s.G, s.H, s.gs, s.groups);
  }
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DFLASH2_OK : fail(DFLASH2_ERR_CUDA, "conv side0 launch failed: %s", cudaGetErrorString(e));
}

template <typename T>
static int side1_typed(const ConvShape& s, const void* y, const void* coef1, const float* base, const void* residual,
                       void* out, const void* next_w, float eps, void* next_n, int next_row0, cudaStream_t st) {
  int threads, ctas;
  apply_geometry(s.H, &threads, &ctas);
  const dim3 grid(ctas, s.B);
  const size_t smem = sizeof(float) * s.G * 2 * slab_groups(s.H, s.gs, threads * 8);
  static unsigned done_plain = 0, done_norm = 0;
  if (!ensure_smem_attr(conv_side1_kernel<T, false>, kApplySmemMax, &done_plain) ||
      !ensure_smem_attr(conv_side1_kernel<T, true>, kApplySmemMax, &done_norm))
    return fail(DFLASH2_ERR_CUDA, "cudaFuncSetAttribute failed (side1)");
  const T* yp = static_cast<const T*>(y);
  const T* cp = static_cast<const T*>(coef1);
  const T* rp = static_cast<const T*>(residual);
  T* op = static_cast<T*>(out);
  if (next_n == nullptr) {
    conv_side1_kernel<T, false><<<grid, threads, smem, st>>>(yp, cp, base, rp, op, nullptr, eps, nullptr, 0, s.G,
                                                             s.H, s.gs, s.groups);
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, conv_side1_kernel<T, true>, yp, cp, base, rp, op,
                                             static_cast<const T*>(next_w), eps, static_cast<T*>(next_n), next_row0,
                                             s.G, s.H, s.gs, s.groups);
    if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "conv side1 (cluster) launch failed: %s", cudaGetErrorString(e));
  }
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DFLASH2_OK : fail(DFLASH2_ERR_CUDA, "conv side1 launch failed: %s", cudaGetErrorString(e));
}

int launch_conv_side1(const ConvShape& s, const void* y, const void* coef1, const float* base, const void* residual,
                      void* out, const void* next_w, float eps, void* next_n, int next_row0, cudaStream_t st) {
  if (s.dtype == DFLASH2_F32)
    return side1_typed<float>(s, y, coef1, base, residual, out, next_w, eps, next_n, next_row0, st);
  return side1_typed<__nv_bfloat16>(s, y, coef1, base, residual, out, next_w, eps, next_n, next_row0, st);
}

}  // namespace dfl
