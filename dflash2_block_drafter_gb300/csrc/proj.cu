// Sublayer projections around a conv site, on the tcgen05 tensor cores:
//
//   Y[m, n] = sum_k A[m, k] * W[n, k]        (A [M, K] bf16, W [N, K], fp32 accumulation in TMEM)
//
// with two fusions of the grouped conv and one weight format:
//   * A producer "conv side 0": A = Conv_0(n), A[m, k] = coef[m, 0, 0, k] * n[m, k] +
//     coef[m, 0, 1, k] * n[m - 1, k] (n[m - 1] = 0 at a block's first row), coef = base[0] + D0
//     broadcast over each group (MAX DFlash2TransformerBlock: prepare's output feeds the sublayer's
//     input projections; dflash2.ts #block: a = #conv(n, coef, 0) then q/k/v or gate/up of a).
//     Producer warps read the normed rows n and compute A straight into the operand tile, so the
//     side-0 output never goes through memory.
//   * epilogue "conv side 1 + residual": out = residual + Conv_1(Y) with the side-1 coefficients
//     of the same site (dflash2.ts #block: x = x + #conv(o(attn) or down(mlp), coef, 1); MAX
//     DFlash2TransformerBlock: r += conv.finish(h)). A row's previous row is in the neighbouring
//     TMEM lane (one warp shuffle): blocks of G rows with G dividing 32 never cross a warp.
//   * B producer "W4A16": affine 4-bit weights in groups of 64 along K, W[n, k] = scale[n, k/64] *
//     q[n, k] + bias[n, k/64] (dflash2.ts quantizedWeight: quantize(w, 64, bits), mode "affine"),
//     dequantised to bf16 in shared memory by producer warps; the MMA stays kind::f16.
//
// One CTA per SM, persistent over 128 x 256 output tiles (M fastest, so neighbouring CTAs share
// a weight tile in L2). K advances in 64-element stages: every operand row is one 128-byte
// swizzled row, as TMA writes it, and the producer warps write their tiles in the same layout
// (16-byte chunk c of row r at chunk position c ^ (r & 7) of the row, 1024-byte aligned tiles).
// Warp roles: 0 TMA, 1 TMEM + MMA issue (one lane), 2-5 epilogue (TMEM lanes 32 (w % 4) ..),
// then 4 conv-producer warps (one tile row per thread) and/or 4 dequant warps (two weight rows
// per thread). The accumulator is double-buffered in TMEM (2 x 256 columns). Every wait is
// bounded: a timeout raises a CTA-wide abort flag, records DFLASH2_ERR_TIMEOUT, drains the copies
// and MMAs in flight and frees TMEM before the kernel returns.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {
namespace {

constexpr int kPM = 128;                     // rows per tile
constexpr int kPN = 256;                     // columns per tile
constexpr int kPK = 64;                      // K per stage (one 128-byte bf16 row)
constexpr int kAOp = kPM * 128;              // A operand tile bytes
constexpr int kBOp = kPN * 128;              // B operand tile bytes
constexpr int kARaw = kPM * 128 + 1024;      // normed rows + side-0 base chunk (2 x 64 fp32), padded
constexpr int kBRaw = kPN * 32;              // 64 packed 4-bit values per weight row
constexpr int kQGroup = 64;                  // quantisation group along K
constexpr uint64_t kPDrainNs = 100000000ull; // 100 ms
constexpr int kPSmemLimit = 232448;

template <int AM, int BM, int EM>
struct PCfg {
  static constexpr int kProdWarps = (AM ? 4 : 0) + (BM ? 4 : 0);
  static constexpr int kThreads = 64 + 128 + 32 * kProdWarps;
  static constexpr int kStageBytes = kAOp + kBOp + (AM ? kARaw : 0) + (BM ? kBRaw : 0);
  static constexpr int kBarBytes = 256;
  static constexpr int kFit = (kPSmemLimit - 1024 - kBarBytes) / kStageBytes;
  static constexpr int kStages = kFit > 6 ? 6 : kFit;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes;
};

struct ProjArgs {
  int M, N, K;
  int tiles_m, tiles_n;
  int G, gs, groups;           // conv shape (G rows per block, group size, H / group size)
  const float* d0;             // AM: side-0 deltas [M][2][groups] fp32
  const __nv_bfloat16* coef1;  // EM: side-1 deltas [M][2][groups] bf16
  const float* base;           // [2][2][H] fp32 (AM: side 0 over K; EM: side 1 over N)
  const __nv_bfloat16* residual;  // EM: [M][N] or null
  const __nv_bfloat16* scales;    // BM: [N][K / 64]
  const __nv_bfloat16* qbias;     // BM: [N][K / 64]
  __nv_bfloat16* out;          // [M][N]
  int* err;
};

__device__ __forceinline__ void p_abort(volatile int* abort_flag, int* err) {
  *abort_flag = 1;
  if (err != nullptr) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_TIMEOUT));
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ int sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}
__device__ __forceinline__ uint4 f32x8_to_bf16(const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

template <int AM, int BM, int EM>
__global__ void __launch_bounds__(PCfg<AM, BM, EM>::kThreads, 1)
    proj_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmBase, const ProjArgs a) {
  using C = PCfg<AM, BM, EM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* bar_area = smem + C::kStages * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(bar_area);  // TMA bytes landed
  uint64_t* ready = full + C::kStages;                     // producer warps done (AM / BM)
  uint64_t* empty = ready + C::kStages;                    // MMAs done reading the stage
  uint64_t* acc_full = empty + C::kStages;                 // [2]
  uint64_t* acc_empty = acc_full + 2;                      // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int k_stages = a.K / kPK;
  const int n_tiles = a.tiles_m * a.tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&ready[s]), C::kProdWarps > 0 ? C::kProdWarps : 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 4);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (AM) prefetch_tmap(&tmBase);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();
  pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_last();   // activations: re-read by every column tile
      const uint64_t pol_w = policy_evict_normal(); // weights: shared by the CTAs of one column tile
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        const int m0 = (t % a.tiles_m) * kPM;
        const int n0 = (t / a.tiles_m) * kPN;
        for (int kb = 0; kb < k_stages; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          uint8_t* st = smem + stage * C::kStageBytes;
          uint8_t* a_dst = AM ? st + kAOp + kBOp : st;                             // raw rows or the operand
          uint8_t* b_dst = BM ? st + kAOp + kBOp + (AM ? kARaw : 0) : st + kAOp;  // packed or the operand
          mbar_arrive_expect_tx(fb, static_cast<uint32_t>(kPM * 128 + (AM ? 2 * kPK * 4 : 0) + (BM ? kBRaw : kBOp)));
          tma_load_2d(smem_u32(a_dst), &tmA, fb, kb * kPK, m0, pol_a);
          if (AM) tma_load_2d(smem_u32(a_dst + kPM * 128), &tmBase, fb, kb * kPK, 0, pol_a);
          tma_load_2d(smem_u32(b_dst), &tmB, fb, BM ? kb * (kPK / 8) : kb * kPK, n0, pol_w);
          ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        p_abort(abort_flag, a.err);
        int s = stage;
        uint32_t ph = phase;
        const int n = min(issued, C::kStages);
        for (int i = 0; i < n; ++i) {  // the copies still in flight land before the CTA exits
          if (s == 0) {
            s = C::kStages - 1;
            ph ^= 1u;
          } else {
            --s;
          }
          mbar_wait_bounded(smem_u32(&full[s]), ph, nullptr, kPDrainNs);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, tile_i = 0;
      uint32_t phase = 0;
      bool ok = true, any = false;
      const uint32_t idesc = make_idesc(false, kPM, kPN);
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++tile_i) {
        const int ab = tile_i & 1;
        const uint32_t acc_par = static_cast<uint32_t>(tile_i >> 1) & 1u;
        if (!mbar_wait_bounded(smem_u32(&acc_empty[ab]), acc_par ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < k_stages; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs) ||
              (C::kProdWarps > 0 && !mbar_wait_bounded(smem_u32(&ready[stage]), phase, abort_flag, kWaitLimitNs))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
          const uint64_t adesc = desc_kmajor_swizzled<128>(sa);
          const uint64_t bdesc = desc_kmajor_swizzled<128>(sa + kAOp);
#pragma unroll
          for (int k = 0; k < 4; ++k)  // 16-element (32-byte) steps along the swizzled row
            mma_f16(tmem_base + static_cast<uint32_t>(ab * kPN), adesc + static_cast<uint64_t>(2 * k),
                    bdesc + static_cast<uint64_t>(2 * k), idesc, (kb > 0 || k > 0) ? 1u : 0u);
          mma_commit(smem_u32(&empty[stage]));
          any = true;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&acc_full[ab]));
      }
      if (!ok) {
        p_abort(abort_flag, a.err);
        if (any) {
          mma_commit(smem_u32(drain));
          mbar_wait_bounded(smem_u32(drain), 0, nullptr, kPDrainNs);
        }
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lanes 32q .. 32q + 31
    int tile_i = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tile_i) {
      const int m0 = (t % a.tiles_m) * kPM;
      const int n0 = (t / a.tiles_m) * kPN;
      const int row = m0 + q * 32 + lane;
      const bool valid = row < a.M;
      const int ab = tile_i & 1;
      const uint32_t acc_par = static_cast<uint32_t>(tile_i >> 1) & 1u;
      if (!mbar_wait_bounded(smem_u32(&acc_full[ab]), acc_par, abort_flag, kWaitLimitNs)) {
        if (lane == 0) p_abort(abort_flag, a.err);
        break;
      }
      tc_fence_after();
      const int trow = row % a.G;  // EM: the row's position in its block
      for (int cc = 0; cc < kPN / 32; ++cc) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(ab * kPN + cc * 32),
                           r);
        tmem_ld_wait();
        const int col0 = n0 + cc * 32;
        float y[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(r[j]);
        if (EM) {
          // x = residual + (b10 + d10) * y[m] + (b11 + d11) * y[m - 1]; y[m - 1] is lane - 1's value
          // (lane 0's row 32w starts a block, as G divides 32)
          float d[2][32 / 8];
          const int gpc = 32 / a.gs;  // groups in these 32 columns (gs >= 8)
#pragma unroll
          for (int tap = 0; tap < 2; ++tap)
#pragma unroll
            for (int gi = 0; gi < 4; ++gi)
              d[tap][gi] = (valid && gi < gpc)
                               ? __bfloat162float(a.coef1[(static_cast<size_t>(row) * 2 + tap) * a.groups +
                                                          col0 / a.gs + gi])
                               : 0.f;
          // side 1's base kernel of these columns (the same for every lane: broadcast loads)
          float b1[2][32];
#pragma unroll
          for (int tap = 0; tap < 2; ++tap)
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const float4 f4 = col0 + 4 * v < a.N
                                    ? __ldg(reinterpret_cast<const float4*>(a.base + (2 + tap) * static_cast<size_t>(a.N) +
                                                                            col0 + 4 * v))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
              b1[tap][4 * v] = f4.x;
              b1[tap][4 * v + 1] = f4.y;
              b1[tap][4 * v + 2] = f4.z;
              b1[tap][4 * v + 3] = f4.w;
            }
          float res[32];
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float f[8];
            if (valid && a.residual != nullptr && col0 + 8 * v < a.N) {
              bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(a.residual + static_cast<size_t>(row) * a.N +
                                                                 col0 + 8 * v)),
                            f);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) res[8 * v + e] = f[e];
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float yp = __shfl_up_sync(0xffffffffu, y[j], 1);
            if (lane == 0 || trow == 0) yp = 0.f;
            const int gi = j / a.gs;
            const float c0 = b1[0][j] + d[0][gi];
            const float c1 = b1[1][j] + d[1][gi];
            y[j] = res[j] + (c0 * y[j] + c1 * yp);
          }
        }
        if (valid) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            if (col0 + 8 * v < a.N) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = y[8 * v + e];
              *reinterpret_cast<uint4*>(a.out + static_cast<size_t>(row) * a.N + col0 + 8 * v) = f32x8_to_bf16(f);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
    }
  } else if (AM && warp < 10) {
    // ------------------------------------------------------------------ conv side-0 producer
    // Thread r owns tile row r: A[r, k] = (b00[k] + d00) n[r, k] + (b01[k] + d01) n[r - 1, k].
    const int r = threadIdx.x - 192;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
      const int m0 = (t % a.tiles_m) * kPM;
      const int row = m0 + r;
      const bool first = (row % a.G) == 0 || row >= a.M;
      for (int kb = 0; kb < k_stages; ++kb) {
        // this row's side-0 deltas of the stage's groups (at most 8: gs >= 8)
        const int gpc = kPK / a.gs;
        float d0[2][8];
#pragma unroll
        for (int tap = 0; tap < 2; ++tap)
#pragma unroll
          for (int gi = 0; gi < 8; ++gi)
            d0[tap][gi] = (row < a.M && gi < gpc)
                              ? __ldg(a.d0 + (static_cast<size_t>(row) * 2 + tap) * a.groups + kb * gpc + gi)
                              : 0.f;
        if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + stage * C::kStageBytes;
        const uint8_t* raw = st + kAOp + kBOp;
        const float* b0 = reinterpret_cast<const float*>(raw + kPM * 128);  // [2][64]
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float cur[8], prv[8], o[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(raw + sw128(r, c)), cur);
          if (!first) {
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(raw + sw128(r - 1, c)), prv);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) prv[e] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int k = 8 * c + e;
            const int gi = k / a.gs;
            o[e] = (b0[k] + d0[0][gi]) * cur[e] + (b0[kPK + k] + d0[1][gi]) * prv[e];
          }
          *reinterpret_cast<uint4*>(st + sw128(r, c)) = f32x8_to_bf16(o);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ready[stage]));
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) p_abort(abort_flag, a.err);
  } else if (BM) {
    // ------------------------------------------------------------------ W4A16 dequant producer
    // Thread i owns weight rows i and i + 128 of the tile: W = scale * q + bias in bf16 (one
    // rounding of the exact value), written as swizzled 128-byte rows of the B operand.
    const int i = threadIdx.x - 192 - (AM ? 128 : 0);
    const int kq = a.K / kQGroup;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
      const int n0 = (t / a.tiles_m) * kPN;
      for (int kb = 0; kb < k_stages; ++kb) {
        __nv_bfloat162 sc2[2], bi2[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = n0 + i + 128 * h;
          const __nv_bfloat16 s = n < a.N ? a.scales[static_cast<size_t>(n) * kq + kb] : __float2bfloat16(0.f);
          const __nv_bfloat16 b = n < a.N ? a.qbias[static_cast<size_t>(n) * kq + kb] : __float2bfloat16(0.f);
          sc2[h] = __halves2bfloat162(s, s);
          bi2[h] = __halves2bfloat162(b, b);
        }
        if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + stage * C::kStageBytes;
        const uint8_t* raw = st + kAOp + kBOp + (AM ? kARaw : 0);
        const __nv_bfloat162 k128 = __floats2bfloat162_rn(128.f, 128.f);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int rr = i + 128 * h;
          const uint4 p0 = *reinterpret_cast<const uint4*>(raw + rr * 32);
          const uint4 p1 = *reinterpret_cast<const uint4*>(raw + rr * 32 + 16);
          const uint32_t words[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // word c holds k = 8c .. 8c + 7, nibble j = k - 8c
            const uint32_t w = words[c];
            uint32_t o[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              // bf16 pair (128 + q[2jj], 128 + q[2jj + 1]): 0x4300 | nibble is 128 + nibble exactly
              const uint32_t lo = (w >> (8 * jj)) & 0xFu;
              const uint32_t hi = (w >> (8 * jj + 4)) & 0xFu;
              const uint32_t pair = 0x43004300u | lo | (hi << 16);
              __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&pair);
              v = __hsub2(v, k128);              // exact: q
              v = __hfma2(sc2[h], v, bi2[h]);    // scale * q + bias, one rounding
              o[jj] = *reinterpret_cast<const uint32_t*>(&v);
            }
            *reinterpret_cast<uint4*>(st + kAOp + sw128(rr, c)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ready[stage]));
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) p_abort(abort_flag, a.err);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// Sums the split-K partial sums of kernel_projection into the side-0 deltas (fp32) and the side-1
// deltas (activation dtype) of every row: D[m, side, tap, g] = sum_s part[s][m][(side*2+tap)*groups + g].
template <typename T>
__global__ void __launch_bounds__(256)
    conv_coef_kernel(const float* __restrict__ part, int k_splits, int M, int groups, float* __restrict__ d0,
                     T* __restrict__ coef1) {
  pdl_trigger();
  pdl_wait();
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // (row, group)
  if (i >= static_cast<size_t>(M) * groups) return;
  const size_t m = i / groups;
  const int g = static_cast<int>(i % groups);
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < k_splits; ++s) {
    const float* p = part + (static_cast<size_t>(s) * M + m) * 4 * groups + g;
#pragma unroll
    for (int c = 0; c < 4; ++c) d[c] += p[c * groups];
  }
  d0[(m * 2 + 0) * groups + g] = d[0];
  d0[(m * 2 + 1) * groups + g] = d[1];
  if (sizeof(T) == 2) {
    reinterpret_cast<__nv_bfloat16*>(coef1)[(m * 2 + 0) * groups + g] = __float2bfloat16_rn(d[2]);
    reinterpret_cast<__nv_bfloat16*>(coef1)[(m * 2 + 1) * groups + g] = __float2bfloat16_rn(d[3]);
  } else {
    reinterpret_cast<float*>(coef1)[(m * 2 + 0) * groups + g] = d[2];
    reinterpret_cast<float*>(coef1)[(m * 2 + 1) * groups + g] = d[3];
  }
}

}  // namespace

template <int AM, int BM, int EM>
static int launch_proj_t(const ProjSpec& p, cudaStream_t st) {
  using C = PCfg<AM, BM, EM>;
  static_assert(C::kStages >= 2, "at least two pipeline stages");
  CUtensorMap mA, mB, mBase;
  if (!make_tmap_sw128(&mA, p.a, static_cast<uint64_t>(p.M), static_cast<uint64_t>(p.K), kPM))
    return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (projection A)");
  if (BM) {
    // packed weights [N][K / 8] 32-bit words, a box of 8 words (64 values) x 256 rows
    const uint64_t dims[2] = {static_cast<uint64_t>(p.K / 8), static_cast<uint64_t>(p.N)};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.K / 8) * 4};
    const uint32_t box[2] = {8, static_cast<uint32_t>(kPN)};
    if (!make_tmap_plain(&mB, p.w, DFLASH2_F32, 2, dims, strides, box))
      return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (packed weights)");
  } else if (!make_tmap_sw128(&mB, p.w, static_cast<uint64_t>(p.N), static_cast<uint64_t>(p.K), kPN)) {
    return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (projection W)");
  }
  if (AM) {
    // base [2][2][K] fp32 as [4][K]: rows 0, 1 are side 0's taps; a box of 64 channels x 2 rows
    const uint64_t dims[2] = {static_cast<uint64_t>(p.K), 4};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.K) * 4};
    const uint32_t box[2] = {static_cast<uint32_t>(kPK), 2};
    if (!make_tmap_plain(&mBase, p.base, DFLASH2_F32, 2, dims, strides, box))
      return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (base kernel)");
  } else {
    mBase = mA;
  }
  ProjArgs args{};
  args.M = p.M;
  args.N = p.N;
  args.K = p.K;
  args.tiles_m = (p.M + kPM - 1) / kPM;
  args.tiles_n = (p.N + kPN - 1) / kPN;
  args.G = p.G > 0 ? p.G : 1;
  args.gs = p.gs > 0 ? p.gs : 8;
  args.groups = p.groups;
  args.d0 = p.d0;
  args.coef1 = static_cast<const __nv_bfloat16*>(p.coef1);
  args.base = p.base;
  args.residual = static_cast<const __nv_bfloat16*>(p.residual);
  args.scales = static_cast<const __nv_bfloat16*>(p.scales);
  args.qbias = static_cast<const __nv_bfloat16*>(p.qbias);
  args.out = static_cast<__nv_bfloat16*>(p.out);
  args.err = device_error_word();
  const int tiles = args.tiles_m * args.tiles_n;
  const int grid = std::min(tiles, sm_count());
  static unsigned done = 0;
  auto kern = proj_kernel<AM, BM, EM>;
  if (!ensure_smem_attr(kern, C::kSmem, &done))
    return fail(DFLASH2_ERR_CUDA, "cudaFuncSetAttribute failed (projection)");
  const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmem, st, nullptr, 0, mA, mB, mBase, args);
  return e == cudaSuccess ? DFLASH2_OK : fail(DFLASH2_ERR_CUDA, "projection launch failed: %s", cudaGetErrorString(e));
}

int launch_proj(const ProjSpec& p, cudaStream_t st) {
  const bool am = p.d0 != nullptr, bm = p.wbits == 4, em = p.coef1 != nullptr;
  if (am && bm && em) return launch_proj_t<1, 1, 1>(p, st);
  if (am && bm) return launch_proj_t<1, 1, 0>(p, st);
  if (am && em) return launch_proj_t<1, 0, 1>(p, st);
  if (bm && em) return launch_proj_t<0, 1, 1>(p, st);
  if (am) return launch_proj_t<1, 0, 0>(p, st);
  if (bm) return launch_proj_t<0, 1, 0>(p, st);
  if (em) return launch_proj_t<0, 0, 1>(p, st);
  return launch_proj_t<0, 0, 0>(p, st);
}

int launch_conv_coefficients(const float* part, int k_splits, int M, int groups, int dtype, float* d0, void* coef1,
                             cudaStream_t st) {
  const size_t n = static_cast<size_t>(M) * groups;
  const dim3 grid(static_cast<unsigned>((n + 255) / 256));
  const cudaError_t e =
      dtype == DFLASH2_F32
          ? launch_pdl(conv_coef_kernel<float>, grid, dim3(256), 0, st, nullptr, 0, part, k_splits, M, groups, d0,
                       static_cast<float*>(coef1))
          : launch_pdl(conv_coef_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, nullptr, 0, part, k_splits, M, groups,
                       d0, static_cast<__nv_bfloat16*>(coef1));
  return e == cudaSuccess ? DFLASH2_OK
                          : fail(DFLASH2_ERR_CUDA, "conv coefficient launch failed: %s", cudaGetErrorString(e));
}

}  // namespace dfl
