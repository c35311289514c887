// Sublayer projections for a few rows (M <= 128), with the same fusions as proj_kernel:
//
//   Y[m, n] = sum_k A[m, k] W[n, k]      (A [M, K] bf16; W [N, K] bf16 or affine 4-bit)
//
//   * "conv side 0" in the activation operand: A = Conv_0(n) (MAX DFlash2TransformerBlock:
//     prepare's output feeds the sublayer's input projections; dflash2.ts #block);
//   * "conv side 1 + residual" on the output: out = residual + Conv_1(Y) (dflash2.ts #block:
//     x = x + #conv(o(attn) or down(mlp), coef, 1));
//   * "W4A16": W[n, k] = scale[k / 64][n] q[n, k] + bias[k / 64][n] (dflash2.ts quantizedWeight,
//     groups of 64, mode "affine"), dequantised to bf16 in shared memory.
//
// With few rows a projection is a weight stream, so the operands are swapped: a tile's 128 weight
// rows are the tcgen05 MMA's M = 128 side and the activation rows its N side (16 .. 128), and the
// accumulator is one 128 x N fp32 tile in TMEM. K is split over the ks CTAs of a thread-block
// cluster. Each CTA stages its partial tile as P[weight row][activation row] in shared memory; CTA
// r owns a slice of the tile's weight rows (8-row chunks) and receives the other CTAs' partial rows
// of that slice by bulk copies into its shared memory (counted on an mbarrier of r). The owner adds
// the ks partials in K order and writes its output columns for every activation row, so the side-1
// conv's previous row is its own data.
//
// Warp roles: 0 TMA (one lane), 1 TMEM + MMA issue (one lane), 2-5 accumulator -> shared memory,
// then 8 conv warps (AM: side 0 applied in place to the staged rows) and/or 8 dequant warps (BM).
// All warps reduce. Every mbarrier wait is bounded; a CTA whose wait ran out records
// DFLASH2_ERR_TIMEOUT, still takes part in the cluster barriers and sends its partial, and writes
// no output.
#include <cuda_bf16.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {
namespace {

constexpr int kQK = 64;               // K per stage
constexpr int kQWBytes = 128 * 128;   // the weight operand: 128 rows of 128 bytes
constexpr int kQMaxRows = 128;        // activation rows (the MMA's N side) at most
constexpr int kQMaxSplits = 8;
constexpr int kQMaxStages = 8;
constexpr int kQChunks = 16;          // 8-row chunks of a tile's weight rows, dealt to the owners
constexpr int kQSmemLimit = 232448;
constexpr int kQBarBytes = 256;
constexpr int kQMinSmem = 64 * 1024;  // at most three CTAs per SM: their TMEM (<= 128 columns) always fits
constexpr uint64_t kQDrainNs = 100000000ull;

template <int AM, int BM>
struct QCfg {
  static constexpr int kConvWarps = AM ? 8 : 0;
  static constexpr int kDeqWarps = BM ? 8 : 0;
  static constexpr int kProdWarps = kConvWarps + kDeqWarps;
  static constexpr int kThreads = 192 + 32 * kProdWarps;
};

struct QArgs {
  int M, N, K, G, gs, groups;
  int k_blocks, ks, np, stride, n_stages, stage_bytes, r_off, region, maxrows;
  // a stage holds kpb k-blocks of 64: [A sub-tiles 16 KB each][B sub-tiles np x 128 B each]
  // (AM: [base 2 x 64 kpb fp32][d0 2 x 4 kpb x np fp32]) (BM: [codes 128 x 8 kpb words][scales kpb x 128][biases])
  int kpb, off_b, off_base, off_d0, off_raw, off_sc, off_bi;
  const __nv_bfloat16* coef1;     // EM: [M][2][groups]
  const float* base;              // EM: [2][2][N] (side 1 used)
  const __nv_bfloat16* residual;  // EM: [M][N] or null
  __nv_bfloat16* out;             // [M][N]
  int* err;
};

struct QMaps {
  CUtensorMap w, a, scales, biases, base, d0;
};

__device__ __forceinline__ void q_abort(volatile int* abort_flag, int* err) {
  *abort_flag = 1;
  if (err != nullptr) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_TIMEOUT));
}

__device__ __forceinline__ int q_sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// The weight rows [w0, w1) of a tile that CTA `r` of a cluster of ks owns.
__device__ __forceinline__ int q_chunk_begin(int r, int ks) { return 8 * (kQChunks * r / ks); }

template <int AM, int BM, int EM>
__global__ void __launch_bounds__(QCfg<AM, BM>::kThreads, 1)
    proj_small_kernel(const __grid_constant__ QMaps maps, const QArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.region);
  uint64_t* ready = full + a.n_stages;
  uint64_t* empty = ready + a.n_stages;
  uint64_t* acc_full = empty + a.n_stages;
  uint64_t* recv = acc_full + 1;
  uint64_t* drain = recv + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int n0 = (static_cast<int>(blockIdx.x) / a.ks) * 128;  // the tile's first weight row
  // this CTA's k-blocks [kb_begin, kb_end) (the split is in k-blocks whatever kpb is, so that every
  // weight format sums the same partials in the same order), kpb per stage, the last stage partial
  const int kb_begin = a.k_blocks * rank / a.ks;
  const int kb_end = a.k_blocks * (rank + 1) / a.ks;
  const int nst = (kb_end - kb_begin + a.kpb - 1) / a.kpb;
  const int S = a.stride;
  const int w0 = q_chunk_begin(rank, a.ks), w1 = q_chunk_begin(rank + 1, a.ks);  // owned weight rows
  const int np = a.np;
  const uint32_t tmem_cols = np <= 32 ? 32u : (np <= 64 ? 64u : 128u);
  constexpr int kProd = QCfg<AM, BM>::kProdWarps;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.n_stages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&ready[s]), kProd > 0 ? kProd : 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(recv), 1);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
    mbar_arrive_expect_tx(smem_u32(recv), static_cast<uint32_t>((a.ks - 1) * (w1 - w0) * S * 4));
    prefetch_tmap(&maps.w);
    prefetch_tmap(&maps.a);
    if (BM) {
      prefetch_tmap(&maps.scales);
      prefetch_tmap(&maps.biases);
    }
    if (AM) {
      prefetch_tmap(&maps.base);
      prefetch_tmap(&maps.d0);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  cluster_arrive_relaxed();
  pdl_trigger();
  if (threadIdx.x != 0) pdl_wait();  // the producer waits after requesting the first weight tiles

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();  // each weight row is read by one cluster
      const uint64_t pol_a = policy_evict_last();   // the activations are read by every tile
      const int kpb = a.kpb;
      // bytes of stage i: the 4-bit boxes, base and d0 always span kpb k-blocks (zero fill past K)
      auto stage_tx = [&](int nsub) {
        return static_cast<uint32_t>((BM ? kpb * (128 * 32 + 2 * 128 * 2) : nsub * kQWBytes) + nsub * np * 128 +
                                     (AM ? kpb * (2 * kQK * 4 + 2 * 4 * np * 4) : 0));
      };
      auto load_w = [&](int i, uint32_t fb, uint8_t* st) {
        const int kb = kb_begin + i * kpb;  // the stage's first k-block
        const int nsub = min(kpb, kb_end - kb);
        if (BM) {
          // 8 kpb code words (128 bytes at kpb = 4) of each of the 128 rows in one box
          tma_load_2d(smem_u32(st + a.off_raw), &maps.w, fb, kb * (kQK / 8), n0, pol_w);
          tma_load_2d(smem_u32(st + a.off_sc), &maps.scales, fb, n0, kb, pol_w);
          tma_load_2d(smem_u32(st + a.off_bi), &maps.biases, fb, n0, kb, pol_w);
        } else {
          for (int sb = 0; sb < nsub; ++sb)
            tma_load_2d(smem_u32(st + sb * kQWBytes), &maps.w, fb, (kb + sb) * kQK, n0, pol_w);
        }
      };
      const int pre = min(nst, a.n_stages);
      for (int i = 0; i < pre; ++i) {  // weights are never written by the kernels this launch overlaps
        const uint32_t fb = smem_u32(&full[i]);
        mbar_arrive_expect_tx(fb, stage_tx(min(kpb, kb_end - kb_begin - i * kpb)));
        load_w(i, fb, smem + i * a.stage_bytes);
      }
      pdl_wait();
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < nst; ++i) {
        const int stage = i % a.n_stages;
        const uint32_t phase = static_cast<uint32_t>(i / a.n_stages) & 1u;
        const uint32_t fb = smem_u32(&full[stage]);
        uint8_t* st = smem + stage * a.stage_bytes;
        if (i >= pre) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(fb, stage_tx(min(kpb, kb_end - kb_begin - i * kpb)));
          load_w(i, fb, st);
        }
        const int kb = kb_begin + i * kpb;
        for (int sb = 0; sb < min(kpb, kb_end - kb); ++sb)
          tma_load_2d(smem_u32(st + a.off_b + sb * np * 128), &maps.a, fb, (kb + sb) * kQK, 0, pol_a);
        if (AM) {
          tma_load_2d(smem_u32(st + a.off_base), &maps.base, fb, kb * kQK, 0, pol_a);
          tma_load_3d(smem_u32(st + a.off_d0), &maps.d0, fb, 0, kb * (kQK / 16), 0, pol_a);
        }
        issued = i + 1;
      }
      if (!ok) {
        q_abort(abort_flag, a.err);
        for (int i = max(0, issued - a.n_stages); i < issued; ++i)
          mbar_wait_bounded(smem_u32(&full[i % a.n_stages]), static_cast<uint32_t>(i / a.n_stages) & 1u, nullptr,
                            kQDrainNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc(false, 128, np);
      bool ok = true, any = false;
      for (int i = 0; i < nst; ++i) {
        const int stage = i % a.n_stages;
        const uint32_t phase = static_cast<uint32_t>(i / a.n_stages) & 1u;
        if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs) ||
            (kProd > 0 && !mbar_wait_bounded(smem_u32(&ready[stage]), phase, abort_flag, kWaitLimitNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * a.stage_bytes);
        const int nsub = min(a.kpb, kb_end - kb_begin - i * a.kpb);
        for (int sb = 0; sb < nsub; ++sb) {
          const uint64_t adesc = desc_kmajor_swizzled<128>(sa + sb * kQWBytes);
          const uint64_t bdesc = desc_kmajor_swizzled<128>(sa + a.off_b + sb * np * 128);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f16(tmem, adesc + static_cast<uint64_t>(2 * k), bdesc + static_cast<uint64_t>(2 * k), idesc,
                    (i > 0 || sb > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&empty[stage]));
        any = true;
      }
      if (ok) {
        mma_commit(smem_u32(acc_full));
      } else {
        q_abort(abort_flag, a.err);
        if (any) {
          mma_commit(smem_u32(drain));
          mbar_wait_bounded(smem_u32(drain), 0, nullptr, kQDrainNs);
        }
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------------ accumulator -> shared memory
    // TMEM lane w = weight row w of the tile, one column per activation row: P[w][m] (the ring is
    // idle once the accumulator is complete).
    const int p = warp & 3;
    if (mbar_wait_bounded(smem_u32(acc_full), 0, abort_flag, kWaitLimitNs)) {
      tc_fence_after();
      float* prow = reinterpret_cast<float*>(smem) + (32 * p + lane) * S;
      for (int cc = 0; cc * 32 < np; ++cc) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * p) << 16) + static_cast<uint32_t>(cc * 32), r);
        tmem_ld_wait();
#pragma unroll
        for (int v = 0; v < 8; ++v)
          if (cc * 32 + 4 * v < np)
            *reinterpret_cast<float4*>(prow + cc * 32 + 4 * v) =
                make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]), __uint_as_float(r[4 * v + 2]),
                            __uint_as_float(r[4 * v + 3]));
      }
      fence_proxy_async_smem();  // the bulk copies below read these rows
    } else if (lane == 0) {
      q_abort(abort_flag, a.err);
    }
    __syncwarp();
  } else if (AM && warp < 6 + QCfg<AM, BM>::kConvWarps) {
    // ------------------------------------------------------------------ conv side-0 producer
    // Thread (rg, c) owns 16-byte chunk c (8 channels of one 16-channel group) of the staged rows
    // rg * rpt .. rg * rpt + rpt - 1 of every sub-tile, turned in place into
    //   A[r, k] = (b00[k] + d00[r]) n[r, k] + (b01[k] + d01[r]) n[r - 1, k]   (n[r - 1] = 0 at a block start)
    // in the arithmetic of proj_kernel's producer. The row before a thread's first row belongs to
    // another thread: every thread reads its rows before the conv warps' barrier, writes after it.
    constexpr int kConvThreads = QCfg<AM, BM>::kConvWarps > 0 ? 32 * QCfg<AM, BM>::kConvWarps : 32;
    const int pt = threadIdx.x - 192;
    const int c = pt & 7;
    const int rg = pt >> 3;
    const int rpt = (np + kConvThreads / 8 - 1) / (kConvThreads / 8);  // rows per thread (<= 4)
    const int r_first = rg * rpt;
    const int nr = max(0, min(rpt, a.M - r_first));
    const int gi = c >> 1;
    const int t_first = r_first % a.G;
    const int kpb = a.kpb;
    bool ok = true;
    for (int i = 0; i < nst; ++i) {
      const int stage = i % a.n_stages;
      const uint32_t phase = static_cast<uint32_t>(i / a.n_stages) & 1u;
      if (!mbar_wait_bounded_suspend(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs, 200)) {
        ok = false;
        break;
      }
      uint8_t* st = smem + stage * a.stage_bytes;
      const float* b0 = reinterpret_cast<const float*>(st + a.off_base);  // [2][64 kpb]
      const float* d0s = reinterpret_cast<const float*>(st + a.off_d0);   // [2][4 kpb][np]
      const int nsub = min(kpb, kb_end - kb_begin - i * kpb);
      for (int sb_i = 0; sb_i < nsub; ++sb_i) {
        uint8_t* sb = st + a.off_b + sb_i * np * 128;
        uint4 raw[5];  // raw[0]: the row before the first; raw[1 + j]: row r_first + j
        raw[0] = (nr > 0 && t_first != 0) ? *reinterpret_cast<const uint4*>(sb + q_sw128(r_first - 1, c))
                                          : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          raw[1 + j] = j < nr ? *reinterpret_cast<const uint4*>(sb + q_sw128(r_first + j, c))
                              : make_uint4(0u, 0u, 0u, 0u);
        asm volatile("bar.sync 1, %0;" ::"n"(kConvThreads) : "memory");  // all reads before any write
        if (nr > 0) {
          const float* bs = b0 + sb_i * kQK;
          const float4 x0 = *reinterpret_cast<const float4*>(bs + 8 * c);
          const float4 x1 = *reinterpret_cast<const float4*>(bs + 8 * c + 4);
          const float4 y0 = *reinterpret_cast<const float4*>(bs + kQK * kpb + 8 * c);
          const float4 y1 = *reinterpret_cast<const float4*>(bs + kQK * kpb + 8 * c + 4);
          const float2 k0[4] = {make_float2(x0.x, x0.y), make_float2(x0.z, x0.w), make_float2(x1.x, x1.y),
                                make_float2(x1.z, x1.w)};
          const float2 k1[4] = {make_float2(y0.x, y0.y), make_float2(y0.z, y0.w), make_float2(y1.x, y1.y),
                                make_float2(y1.z, y1.w)};
          const float* dt0 = d0s + (4 * sb_i + gi) * np;            // tap 0 of the chunk's group
          const float* dt1 = d0s + (4 * kpb + 4 * sb_i + gi) * np;  // tap 1
          int trow = t_first;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (j < nr) {
              const float dd0 = dt0[r_first + j];
              const float dd1 = dt1[r_first + j];
              const __nv_bfloat162* hc = reinterpret_cast<const __nv_bfloat162*>(&raw[1 + j]);
              const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
              const float2 d0p = make_float2(dd0, dd0), d1p = make_float2(dd1, dd1);
              const float2 keep = trow == 0 ? make_float2(0.f, 0.f) : make_float2(1.f, 1.f);
              uint4 o;
              __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 cur = __bfloat1622float2(hc[e]);
                const float2 prv = __fmul2_rn(__bfloat1622float2(hp[e]), keep);
                const float2 v = __ffma2_rn(__fadd2_rn(k0[e], d0p), cur, __fmul2_rn(__fadd2_rn(k1[e], d1p), prv));
                oh[e] = __floats2bfloat162_rn(v.x, v.y);
              }
              *reinterpret_cast<uint4*>(sb + q_sw128(r_first + j, c)) = o;
              if (++trow == a.G) trow = 0;
            }
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ready[stage]));
    }
    if (!ok && lane == 0) q_abort(abort_flag, a.err);
  } else if (BM) {
    // ------------------------------------------------------------------ W4A16 dequant producer
    // Job (row, word c): the 8 codes of word c of a weight row become 8 bf16 values scale * q + bias
    // (one rounding of the exact value), a 16-byte chunk of sub-tile c / 8 of the weight operand.
    constexpr int kDeqThreads = QCfg<AM, BM>::kDeqWarps > 0 ? 32 * QCfg<AM, BM>::kDeqWarps : 32;
    const int pt = threadIdx.x - 192 - 32 * QCfg<AM, BM>::kConvWarps;
    const int wpr = 8 * a.kpb;  // code words per row in a stage
    const int lg_wpr = 31 - __clz(wpr);
    const int n_jobs = 128 * wpr;
    const __nv_bfloat162 k128 = __floats2bfloat162_rn(128.f, 128.f);
    bool ok = true;
    for (int i = 0; i < nst; ++i) {
      const int stage = i % a.n_stages;
      const uint32_t phase = static_cast<uint32_t>(i / a.n_stages) & 1u;
      if (!mbar_wait_bounded_suspend(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs, 200)) {
        ok = false;
        break;
      }
      uint8_t* st = smem + stage * a.stage_bytes;
      const uint32_t* words = reinterpret_cast<const uint32_t*>(st + a.off_raw);  // [128][8 kpb]
      const __nv_bfloat16* sc = reinterpret_cast<const __nv_bfloat16*>(st + a.off_sc);  // [kpb][128]
      const __nv_bfloat16* bi = reinterpret_cast<const __nv_bfloat16*>(st + a.off_bi);
      for (int job = pt; job < n_jobs; job += kDeqThreads) {
        const int rr = job >> lg_wpr;
        const int cw = job & (wpr - 1);
        const int sbi = cw >> 3;
        const uint32_t w = words[job];
        const __nv_bfloat162 s2 = __halves2bfloat162(sc[sbi * 128 + rr], sc[sbi * 128 + rr]);
        const __nv_bfloat162 b2 = __halves2bfloat162(bi[sbi * 128 + rr], bi[sbi * 128 + rr]);
        const uint32_t lo = w & 0x0F0F0F0Fu;         // codes 0, 2, 4, 6 in bytes 0..3
        const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // codes 1, 3, 5, 7
        uint32_t o[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          // bf16 pair (128 + q[2jj], 128 + q[2jj + 1]): 0x4300 | nibble is 128 + nibble exactly;
          // byte 0 <- byte jj of lo, byte 2 <- byte jj of hi (bytes 1 and 3 are masked off)
          const uint32_t pr = __byte_perm(lo, hi, static_cast<uint32_t>(jj) | ((4u + jj) << 8));
          const uint32_t pair = (pr & 0x00FF00FFu) | 0x43004300u;
          __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&pair);
          v = __hsub2(v, k128);    // exact: q
          v = __hfma2(s2, v, b2);  // scale * q + bias, one rounding
          o[jj] = *reinterpret_cast<const uint32_t*>(&v);
        }
        *reinterpret_cast<uint4*>(st + sbi * kQWBytes + q_sw128(rr, cw & 7)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ready[stage]));
    }
    if (!ok && lane == 0) q_abort(abort_flag, a.err);
  }

  tc_fence_before();
  cluster_wait();   // matches the arrive after initialization: every peer's barriers exist
  __syncthreads();  // this CTA's partial is in shared memory (the receive area is separate from it)

  const float* P = reinterpret_cast<const float*>(smem);
  const float* R = reinterpret_cast<const float*>(smem + a.r_off);  // [sender][owned row][m]
  if (warp == 0 && lane >= 1 && lane < a.ks) {
    const int dst = (rank + lane) % a.ks;
    const int d0w = q_chunk_begin(dst, a.ks), d1w = q_chunk_begin(dst + 1, a.ks);
    const uint32_t bar = mapa_shared(smem_u32(recv), static_cast<uint32_t>(dst));
    const uint32_t to = mapa_shared(smem_u32(R + rank * a.maxrows * S), static_cast<uint32_t>(dst));
    bulk_copy_to_cluster(to, smem_u32(P + d0w * S), static_cast<uint32_t>((d1w - d0w) * S * 4), bar);
  }
  if (!mbar_wait_bounded(smem_u32(recv), 0, nullptr, kWaitLimitNs) && threadIdx.x == 0) q_abort(abort_flag, a.err);
  const bool ok = *abort_flag == 0;

  // The owned columns n0 + w0 .. n0 + w1 - 1 for every row: item = (row m, 8 consecutive columns),
  // rows fastest so that a warp's shared-memory reads fall in distinct banks.
  const int nch = (w1 - w0) >> 3;
  const int n_items = ok ? a.M * nch : 0;
  for (int it = threadIdx.x; it < n_items; it += QCfg<AM, BM>::kThreads) {
    const int ch = it / a.M;
    const int m = it - ch * a.M;
    const int wc = w0 + 8 * ch;
    const int col = n0 + wc;
    if (col >= a.N) continue;
    float y[8], yp[8];
    const bool prev = EM && (m % a.G) != 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      y[e] = 0.f;
      yp[e] = 0.f;
    }
    for (int s = 0; s < a.ks; ++s) {
      const float* src = s == rank ? P + wc * S : R + (s * a.maxrows + (wc - w0)) * S;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        y[e] += src[e * S + m];
        if (prev) yp[e] += src[e * S + m - 1];
      }
    }
    float o[8];
    if (EM) {
      const float d0 = __bfloat162float(a.coef1[(static_cast<size_t>(m) * 2 + 0) * a.groups + col / a.gs]);
      const float d1 = __bfloat162float(a.coef1[(static_cast<size_t>(m) * 2 + 1) * a.groups + col / a.gs]);
      float res[8] = {};
      if (a.residual != nullptr) {
        const uint4 u = *reinterpret_cast<const uint4*>(a.residual + static_cast<size_t>(m) * a.N + col);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(h[e]);
          res[2 * e] = f.x;
          res[2 * e + 1] = f.y;
        }
      }
      const float4 b0a = *reinterpret_cast<const float4*>(a.base + 2 * static_cast<size_t>(a.N) + col);
      const float4 b0b = *reinterpret_cast<const float4*>(a.base + 2 * static_cast<size_t>(a.N) + col + 4);
      const float4 b1a = *reinterpret_cast<const float4*>(a.base + 3 * static_cast<size_t>(a.N) + col);
      const float4 b1b = *reinterpret_cast<const float4*>(a.base + 3 * static_cast<size_t>(a.N) + col + 4);
      const float bb0[8] = {b0a.x, b0a.y, b0a.z, b0a.w, b0b.x, b0b.y, b0b.z, b0b.w};
      const float bb1[8] = {b1a.x, b1a.y, b1a.z, b1a.w, b1b.x, b1b.y, b1b.z, b1b.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = res[e] + ((bb0[e] + d0) * y[e] + (bb1[e] + d1) * yp[e]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = y[e];
    }
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(o[2 * e], o[2 * e + 1]);
    *reinterpret_cast<uint4*>(a.out + static_cast<size_t>(m) * a.N + col) = u;
  }

  cluster_sync_all();  // every copy into every CTA of the cluster has landed before any CTA leaves
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

__host__ __device__ constexpr int q_round1024(int b) { return (b + 1023) & ~1023; }

struct QPlan {
  int tiles, ks, np, stride, n_stages, stage_bytes, r_off, region, maxrows, smem;
  int kpb, off_b, off_base, off_d0, off_raw, off_sc, off_bi;
};

template <int AM, int BM, int EM>
int q_capacity(int ks, int smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static std::mutex mu;
  static std::map<std::tuple<int, int, int>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(dev, ks, smem);
  const auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  static unsigned done = 0;
  int n = 0;
  auto kern = proj_small_kernel<AM, BM, EM>;
  if (ensure_smem_attr(kern, kQSmemLimit, &done)) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ks);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ks));
    cfg.blockDim = dim3(QCfg<AM, BM>::kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  cache[key] = n;
  return n;
}

// k-blocks per stage, at most: four for 4-bit weights (a 128-byte run of code words per weight row
// and TMA box, where one k-block has 32 bytes: the stream is bound by the rows' requests, not their
// bytes), two with the side-0 producer (half the per-stage barrier work), else one.
template <int AM, int BM>
constexpr int q_kpb_max() {
  return BM ? 4 : (AM ? 2 : 1);
}

template <int AM, int BM>
bool q_layout_kpb(int M, int K, int N, int ks, int kpb, QPlan* p) {
  p->tiles = (N + 127) / 128;
  p->ks = ks;
  p->np = std::max(16, (M + 15) / 16 * 16);
  p->stride = p->np + 4;
  p->kpb = kpb;
  p->off_b = kpb * kQWBytes;
  int off = p->off_b + kpb * p->np * 128;
  p->off_base = off;
  if (AM) off += q_round1024(kpb * 2 * kQK * 4);
  p->off_d0 = off;
  if (AM) off += q_round1024(kpb * 2 * 4 * p->np * 4);
  p->off_raw = off;
  p->off_sc = off + kpb * 128 * 32;
  p->off_bi = p->off_sc + kpb * 128 * 2;
  if (BM) off = q_round1024(p->off_bi + kpb * 128 * 2);
  p->stage_bytes = off;
  p->maxrows = 8 * ((kQChunks + ks - 1) / ks);
  const int r_bytes = q_round1024(ks * p->maxrows * p->stride * 4);
  const int p_bytes = q_round1024(128 * p->stride * 4);
  const int avail = kQSmemLimit - 1024 - kQBarBytes - r_bytes;
  if (ks > K / kQK) return false;
  const int nst = ((K / kQK + ks - 1) / ks + kpb - 1) / kpb;  // stages of the longest K range
  p->n_stages = std::min(std::min(nst, kQMaxStages), avail / p->stage_bytes);
  if (p->n_stages < 1) return false;
  const int ring = q_round1024(std::max(p->n_stages * p->stage_bytes, p_bytes));
  if (ring > avail) return false;
  p->r_off = ring;
  p->region = ring + r_bytes;
  p->smem = std::max(1024 + p->region + kQBarBytes, kQMinSmem);
  return p->smem <= kQSmemLimit;
}

// The widest stage (kpb) that fits with two stages in the ring (one where the K range needs only
// one), else the widest that fits at all.
template <int AM, int BM>
bool q_layout(int M, int K, int N, int ks, QPlan* p) {
  for (int kpb = q_kpb_max<AM, BM>(); kpb >= 1; kpb /= 2) {
    const int need = std::min(2, ((K / kQK + ks - 1) / ks + kpb - 1) / kpb);
    if (q_layout_kpb<AM, BM>(M, K, N, ks, kpb, p) && p->n_stages >= need) return true;
  }
  for (int kpb = q_kpb_max<AM, BM>(); kpb >= 1; kpb /= 2)
    if (q_layout_kpb<AM, BM>(M, K, N, ks, kpb, p)) return true;
  return false;
}

// The most K splits (<= 8, <= the k-blocks, at most one CTA per SM) whose clusters the device holds
// at once when it can say.
template <int AM, int BM, int EM>
bool q_plan(int M, int K, int N, int sms, QPlan* p, bool query) {
  if (M < 1 || M > kQMaxRows || K % kQK != 0) return false;
  const int tiles = (N + 127) / 128;
  for (int ks = std::max(1, std::min(std::min(kQMaxSplits, K / kQK), sms / tiles)); ks >= 1; --ks) {
    if (!q_layout<AM, BM>(M, K, N, ks, p)) continue;
    if (query && ks > 1) {
      const int cap = q_capacity<AM, BM, EM>(ks, p->smem);
      if (cap > 0 && cap < tiles) continue;
    }
    return true;
  }
  return false;
}

template <int AM, int BM, int EM>
int launch_small_t(const ProjSpec& s, cudaStream_t st) {
  QPlan p;
  if (!q_plan<AM, BM, EM>(s.M, s.K, s.N, sm_count(), &p, true))
    return fail(DFLASH2_ERR_UNSUPPORTED, "no small-row projection plan (M=%d K=%d N=%d)", s.M, s.K, s.N);
  QMaps maps;
  if (!make_tmap_sw128(&maps.a, s.a, static_cast<uint64_t>(s.M), static_cast<uint64_t>(s.K),
                       static_cast<uint32_t>(p.np)))
    return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (small projection activations)");
  maps.w = maps.scales = maps.biases = maps.base = maps.d0 = maps.a;
  if (BM) {
    // packed codes [N][K / 8] 32-bit words: 8 kpb words (64 kpb codes) x 128 rows; scales and
    // biases [K / 64][N] bf16: 128 values of kpb groups
    const uint64_t dims[2] = {static_cast<uint64_t>(s.K / 8), static_cast<uint64_t>(s.N)};
    const uint64_t strides[1] = {static_cast<uint64_t>(s.K / 8) * 4};
    const uint32_t box[2] = {static_cast<uint32_t>(8 * p.kpb), 128};
    const uint64_t sdims[2] = {static_cast<uint64_t>(s.N), static_cast<uint64_t>(s.K / 64)};
    const uint64_t sstr[1] = {static_cast<uint64_t>(s.N) * 2};
    const uint32_t sbox[2] = {128, static_cast<uint32_t>(p.kpb)};
    if (!make_tmap_plain(&maps.w, s.w, DFLASH2_F32, 2, dims, strides, box) ||
        !make_tmap_plain(&maps.scales, s.scales, DFLASH2_BF16, 2, sdims, sstr, sbox) ||
        !make_tmap_plain(&maps.biases, s.qbias, DFLASH2_BF16, 2, sdims, sstr, sbox))
      return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (small projection 4-bit weights)");
  } else if (!make_tmap_sw128(&maps.w, s.w, static_cast<uint64_t>(s.N), static_cast<uint64_t>(s.K), 128)) {
    return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (small projection weights)");
  }
  if (AM) {
    // base [2][2][K] fp32 as [4][K]: rows 0, 1 (side 0); d0 [2][groups][M]: the rows x 4 groups x 2 taps
    const uint64_t dims[2] = {static_cast<uint64_t>(s.K), 4};
    const uint64_t strides[1] = {static_cast<uint64_t>(s.K) * 4};
    const uint32_t box[2] = {static_cast<uint32_t>(kQK * p.kpb), 2};
    const uint64_t ddims[3] = {static_cast<uint64_t>(s.M), static_cast<uint64_t>(s.groups), 2};
    const uint64_t dstr[2] = {static_cast<uint64_t>(s.M) * 4, static_cast<uint64_t>(s.M) * s.groups * 4};
    const uint32_t dbox[3] = {static_cast<uint32_t>(p.np), static_cast<uint32_t>(p.kpb * kQK / 16), 2};
    if (!make_tmap_plain(&maps.base, s.base, DFLASH2_F32, 2, dims, strides, box) ||
        !make_tmap_plain(&maps.d0, s.d0, DFLASH2_F32, 3, ddims, dstr, dbox))
      return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (small projection side 0)");
  }
  QArgs a{};
  a.M = s.M;
  a.N = s.N;
  a.K = s.K;
  a.G = s.G > 0 ? s.G : 1;
  a.gs = s.gs > 0 ? s.gs : 8;
  a.groups = s.groups > 0 ? s.groups : 1;
  a.k_blocks = s.K / kQK;
  a.ks = p.ks;
  a.np = p.np;
  a.stride = p.stride;
  a.n_stages = p.n_stages;
  a.stage_bytes = p.stage_bytes;
  a.r_off = p.r_off;
  a.region = p.region;
  a.maxrows = p.maxrows;
  a.kpb = p.kpb;
  a.off_b = p.off_b;
  a.off_base = p.off_base;
  a.off_d0 = p.off_d0;
  a.off_raw = p.off_raw;
  a.off_sc = p.off_sc;
  a.off_bi = p.off_bi;
  a.coef1 = static_cast<const __nv_bfloat16*>(s.coef1);
  a.base = s.base;
  a.residual = static_cast<const __nv_bfloat16*>(s.residual);
  a.out = static_cast<__nv_bfloat16*>(s.out);
  a.err = device_error_word();
  static unsigned done = 0;
  auto kern = proj_small_kernel<AM, BM, EM>;
  if (!ensure_smem_attr(kern, kQSmemLimit, &done))
    return fail(DFLASH2_ERR_CUDA, "cudaFuncSetAttribute failed (small projection)");
  cudaLaunchAttribute cl[1];
  cl[0].id = cudaLaunchAttributeClusterDimension;
  cl[0].val.clusterDim.x = static_cast<unsigned>(p.ks);
  cl[0].val.clusterDim.y = 1;
  cl[0].val.clusterDim.z = 1;
  const cudaError_t e = launch_pdl(kern, dim3(p.tiles * p.ks), dim3(QCfg<AM, BM>::kThreads), p.smem, st, cl, 1,
                                   maps, a);
  return e == cudaSuccess ? DFLASH2_OK
                          : fail(DFLASH2_ERR_CUDA, "small projection launch failed: %s", cudaGetErrorString(e));
}

}  // namespace

bool proj_small_eligible(int M, int N, int K) {
  QPlan p;
  return q_plan<1, 1, 1>(M, K, N, 152, &p, false) && q_plan<0, 0, 0>(M, K, N, 152, &p, false);
}

int launch_proj_small(const ProjSpec& s, cudaStream_t st) {
  const bool am = s.d0 != nullptr, bm = s.wbits == 4, em = s.coef1 != nullptr;
  if (am && bm && em) return launch_small_t<1, 1, 1>(s, st);
  if (am && bm) return launch_small_t<1, 1, 0>(s, st);
  if (am && em) return launch_small_t<1, 0, 1>(s, st);
  if (bm && em) return launch_small_t<0, 1, 1>(s, st);
  if (am) return launch_small_t<1, 0, 0>(s, st);
  if (bm) return launch_small_t<0, 1, 0>(s, st);
  if (em) return launch_small_t<0, 0, 1>(s, st);
  return launch_small_t<0, 0, 0>(s, st);
}

}  // namespace dfl
