// kernel_projection and prepare's side-0 pass for a few rows, in one kernel.
//
// With M <= 128 rows (up to 8 blocks of 16), D = n W_kp^T is a weight stream: 4 * groups weight
// rows of H bf16 each against a handful of normed rows. The tcgen05 MMA takes the weight rows as
// its M = 128 side and the rows of n as its N side (16 .. 128, a multiple of 16; rows past M are
// TMA zero fill), so the accumulator is one 128 x N fp32 tile in TMEM. A tile holds the four
// (side, tap) weight rows of TG groups (TG = 32; the kernel also takes 16, which fills 64 of the 128
// operand rows and leaves the other accumulator lanes unread; one three-dimensional TMA box per
// k-block picks them out of W's (side, tap, group) order), so one tile's D is everything side 0
// needs for those groups.
//
// K is split over the ks CTAs of a thread-block cluster (ks <= 8). Each CTA stages its partial tile
// in shared memory as P[row of n][weight row] (rows padded by 4 floats). CTA r of the cluster owns
// the rows [np r / ks, np (r + 1) / ks) of n; every other CTA sends it those rows of its partial
// with one bulk copy into r's shared memory (distributed shared memory, counted as transaction
// bytes on an mbarrier of r). The owner adds the ks partials in K order (in place, in its own P),
// writes side 1's deltas (coef1) and D (d_full, optional), and applies side 0 to its rows
//   out[m, c] = (base[0][0][c] + D[m, 0, 0, g]) n[m, c] + (base[0][1][c] + D[m, 0, 1, g]) n[m - 1, c]
// with n[m - 1] = 0 at a block's first row and g = c / group size (MAX DFlash2TransformerBlock:
// norm -> conv.prepare; dflash2.ts #coefficients: the projection of the normed hidden, reshaped to
// (side, tap, group); #conv with side 0). The coefficients-only entry writes side 0's deltas
// (d0 [tap][group][row]) instead of applying them.
//
// Warp roles: 0 TMA (one lane), 1 TMEM allocation + MMA issue (one lane), 2-5 read the accumulator
// (warp w reads TMEM lanes 32 (w % 4) .. +31). All six warps then reduce and apply. Every mbarrier
// wait is bounded. A CTA whose wait ran out records DFLASH2_ERR_TIMEOUT, still takes part in the
// cluster barriers and sends its (meaningless) partial so that its peers never wait for it, and
// writes no output.
#include <cuda_bf16.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {
namespace {

constexpr int kKsK = 64;              // K per stage: one 128-byte swizzled bf16 row
constexpr int kKsWBytes = 128 * 128;  // the A operand: 128 weight rows (64 of them loaded when TG = 16)
constexpr int kKsThreads = 192;
constexpr int kKsMaxRows = 128;  // rows of n (the MMA's N side) at most
constexpr int kKsMaxSplits = 8;
constexpr int kKsTileGroups = 32;  // groups per tile the plan uses
constexpr int kKsMaxStages = 12;
constexpr int kKsSmemLimit = 232448;
constexpr int kKsBarBytes = 256;
constexpr int kKsMinSmem = 64 * 1024;  // at most three CTAs per SM: their TMEM (<= 128 columns each) always fits
constexpr int kKsHalfSmem = 112 * 1024;  // two CTAs per SM
#ifndef DFL_KS_TWO_PER_SM
#define DFL_KS_TWO_PER_SM 1
#endif
constexpr uint64_t kKsDrainNs = 100000000ull;  // 100 ms

struct KsArgs {
  const __nv_bfloat16* n;  // [M][H] normed rows
  const float* base;       // [2][2][H]
  __nv_bfloat16* out;      // [M][H] side-0 output, or null: coefficients only (d0 instead)
  __nv_bfloat16* coef1;    // [M][2][groups] side 1's deltas
  float* d_full;           // [M][4][groups] or null
  float* d0;               // [2][groups][M] side 0's deltas (coefficients only) or null
  int M, H, G, gs, groups;
  int tg;                  // groups per tile (16 or 32)
  int k_blocks, ks, np, stride, n_stages, stage_bytes, r_off, region;
  int stg_off, stg_rows, lg_box, nbox;  // side-0 operands staged by TMA: rows r0 - 1 .. r1 - 1 of n, base
  int* err;
};

__device__ __forceinline__ void ks_abort(volatile int* abort_flag, int* err) {
  *abort_flag = 1;
  if (err != nullptr) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_TIMEOUT));
}

__global__ void __launch_bounds__(kKsThreads, 1)
    kp_small_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmN,
                    const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmB, const KsArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.region);
  uint64_t* empty = full + a.n_stages;
  uint64_t* acc_full = empty + a.n_stages;
  uint64_t* recv = acc_full + 1;
  uint64_t* drain = recv + 1;
  uint64_t* stg_full = drain + 1;  // the side-0 operands have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stg_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int tg = a.tg;
  const int wrows = 4 * tg;                                   // weight rows of the tile
  const int g0 = (static_cast<int>(blockIdx.x) / a.ks) * tg;  // the tile's first group
  const int kb0 = a.k_blocks * rank / a.ks;
  const int nkb = a.k_blocks * (rank + 1) / a.ks - kb0;
  const int S = a.stride;                                            // floats per row of P
  const int r0 = a.np * rank / a.ks, r1 = a.np * (rank + 1) / a.ks;  // the rows this CTA owns
  const int maxr = (a.np + a.ks - 1) / a.ks;
  const uint32_t tmem_cols = a.np <= 32 ? 32u : (a.np <= 64 ? 64u : 128u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.n_stages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(recv), 1);
    mbar_init(smem_u32(drain), 1);
    mbar_init(smem_u32(stg_full), 1);
    *abort_flag = 0;
    fence_mbar_init();
    // the peers' partial rows of this CTA's rows: (ks - 1) senders (none when ks = 1)
    mbar_arrive_expect_tx(smem_u32(recv), static_cast<uint32_t>((a.ks - 1) * (r1 - r0) * S * 4));
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmN);
    if (a.out != nullptr) {
      prefetch_tmap(&tmS);
      prefetch_tmap(&tmB);
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
  cluster_arrive_relaxed();  // this CTA's barriers exist for a peer once its matching wait returns
  pdl_trigger();
  if (threadIdx.x != 0) pdl_wait();  // the producer waits after requesting the first weight tiles

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();  // each weight row is read by one CTA
      const uint64_t pol_n = policy_evict_last();   // the rows of n are read by every tile
      const uint32_t tx = static_cast<uint32_t>(wrows * 128 + a.np * 128);
      const int pre = min(nkb, a.n_stages);
      // The weights are never written by the kernels this launch overlaps: the first stages'
      // weight tiles are requested before the dependent-launch wait.
      for (int i = 0; i < pre; ++i) {
        const uint32_t fb = smem_u32(&full[i]);
        mbar_arrive_expect_tx(fb, tx);
        tma_load_3d(smem_u32(smem + i * a.stage_bytes), &tmW, fb, (kb0 + i) * kKsK, g0, 0, pol_w);
      }
      pdl_wait();
      if (a.out != nullptr) {
        // side 0's operands for this CTA's rows and the tile's channels (row r0 - 1 is the first
        // row's predecessor; rows outside [0, M) are zero fill)
        const int box = 1 << a.lg_box;
        const uint32_t sb = smem_u32(stg_full);
        mbar_arrive_expect_tx(sb, static_cast<uint32_t>(a.nbox * box * (a.stg_rows * 2 + 2 * 4)));
        uint8_t* sn = smem + a.stg_off;
        uint8_t* sbase = sn + a.nbox * a.stg_rows * box * 2;
        for (int j = 0; j < a.nbox; ++j) {
          const int x = g0 * a.gs + j * box;
          tma_load_2d(smem_u32(sn + j * a.stg_rows * box * 2), &tmS, sb, x, r0 - 1, pol_n);
          tma_load_2d(smem_u32(sbase + j * 2 * box * 4), &tmB, sb, x, 0, pol_n);
        }
      }
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < nkb; ++i) {
        const int stage = i % a.n_stages;
        const uint32_t phase = static_cast<uint32_t>(i / a.n_stages) & 1u;
        const uint32_t fb = smem_u32(&full[stage]);
        uint8_t* st = smem + stage * a.stage_bytes;
        if (i >= pre) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(fb, tx);
          tma_load_3d(smem_u32(st), &tmW, fb, (kb0 + i) * kKsK, g0, 0, pol_w);
        }
        tma_load_2d(smem_u32(st + kKsWBytes), &tmN, fb, (kb0 + i) * kKsK, 0, pol_n);
        issued = i + 1;
      }
      if (!ok) {
        ks_abort(abort_flag, a.err);
        // the copies still in flight land before the shared memory is reused
        for (int i = max(0, issued - a.n_stages); i < issued; ++i)
          mbar_wait_bounded(smem_u32(&full[i % a.n_stages]), static_cast<uint32_t>(i / a.n_stages) & 1u, nullptr,
                            kKsDrainNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc(false, 128, a.np);
      bool ok = true, any = false;
      for (int i = 0; i < nkb; ++i) {
        const int stage = i % a.n_stages;
        const uint32_t phase = static_cast<uint32_t>(i / a.n_stages) & 1u;
        if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * a.stage_bytes);
        const uint64_t adesc = desc_kmajor_swizzled<128>(sa);
        const uint64_t bdesc = desc_kmajor_swizzled<128>(sa + kKsWBytes);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // 16-element (32-byte) steps along the swizzled rows
          mma_f16(tmem, adesc + static_cast<uint64_t>(2 * k), bdesc + static_cast<uint64_t>(2 * k), idesc,
                  (i > 0 || k > 0) ? 1u : 0u);
        mma_commit(smem_u32(&empty[stage]));
        any = true;
      }
      if (ok) {
        mma_commit(smem_u32(acc_full));
      } else {
        ks_abort(abort_flag, a.err);
        if (any) {
          mma_commit(smem_u32(drain));
          mbar_wait_bounded(smem_u32(drain), 0, nullptr, kKsDrainNs);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ accumulator -> shared memory
    // TMEM lane w holds weight row w of the tile, one column per row of n. The ring is idle once
    // the accumulator is complete, so the partial P[row][w] reuses it.
    const int p = warp & 3;  // TMEM lanes 32 p .. 32 p + 31
    if (32 * p < wrows) {
      if (mbar_wait_bounded(smem_u32(acc_full), 0, abort_flag, kWaitLimitNs)) {
        tc_fence_after();
        float* P = reinterpret_cast<float*>(smem);
        const int w = 32 * p + lane;
        for (int cc = 0; cc * 32 < a.np; ++cc) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * p) << 16) + static_cast<uint32_t>(cc * 32), r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (cc * 32 + j < a.np) P[(cc * 32 + j) * S + w] = __uint_as_float(r[j]);
        }
        fence_proxy_async_smem();  // the bulk copies below read these rows
      } else if (lane == 0) {
        ks_abort(abort_flag, a.err);
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  cluster_wait();   // matches the arrive after initialization: every peer's barriers exist
  __syncthreads();  // this CTA's partial is in shared memory (the receive area is separate from it)

  float* P = reinterpret_cast<float*>(smem);
  const float* R = reinterpret_cast<const float*>(smem + a.r_off);  // [sender][owned row][w]
  if (warp == 0 && lane >= 1 && lane < a.ks) {
    // lane j sends the rows of owner rank + j, so that the copies issue in parallel
    const int dst = (rank + lane) % a.ks;
    const int d0r = a.np * dst / a.ks, d1r = a.np * (dst + 1) / a.ks;
    const uint32_t bar = mapa_shared(smem_u32(recv), static_cast<uint32_t>(dst));
    const uint32_t to = mapa_shared(smem_u32(R + rank * maxr * S), static_cast<uint32_t>(dst));
    bulk_copy_to_cluster(to, smem_u32(P + d0r * S), static_cast<uint32_t>((d1r - d0r) * S * 4), bar);
  }
  // Every peer sends, so this wait ends; it ignores the abort flag so that no copy into this CTA
  // is still in flight when the CTA leaves.
  if (!mbar_wait_bounded(smem_u32(recv), 0, nullptr, kWaitLimitNs) && threadIdx.x == 0)
    ks_abort(abort_flag, a.err);
  const bool ok = *abort_flag == 0;

  // D of the owned rows: the ks partials in K order, summed in place in P; coef1 and d_full from it.
  // Thread item = 4 consecutive weight rows (4 groups of one section) of one row of n; tg and the
  // group size are powers of two, so every index below is a shift or a mask.
  const int M = a.M;
  const int rows = max(0, min(r1, M) - r0);
  const int lg_tg = 31 - __clz(tg);
  const bool vec_ok = (a.groups & 3) == 0;  // 4 groups' coef1 / d_full values as one aligned store
  for (int it = threadIdx.x; it < (rows << (lg_tg)); it += kKsThreads) {
    const int w = (it & (tg - 1)) << 2;
    const int m = r0 + (it >> lg_tg);
    float4 v[kKsMaxSplits];
#pragma unroll
    for (int s = 0; s < kKsMaxSplits; ++s)
      v[s] = s >= a.ks ? make_float4(0.f, 0.f, 0.f, 0.f)
                       : *reinterpret_cast<const float4*>(s == rank ? P + m * S + w
                                                                    : R + (s * maxr + (m - r0)) * S + w);
    float4 d = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < kKsMaxSplits; ++s)
      if (s < a.ks) {
        d.x += v[s].x;
        d.y += v[s].y;
        d.z += v[s].z;
        d.w += v[s].w;
      }
    *reinterpret_cast<float4*>(P + m * S + w) = d;
    if (!ok) continue;
    const int q = w >> lg_tg;
    const int g = g0 + (w & (tg - 1));
    const float dv[4] = {d.x, d.y, d.z, d.w};
    if (q >= 2) {
      __nv_bfloat16* dst = a.coef1 + (static_cast<size_t>(m) * 2 + (q - 2)) * a.groups + g;
      if (vec_ok && g + 3 < a.groups) {
        uint2 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
        h[0] = __floats2bfloat162_rn(d.x, d.y);
        h[1] = __floats2bfloat162_rn(d.z, d.w);
        *reinterpret_cast<uint2*>(dst) = u;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (g + e < a.groups) dst[e] = __float2bfloat16_rn(dv[e]);
      }
    } else if (a.d0 != nullptr) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (g + e < a.groups) a.d0[(static_cast<size_t>(q) * a.groups + g + e) * M + m] = dv[e];
    }
    if (a.d_full != nullptr) {
      float* dst = a.d_full + (static_cast<size_t>(m) * 4 + q) * a.groups + g;
      if (vec_ok && g + 3 < a.groups) {
        *reinterpret_cast<float4*>(dst) = d;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (g + e < a.groups) dst[e] = dv[e];
      }
    }
  }
  __syncthreads();

  // side 0 over the owned rows and the tile's channels, from the staged operands: thread item = 8
  // channels of one row
  const int lg_vpg = 31 - __clz(a.gs >> 3);  // log2 of the 8-channel vectors per group
  const int lg_vpr = lg_tg + lg_vpg;         // log2 of the vectors per row
  int n_items = (ok && a.out != nullptr) ? rows << lg_vpr : 0;
  if (n_items > 0 && !mbar_wait_bounded(smem_u32(stg_full), 0, abort_flag, kWaitLimitNs)) {
    ks_abort(abort_flag, a.err);
    n_items = 0;
  }
  const int box = 1 << a.lg_box;
  const __nv_bfloat16* sn = reinterpret_cast<const __nv_bfloat16*>(smem + a.stg_off);
  const float* sbase = reinterpret_cast<const float*>(smem + a.stg_off + a.nbox * a.stg_rows * box * 2);
  for (int it = threadIdx.x; it < n_items; it += kKsThreads) {
    const int cl = (it & ((1 << lg_vpr) - 1)) << 3;  // channel within the tile
    const int m = r0 + (it >> lg_vpr);
    const int gl = cl >> (lg_vpg + 3);
    if (g0 + gl >= a.groups) continue;
    const int j = cl >> a.lg_box;
    const int cw = cl & (box - 1);
    const __nv_bfloat16* rowp = sn + (j * a.stg_rows + (m - r0)) * box + cw;  // row m - 1
    const uint4 pu = m % a.G > 0 ? *reinterpret_cast<const uint4*>(rowp) : make_uint4(0u, 0u, 0u, 0u);
    const uint4 cu = *reinterpret_cast<const uint4*>(rowp + box);          // row m
    const float* bp = sbase + j * 2 * box + cw;
    const float4 b0a = *reinterpret_cast<const float4*>(bp);
    const float4 b0b = *reinterpret_cast<const float4*>(bp + 4);
    const float4 b1a = *reinterpret_cast<const float4*>(bp + box);
    const float4 b1b = *reinterpret_cast<const float4*>(bp + box + 4);
    const float b0[8] = {b0a.x, b0a.y, b0a.z, b0a.w, b0b.x, b0b.y, b0b.z, b0b.w};
    const float b1[8] = {b1a.x, b1a.y, b1a.z, b1a.w, b1b.x, b1b.y, b1b.z, b1b.w};
    const float d0 = P[m * S + gl];       // D[m, 0, 0, g]
    const float d1 = P[m * S + tg + gl];  // D[m, 0, 1, g]
    const __nv_bfloat162* ch = reinterpret_cast<const __nv_bfloat162*>(&cu);
    const __nv_bfloat162* ph = reinterpret_cast<const __nv_bfloat162*>(&pu);
    uint4 o;
    __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 cv = __bfloat1622float2(ch[i]);
      const float2 pv = __bfloat1622float2(ph[i]);
      const float lo = fmaf(b0[2 * i] + d0, cv.x, (b1[2 * i] + d1) * pv.x);
      const float hi = fmaf(b0[2 * i + 1] + d0, cv.y, (b1[2 * i + 1] + d1) * pv.y);
      oh[i] = __floats2bfloat162_rn(lo, hi);
    }
    *reinterpret_cast<uint4*>(a.out + static_cast<size_t>(m) * a.H + g0 * a.gs + cl) = o;
  }

  // the staged operands have landed (already so unless a wait ran out) before the CTA leaves
  if (a.out != nullptr && threadIdx.x == 0) mbar_wait_bounded(smem_u32(stg_full), 0, nullptr, kKsDrainNs);
  cluster_sync_all();  // every copy into every CTA of the cluster has landed before any CTA leaves
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

__host__ __device__ constexpr int round1024(int b) { return (b + 1023) & ~1023; }

struct KsPlan {
  int tg, tiles, ks, np, stride, n_stages, stage_bytes, r_off, stg_off, stg_rows, lg_box, nbox, region, smem;
};

// Clusters of ks CTAs with `smem` bytes each that the current device holds at once (0: unknown).
int ks_capacity(int ks, int smem) {
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
  if (ensure_smem_attr(kp_small_kernel, kKsSmemLimit, &done)) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ks);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ks));
    cfg.blockDim = dim3(kKsThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kp_small_kernel, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  cache[key] = n;
  return n;
}

// Shared-memory layout of one (TG, ks) candidate; false if it does not fit.
bool ks_layout(const ConvShape& s, int tg, int ks, KsPlan* p) {
  const int k_blocks = s.H / kKsK;
  p->tg = tg;
  p->tiles = (s.groups + tg - 1) / tg;
  p->ks = ks;
  p->np = std::max(16, (s.rows() + 15) / 16 * 16);
  p->stride = 4 * tg + 4;
  p->stage_bytes = kKsWBytes + p->np * 128;
  const int maxr = (p->np + ks - 1) / ks;
  // [ring, then the partial P over it][receive area R][staged side-0 operands][barriers]
  const int chans = tg * s.gs;  // channels of a tile (a power of two)
  const int box = std::min(256, chans);
  p->lg_box = 31 - __builtin_clz(static_cast<unsigned>(box));
  p->nbox = chans / box;
  p->stg_rows = maxr + 1;
  const int r_bytes = round1024(ks * maxr * p->stride * 4);
  const int stg_bytes = round1024(p->nbox * box * (p->stg_rows * 2 + 2 * 4));
  const int p_bytes = round1024(p->np * p->stride * 4);
  const int avail = kKsSmemLimit - 1024 - kKsBarBytes - r_bytes - stg_bytes;
  const int nkb = (k_blocks + ks - 1) / ks;
  p->n_stages = std::min(std::min(nkb, kKsMaxStages), avail / p->stage_bytes);
  if (p->n_stages < 1) return false;
  // Two CTAs per SM where a ring of at least four stages still fits in half of an SM: the next
  // launch's clusters then start on the SMs this one holds and request their weights before the
  // dependent-launch wait, instead of waiting for this launch's CTAs to leave.
  const int avail_half = kKsHalfSmem - 1024 - kKsBarBytes - r_bytes - stg_bytes;
  const int n_half = std::min(std::min(nkb, kKsMaxStages), std::max(0, avail_half) / p->stage_bytes);
  if (DFL_KS_TWO_PER_SM && n_half >= std::min(nkb, 4) &&
      round1024(std::max(n_half * p->stage_bytes, p_bytes)) <= avail_half)
    p->n_stages = n_half;
  const int ring = round1024(std::max(p->n_stages * p->stage_bytes, p_bytes));
  if (ring > avail) return false;
  p->r_off = ring;
  p->stg_off = ring + r_bytes;
  p->region = ring + r_bytes + stg_bytes;
  p->smem = std::max(1024 + p->region + kKsBarBytes, kKsMinSmem);
  return p->smem <= kKsSmemLimit;
}

// The plan: tiles of 32 groups and the most K splits (<= 8, <= the k-blocks) whose clusters the
// device holds at once (when it can say). Tiles of 16 groups put 1.5x the CTAs on the weight
// stream but measured slower (fewer rows per TMA box, more scattered DRAM rows), so the plan keeps
// 32; the kernel takes either. With query = false (no device needed) it only decides whether a
// plan exists.
bool ks_plan(const ConvShape& s, int sms, KsPlan* p, bool query) {
  const int M = s.rows();
  if (s.dtype != DFLASH2_BF16 || M < 1 || M > kKsMaxRows || s.H % kKsK != 0 || s.gs < 8 || (s.gs & (s.gs - 1)) != 0)
    return false;
  const int k_blocks = s.H / kKsK;
  const int tiles = (s.groups + kKsTileGroups - 1) / kKsTileGroups;
  for (int ks = std::max(1, std::min(std::min(kKsMaxSplits, k_blocks), sms / tiles)); ks >= 1; --ks) {
    if (!ks_layout(s, kKsTileGroups, ks, p)) continue;
    if (query && ks > 1) {
      const int cap = ks_capacity(ks, p->smem);
      if (cap > 0 && cap < tiles) continue;  // a second wave of clusters would double the stream time
    }
    return true;
  }
  return false;
}

}  // namespace

bool kp_small_eligible(const ConvShape& s, int sms) {
  KsPlan p;
  return ks_plan(s, sms, &p, false);
}

int launch_kp_small(const ConvShape& s, const void* n, const void* w_kp, const float* base, void* out, void* coef1,
                    float* d_full, cudaStream_t st, float* d0) {
  KsPlan p;
  if (!ks_plan(s, sm_count(), &p, true)) return fail(DFLASH2_ERR_UNSUPPORTED, "no small-row plan for this shape");
  CUtensorMap mW, mN, mS, mB;
  // W [4 sections][groups][H]: one box brings the four (side, tap) sections of a tile's groups
  if (!make_tmap_sw128_3d(&mW, w_kp, s.H, s.groups, 4, static_cast<uint64_t>(s.groups) * s.H * 2,
                          static_cast<uint32_t>(p.tg), 4) ||
      !make_tmap_sw128(&mN, n, s.rows(), s.H, static_cast<uint32_t>(p.np)))
    return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (small-row kernel_projection)");
  const uint64_t sdims[2] = {static_cast<uint64_t>(s.H), static_cast<uint64_t>(s.rows())};
  const uint64_t sstr[1] = {static_cast<uint64_t>(s.H) * 2};
  const uint32_t sbox[2] = {1u << p.lg_box, static_cast<uint32_t>(p.stg_rows)};
  const uint64_t bdims[2] = {static_cast<uint64_t>(s.H), 4};
  const uint64_t bstr[1] = {static_cast<uint64_t>(s.H) * 4};
  const uint32_t bbox[2] = {1u << p.lg_box, 2};
  if (out != nullptr && (!make_tmap_plain(&mS, n, DFLASH2_BF16, 2, sdims, sstr, sbox) ||
                         !make_tmap_plain(&mB, base, DFLASH2_F32, 2, bdims, bstr, bbox)))
    return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (small-row kernel_projection)");
  static unsigned done = 0;
  if (!ensure_smem_attr(kp_small_kernel, kKsSmemLimit, &done))
    return fail(DFLASH2_ERR_CUDA, "cudaFuncSetAttribute failed (small-row kernel_projection)");
  KsArgs a;
  a.n = static_cast<const __nv_bfloat16*>(n);
  a.base = base;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.coef1 = static_cast<__nv_bfloat16*>(coef1);
  a.d_full = d_full;
  a.d0 = d0;
  a.M = s.rows();
  a.H = s.H;
  a.G = s.G;
  a.gs = s.gs;
  a.groups = s.groups;
  a.tg = p.tg;
  a.k_blocks = s.H / kKsK;
  a.ks = p.ks;
  a.np = p.np;
  a.stride = p.stride;
  a.n_stages = p.n_stages;
  a.stage_bytes = p.stage_bytes;
  a.r_off = p.r_off;
  a.region = p.region;
  a.stg_off = p.stg_off;
  a.stg_rows = p.stg_rows;
  a.lg_box = p.lg_box;
  a.nbox = p.nbox;
  if (out == nullptr) {
    mS = mN;
    mB = mN;
  }
  a.err = device_error_word();
  cudaLaunchAttribute cl[1];
  cl[0].id = cudaLaunchAttributeClusterDimension;
  cl[0].val.clusterDim.x = static_cast<unsigned>(p.ks);
  cl[0].val.clusterDim.y = 1;
  cl[0].val.clusterDim.z = 1;
  const cudaError_t e =
      launch_pdl(kp_small_kernel, dim3(p.tiles * p.ks), dim3(kKsThreads), p.smem, st, cl, 1, mW, mN, mS, mB, a);
  return e == cudaSuccess ? DFLASH2_OK
                          : fail(DFLASH2_ERR_CUDA, "small-row kernel_projection launch failed: %s",
                                 cudaGetErrorString(e));
}

}  // namespace dfl
