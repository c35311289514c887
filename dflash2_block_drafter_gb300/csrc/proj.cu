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
// a weight tile in L2). With at least half as many tiles as SMs the work is split stream-K: CTA c
// takes the k-blocks [c T / C, (c + 1) T / C) of the T = tiles x K/64 k-blocks in tile-major order, so
// every CTA issues the same number of MMAs whatever the tile count. The CTA that holds a tile's
// first k-block owns the tile: the later CTAs that hold the rest of its K range (always their first
// piece, which they compute first) write their fp32 partial tile to a workspace slot and raise one
// flag per 32-row quarter; the owner's epilogue warp of that quarter waits for the flags (bounded),
// adds the partials in K order and applies the epilogue. Without stream-K (few tiles) K is split
// into equal ranges summed by a reduce pass. K advances in 64-element stages: every operand row is one 128-byte
// swizzled row, as TMA writes it, and the producer warps write their tiles in the same layout
// (16-byte chunk c of row r at chunk position c ^ (r & 7) of the row, 1024-byte aligned tiles).
// Warp roles: 0 TMA, 1 TMEM + MMA issue (one lane), 2-5 epilogue (TMEM lanes 32 (w % 4) ..),
// then 8 conv-producer warps and/or 8 dequant warps (a 16-byte chunk of a few rows per thread,
// packed fp32 or bf16 pair arithmetic). Producer and epilogue warps wait with suspending
// try_waits, leaving the issue slots to the warps that work. The accumulator is double-buffered
// in TMEM (2 x 256 columns). Every wait is bounded: a timeout raises a CTA-wide abort flag,
// records DFLASH2_ERR_TIMEOUT, drains the copies and MMAs in flight and frees TMEM before the
// kernel returns.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {
namespace {

constexpr int kPM = 128;                     // rows per tile
constexpr int kPK = 64;                      // K per stage (one 128-byte bf16 row)
constexpr int kAOp = kPM * 128;              // A operand tile bytes
constexpr int kQGroup = 64;                  // quantisation group along K
constexpr uint64_t kPDrainNs = 100000000ull; // 100 ms
constexpr int kPSmemLimit = 232448;

// Stage layout (every part 1024-byte aligned): the A operand (AM: the normed rows n land there
// and the producer warps turn them into Conv_0(n) in place), the B operand, then (AM) side 0's base
// kernel [2][64] fp32 and the rows' side-0 deltas [2 taps][4 groups][128 rows] fp32 (group size 16),
// then (BM) the
// packed codes [NT][8 words] and the scales and biases [NT] of the stage's group.
template <int AM, int BM, int NT>
struct PLayout {
  static constexpr int kBOp = NT * 128;
  static constexpr int kOffBase = kAOp + kBOp;
  static constexpr int kOffD0 = kOffBase + 1024;
  static constexpr int kARaw = AM ? 1024 + kPM * 2 * 4 * 4 : 0;
  static constexpr int kOffBRaw = kOffBase + kARaw;
  static constexpr int kOffScale = kOffBRaw + NT * 32;
  static constexpr int kOffBias = kOffScale + NT * 2;
  static constexpr int kBRaw = BM ? ((NT * 32 + NT * 4 + 1023) / 1024) * 1024 : 0;
  static constexpr int kStageBytes = kAOp + kBOp + kARaw + kBRaw;
};

// P = 1: CTA pairs (cta_group::2) over 256 x NT tiles; each CTA of the pair stages its own 128 rows
// of A and half of the tile's weight rows (kBRows), so a k-block brings it a third fewer bytes. Only
// the plain projection (no producer warps, no conv epilogue) runs in pairs.
template <int AM, int BM, int EM, int NT, int P>
struct PCfg {
  static constexpr int kConvWarps = AM ? 8 : 0;
  static constexpr int kDeqWarps = BM ? 8 : 0;
  static constexpr int kProdWarps = kConvWarps + kDeqWarps;
  static constexpr int kThreads = 64 + 128 + 32 * kProdWarps;
  static constexpr int kBRows = P ? NT / 2 : NT;  // weight rows this CTA stages per k-block
  static constexpr int kTileM = P ? 2 * kPM : kPM;
  static constexpr int kStageBytes = PLayout<AM, BM, kBRows>::kStageBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kFit = (kPSmemLimit - 1024 - kBarBytes) / kStageBytes;
  static constexpr int kStages = kFit > 8 ? 8 : kFit;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes;
  static constexpr int kTmemCols = NT == 256 ? 512 : 128;  // two accumulator buffers
};

struct ProjArgs {
  int M, N, K;
  int k_splits;                // > 1: fp32 partial sums of K ranges to `part`, summed by proj_reduce_kernel
  int stream_k;                // 1: stream-K shares; `part` holds one [128][NT] fp32 slot per CTA
  float* part;                 // [k_splits][M][N], or the stream-K slots
  int a_rows;                  // rows of the A box (up to 128: fewer when M is small)
  int tiles_m, tiles_n;
  int G, gs, groups;           // conv shape (G rows per block, group size, channels / group size)
  const __nv_bfloat16* coef1;  // EM: side-1 deltas [M][2][groups] bf16
  const float* base;           // EM: [2][2][N] fp32 (side 1 is used)
  const __nv_bfloat16* residual;  // EM: [M][N] or null
  __nv_bfloat16* out;          // [M][N]
  int* err;
};

struct ProjMaps {
  CUtensorMap a, b, base, d0, scales, biases;
};

// Stream-K hand-off flags: [CTA][epilogue warp] = 1 once that CTA's partial rows 32 q .. 32 q + 31
// of its first tile are in its slot. The owner resets each flag after reading, so every launch
// starts (and ends) with all flags 0; a CTA also clears its own flags when it starts. Calls that
// overlap on the GPU would share them: keep projections of one device on one stream.
constexpr int kSkMaxCtas = 1024;
#ifndef DFL_PROJ_PAIR
#define DFL_PROJ_PAIR 1
#endif

__device__ int g_sk_flags[kSkMaxCtas][4];

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits (bounded) until a stream-K flag is raised; false on timeout or abort.
__device__ __forceinline__ bool sk_wait(const int* flag, const volatile int* abort_flag) {
  if (ld_acquire_gpu(flag) != 0) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(64);
    if (ld_acquire_gpu(flag) != 0) return true;
    if ((i & 15u) == 0u) {
      if (*abort_flag != 0) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// One piece of this CTA's work: tile t, k-blocks [kb0, kb1), split-K range ks.
struct PSeg {
  int t, kb0, kb1, ks;
};
// Piece `idx` (0, 1, ...) of work unit `unit` (a CTA, or a CTA pair) of `units`: split-K items (tile
// it % n_tiles, K range it / n_tiles) or the idx-th tile touched by the unit's stream-K share; false
// past the last.
__device__ __forceinline__ bool p_seg(const ProjArgs& a, int k_stages, int n_tiles, int unit, int units, int idx,
                                      PSeg& g) {
  if (!a.stream_k) {
    const int it = unit + idx * units;
    if (it >= n_tiles * a.k_splits) return false;
    g.t = it % n_tiles;
    g.ks = it / n_tiles;
    g.kb0 = k_stages * g.ks / a.k_splits;
    g.kb1 = k_stages * (g.ks + 1) / a.k_splits;
    return true;
  }
  const long long total = static_cast<long long>(n_tiles) * k_stages;
  const long long s0 = total * unit / units, e0 = total * (unit + 1) / units;
  const long long s = idx == 0 ? s0 : (s0 / k_stages + idx) * k_stages;
  if (s >= e0) return false;
  g.t = static_cast<int>(s / k_stages);
  g.kb0 = static_cast<int>(s - static_cast<long long>(g.t) * k_stages);
  g.kb1 = static_cast<int>(min(static_cast<long long>(k_stages), e0 - static_cast<long long>(g.t) * k_stages));
  g.ks = 0;
  return true;
}

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

// The epilogue operands of one 32-column chunk of one row (conv side 1 + residual).
struct EpiChunk {
  uint4 res[4];   // residual, bf16
  float d[2][4];  // side-1 deltas of the chunk's groups (up to 4: gs >= 8)
};
__device__ __forceinline__ void load_epi_chunk(EpiChunk& e, const ProjArgs& a, bool valid, int row, int col0) {
  const bool in = valid && col0 < a.N;
#pragma unroll
  for (int v = 0; v < 4; ++v)
    e.res[v] = (in && a.residual != nullptr)
                   ? __ldg(reinterpret_cast<const uint4*>(a.residual + static_cast<size_t>(row) * a.N + col0 + 8 * v))
                   : make_uint4(0u, 0u, 0u, 0u);
  const int gpc = 32 / a.gs;
#pragma unroll
  for (int tap = 0; tap < 2; ++tap)
#pragma unroll
    for (int gi = 0; gi < 4; ++gi)
      e.d[tap][gi] = (in && gi < gpc) ? __bfloat162float(
                                            a.coef1[(static_cast<size_t>(row) * 2 + tap) * a.groups + col0 / a.gs + gi])
                                      : 0.f;
}

template <int AM, int BM, int EM, int NT, int P>
__global__ void __launch_bounds__(PCfg<AM, BM, EM, NT, P>::kThreads, 1)
    proj_kernel(const __grid_constant__ ProjMaps maps, const ProjArgs a) {
  using C = PCfg<AM, BM, EM, NT, P>;
  using L = PLayout<AM, BM, C::kBRows>;
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
  const int gpc = AM ? kPK / 16 : 1;  // groups per stage (conv side 0 over K, group size 16)
  // Pairs (the plain projection only): rank 0 (the leader) issues the MMAs for both CTAs, both CTAs'
  // TMA loads complete on the leader's full barrier (cta_group::2 copies; the leader expects both
  // halves' bytes), and the leader's acc_empty counts both CTAs' epilogue warps.
  static_assert(!P || (C::kProdWarps == 0 && !EM), "CTA pairs only for the plain projection");
  const uint32_t rank = P ? cluster_ctarank() : 0u;
  constexpr bool kLeaderFull = P != 0;
  const int unit = P ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = P ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&ready[s]), C::kProdWarps > 0 ? C::kProdWarps : 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), P ? 8 : 4);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&maps.a);
    prefetch_tmap(&maps.b);
    if (AM) {
      prefetch_tmap(&maps.base);
      prefetch_tmap(&maps.d0);
    }
    if (BM) {
      prefetch_tmap(&maps.scales);
      prefetch_tmap(&maps.biases);
    }
  }
  if (warp == 1) {
    if (P) {
      tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (P)
    cluster_sync_all();  // both CTAs' barriers exist before the peer arrives on the leader's
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();
  pdl_wait();
  if (a.stream_k && threadIdx.x < 4) g_sk_flags[blockIdx.x][threadIdx.x] = 0;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_last();   // activations: re-read by every column tile
      const uint64_t pol_w = policy_evict_normal(); // weights: shared by the CTAs of one column tile
      constexpr int kB = C::kBRows;
      const uint32_t bytes = static_cast<uint32_t>(a.a_rows * 128 + (BM ? kB * 32 + kB * 4 : kB * 128) +
                                                   (AM ? 2 * kPK * 4 + a.a_rows * 2 * gpc * 4 : 0));
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      PSeg g;
      for (int idx = 0; ok && p_seg(a, k_stages, n_tiles, unit, units, idx, g); ++idx) {
        const int m0 = (g.t % a.tiles_m) * C::kTileM + static_cast<int>(rank) * kPM;  // this CTA's rows
        const int n0 = (g.t / a.tiles_m) * NT + static_cast<int>(rank) * C::kBRows;  // its weight rows
        for (int kb = g.kb0; kb < g.kb1; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          uint8_t* st = smem + stage * C::kStageBytes;
          if (kLeaderFull) {
            // both CTAs' operands complete on the leader's barrier, which counts both halves' bytes
            const uint32_t fbl = mapa_shared(fb, 0);
            if (rank == 0) mbar_arrive_expect_tx(fb, 2 * bytes);
            tma_load_2d_pair(smem_u32(st), &maps.a, fbl, kb * kPK, m0, pol_a);
            tma_load_2d_pair(smem_u32(st + kAOp), &maps.b, fbl, kb * kPK, n0, pol_w);
            ++issued;
            if (++stage == C::kStages) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          mbar_arrive_expect_tx(fb, bytes);
          tma_load_2d(smem_u32(st), &maps.a, fb, kb * kPK, m0, pol_a);
          if (AM) {
            tma_load_2d(smem_u32(st + L::kOffBase), &maps.base, fb, kb * kPK, 0, pol_a);
            tma_load_3d(smem_u32(st + L::kOffD0), &maps.d0, fb, m0, kb * gpc, 0, pol_a);
          }
          if (BM) {
            tma_load_2d(smem_u32(st + L::kOffBRaw), &maps.b, fb, kb * (kPK / 8), n0, pol_w);
            tma_load_2d(smem_u32(st + L::kOffScale), &maps.scales, fb, n0, kb, pol_w);
            tma_load_2d(smem_u32(st + L::kOffBias), &maps.biases, fb, n0, kb, pol_w);
          } else {
            tma_load_2d(smem_u32(st + kAOp), &maps.b, fb, kb * kPK, n0, pol_w);
          }
          ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && kLeaderFull && rank != 0) {
        // this CTA's copies complete on the leader's barriers: give them a fixed bounded time
        p_abort(abort_flag, a.err);
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      } else if (!ok) {
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
    if (lane == 0 && rank == 0) {
      int stage = 0, tile_i = 0;
      uint32_t phase = 0;
      bool ok = true, any = false;
      const uint32_t idesc = make_idesc(false, C::kTileM, NT);
      PSeg g;
      for (int idx = 0; ok && p_seg(a, k_stages, n_tiles, unit, units, idx, g); ++idx, ++tile_i) {
        const int kb0 = g.kb0, kb1 = g.kb1;
        const int ab = tile_i & 1;
        const uint32_t acc_par = static_cast<uint32_t>(tile_i >> 1) & 1u;
        if (!mbar_wait_bounded(smem_u32(&acc_empty[ab]), acc_par ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs) ||
              (C::kProdWarps > 0 &&
               !mbar_wait_bounded(smem_u32(&ready[stage]), phase, abort_flag, kWaitLimitNs))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
          const uint64_t adesc = desc_kmajor_swizzled<128>(sa);
          const uint64_t bdesc = desc_kmajor_swizzled<128>(sa + kAOp);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // 16-element (32-byte) steps along the swizzled row
            if (P)
              mma_f16_pair(tmem_base + static_cast<uint32_t>(ab * NT), adesc + static_cast<uint64_t>(2 * k),
                           bdesc + static_cast<uint64_t>(2 * k), idesc, (kb > kb0 || k > 0) ? 1u : 0u);
            else
              mma_f16(tmem_base + static_cast<uint32_t>(ab * NT), adesc + static_cast<uint64_t>(2 * k),
                      bdesc + static_cast<uint64_t>(2 * k), idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          }
          if (P)
            mma_commit_pair(smem_u32(&empty[stage]), 0x3);  // frees the stage in both CTAs
          else
            mma_commit(smem_u32(&empty[stage]));
          any = true;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (P)
          mma_commit_pair(smem_u32(&acc_full[ab]), 0x3);  // the accumulator is complete in both CTAs
        else
          mma_commit(smem_u32(&acc_full[ab]));
      }
      if (!ok) {
        p_abort(abort_flag, a.err);
        if (any) {
          if (P)
            mma_commit_pair(smem_u32(drain), 0x1);
          else
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
    PSeg g;
    for (int idx = 0; p_seg(a, k_stages, n_tiles, unit, units, idx, g); ++idx, ++tile_i) {
      const int t = g.t, ks = g.ks;
      // stream-K: a later piece of its tile (the partial goes to this CTA's slot), or the owner of a
      // tile whose last k-blocks the CTAs [c_first, c_end) hold
      // (the plan never gives the conv epilogue stream-K shares: that code is compiled out there)
      // (units: CTAs, or pairs whose CTAs of the same rank hand rows over)
      const bool sk_part = !EM && a.stream_k && g.kb0 > 0;
      const int c_first = unit + 1;
      int c_end = c_first;
      if (!EM && a.stream_k && g.kb0 == 0 && g.kb1 < k_stages) {
        const long long total = static_cast<long long>(n_tiles) * k_stages;
        const long long tile_end = static_cast<long long>(t + 1) * k_stages;
        while (c_end < units && total * c_end / units < tile_end) ++c_end;
      }
      const int m0 = (t % a.tiles_m) * C::kTileM + static_cast<int>(rank) * kPM;
      const int n0 = (t / a.tiles_m) * NT;
      const int row = m0 + q * 32 + lane;
      const bool valid = row < a.M;
      const int ab = tile_i & 1;
      const uint32_t acc_par = static_cast<uint32_t>(tile_i >> 1) & 1u;
      const int trow = row % a.G;  // EM: the row's position in its block
      EpiChunk nxt;
      if (EM) load_epi_chunk(nxt, a, valid, row, n0);  // the first chunk's operands, before the wait
      if (!mbar_wait_bounded_suspend(smem_u32(&acc_full[ab]), acc_par, abort_flag, kWaitLimitNs)) {
        if (lane == 0) p_abort(abort_flag, a.err);
        break;
      }
      tc_fence_after();
      if (c_end > c_first) {
        // the later pieces of this quarter's rows (lane 0 acquires; the warp barrier orders the
        // other lanes' loads after it, and those loads bypass L1)
        int got = 1;
        if (lane == 0)
          for (int c2 = c_first; got && c2 < c_end; ++c2)
            got = sk_wait(&g_sk_flags[P ? 2 * c2 + static_cast<int>(rank) : c2][q], abort_flag) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        __syncwarp();
        if (!got) {
          if (lane == 0) p_abort(abort_flag, a.err);
          break;
        }
      }
      for (int cc = 0; cc < NT / 32; ++cc) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(ab * NT + cc * 32),
                           r);
        const int col0 = n0 + cc * 32;
        EpiChunk cur;
        if (EM) {
          cur = nxt;
          if (cc + 1 < NT / 32) load_epi_chunk(nxt, a, valid, row, col0 + 32);  // in flight during this chunk
        }
        tmem_ld_wait();
        float y[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(r[j]);
        if (sk_part) {
          // this CTA's k-blocks of a tile another CTA owns: raw partial sums to its slot
          float* dst = a.part + (static_cast<size_t>(blockIdx.x) * kPM + q * 32 + lane) * NT + cc * 32;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<float4*>(dst + 4 * v) = make_float4(y[4 * v], y[4 * v + 1], y[4 * v + 2], y[4 * v + 3]);
          continue;
        }
        for (int c2 = c_first; c2 < c_end; ++c2) {  // the later k-blocks' partial sums, in K order
          const int cta2 = P ? 2 * c2 + static_cast<int>(rank) : c2;
          const float* src = a.part + (static_cast<size_t>(cta2) * kPM + q * 32 + lane) * NT + cc * 32;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float4 u = __ldcg(reinterpret_cast<const float4*>(src + 4 * v));
            y[4 * v] += u.x;
            y[4 * v + 1] += u.y;
            y[4 * v + 2] += u.z;
            y[4 * v + 3] += u.w;
          }
        }
        if (a.k_splits > 1) {
          // a K range's partial sums; the reduce pass adds them and applies the epilogue
          if (valid) {
            float* dst = a.part + (static_cast<size_t>(ks) * a.M + row) * a.N + col0;
#pragma unroll
            for (int v = 0; v < 8; ++v)
              if (col0 + 4 * v < a.N)
                *reinterpret_cast<float4*>(dst + 4 * v) = make_float4(y[4 * v], y[4 * v + 1], y[4 * v + 2], y[4 * v + 3]);
          }
          continue;
        }
        if (EM) {
          // x = residual + (b10 + d10) y[m] + (b11 + d11) y[m - 1]; y[m - 1] is lane - 1's value
          // (lane 0's row 32w starts a block, as G divides 32)
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float res[8];
            bf16x8_to_f32(cur.res[v], res);
            const bool in = col0 + 8 * v < a.N;
            const float4 b0a = in ? __ldg(reinterpret_cast<const float4*>(a.base + 2 * static_cast<size_t>(a.N) +
                                                                          col0 + 8 * v))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 b0b = in ? __ldg(reinterpret_cast<const float4*>(a.base + 2 * static_cast<size_t>(a.N) +
                                                                          col0 + 8 * v + 4))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 b1a = in ? __ldg(reinterpret_cast<const float4*>(a.base + 3 * static_cast<size_t>(a.N) +
                                                                          col0 + 8 * v))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 b1b = in ? __ldg(reinterpret_cast<const float4*>(a.base + 3 * static_cast<size_t>(a.N) +
                                                                          col0 + 8 * v + 4))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            const float bb0[8] = {b0a.x, b0a.y, b0a.z, b0a.w, b0b.x, b0b.y, b0b.z, b0b.w};
            const float bb1[8] = {b1a.x, b1a.y, b1a.z, b1a.w, b1b.x, b1b.y, b1b.z, b1b.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int j = 8 * v + e;
              float yp = __shfl_up_sync(0xffffffffu, y[j], 1);
              if (lane == 0 || trow == 0) yp = 0.f;
              const int gi = j / a.gs;
              y[j] = res[e] + ((bb0[e] + cur.d[0][gi]) * y[j] + (bb1[e] + cur.d[1][gi]) * yp);
            }
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
      if (lane == 0) {
        if (P)
          mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[ab]), 0));  // the leader's
        else
          mbar_arrive(smem_u32(&acc_empty[ab]));
      }
      if (sk_part) {
        __threadfence();  // every lane's partial rows are visible before the flag
        __syncwarp();
        if (lane == 0) st_release_gpu(&g_sk_flags[blockIdx.x][q], 1);
      }
      if (c_end > c_first && lane == 0)  // read: ready for the next launch
        for (int c2 = c_first; c2 < c_end; ++c2) g_sk_flags[P ? 2 * c2 + static_cast<int>(rank) : c2][q] = 0;
    }
  } else if (AM && warp < 6 + C::kConvWarps) {
    // ------------------------------------------------------------------ conv side-0 producer
    // Thread (rg, c) owns 16-byte chunk c (8 channels, inside one 16-channel group) of the tile rows
    // rg * rpt .. rg * rpt + rpt - 1 (32 row groups over the A box's rows, rpt <= 4), turned in place
    // into A[r, k] = (b00[k] + d00[r]) n[r, k] + (b01[k] + d01[r]) n[r - 1, k] (n[r - 1] = 0 at a
    // block start). Every load of the stage is issued before any arithmetic. The row before a
    // thread's first row belongs to another thread: it is read before the producer warps' barrier,
    // and every write follows it.
    const int pt = threadIdx.x - 192;
    const int c = pt & 7;
    const int rg = pt >> 3;
    const int rpt = (a.a_rows + 31) / 32;
    const int r_first = rg * rpt;
    const int nr = max(0, min(rpt, a.a_rows - r_first));
    const int gi = c >> 1;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    PSeg g;
    for (int idx = 0; ok && p_seg(a, k_stages, n_tiles, unit, units, idx, g); ++idx) {
      const int m0 = (g.t % a.tiles_m) * C::kTileM + static_cast<int>(rank) * kPM;
      const int row_first = m0 + r_first;
      const int t_first = row_first % a.G;
      for (int kb = g.kb0; kb < g.kb1; ++kb) {
        if (!mbar_wait_bounded_suspend(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs, 200)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + stage * C::kStageBytes;
        uint4 raw[5];  // raw[0]: the row before the first; raw[1 + i]: row r_first + i
        raw[0] = (nr > 0 && t_first != 0) ? *reinterpret_cast<const uint4*>(st + sw128(r_first - 1, c))
                                          : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          raw[1 + i] = i < nr ? *reinterpret_cast<const uint4*>(st + sw128(r_first + i, c)) : make_uint4(0u, 0u, 0u, 0u);
        asm volatile("bar.sync 1, 256;" ::: "memory");  // every row this stage needs is read before any write
        if (nr > 0) {
          const float* b0 = reinterpret_cast<const float*>(st + L::kOffBase);  // [2][64]
          const float* d0s = reinterpret_cast<const float*>(st + L::kOffD0);   // [2][4][a_rows]
          const float4 x0 = *reinterpret_cast<const float4*>(b0 + 8 * c);
          const float4 x1 = *reinterpret_cast<const float4*>(b0 + 8 * c + 4);
          const float4 y0 = *reinterpret_cast<const float4*>(b0 + kPK + 8 * c);
          const float4 y1 = *reinterpret_cast<const float4*>(b0 + kPK + 8 * c + 4);
          // the thread's rows' deltas: r_first is a multiple of rpt, and rpt divides 4 when it is 4
          float dd0[4], dd1[4];
          if (rpt == 4) {
            const float4 u0 = *reinterpret_cast<const float4*>(d0s + gi * a.a_rows + r_first);
            const float4 u1 = *reinterpret_cast<const float4*>(d0s + (4 + gi) * a.a_rows + r_first);
            dd0[0] = u0.x; dd0[1] = u0.y; dd0[2] = u0.z; dd0[3] = u0.w;
            dd1[0] = u1.x; dd1[1] = u1.y; dd1[2] = u1.z; dd1[3] = u1.w;
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              dd0[i] = i < nr ? d0s[gi * a.a_rows + r_first + i] : 0.f;
              dd1[i] = i < nr ? d0s[(4 + gi) * a.a_rows + r_first + i] : 0.f;
            }
          }
          const float2 k0[4] = {make_float2(x0.x, x0.y), make_float2(x0.z, x0.w), make_float2(x1.x, x1.y),
                                make_float2(x1.z, x1.w)};
          const float2 k1[4] = {make_float2(y0.x, y0.y), make_float2(y0.z, y0.w), make_float2(y1.x, y1.y),
                                make_float2(y1.z, y1.w)};
          int trow = t_first;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (i < nr) {
              const __nv_bfloat162* hc = reinterpret_cast<const __nv_bfloat162*>(&raw[1 + i]);
              const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&raw[i]);
              const float2 d0p = make_float2(dd0[i], dd0[i]), d1p = make_float2(dd1[i], dd1[i]);
              const float2 keep = trow == 0 ? make_float2(0.f, 0.f) : make_float2(1.f, 1.f);
              uint4 o;
              __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 cur = __bfloat1622float2(hc[e]);
                const float2 prv = __fmul2_rn(__bfloat1622float2(hp[e]), keep);  // 0 at a block start
                const float2 v = __ffma2_rn(__fadd2_rn(k0[e], d0p), cur, __fmul2_rn(__fadd2_rn(k1[e], d1p), prv));
                oh[e] = __floats2bfloat162_rn(v.x, v.y);
              }
              *reinterpret_cast<uint4*>(st + sw128(r_first + i, c)) = o;
              if (++trow == a.G) trow = 0;
            }
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
  } else if (BM) {
    // ------------------------------------------------------------------ W4A16 dequant producer
    // Chunk jobs (row, c): the 8 codes of word c of a weight row become 8 bf16 values
    // scale * q + bias (one rounding of the exact value), a 16-byte chunk of the swizzled operand.
    const int pt = threadIdx.x - 192 - 32 * C::kConvWarps;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    const __nv_bfloat162 k128 = __floats2bfloat162_rn(128.f, 128.f);
    PSeg g;
    for (int idx = 0; ok && p_seg(a, k_stages, n_tiles, unit, units, idx, g); ++idx) {
      for (int kb = g.kb0; kb < g.kb1; ++kb) {
        if (!mbar_wait_bounded_suspend(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs, 200)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + stage * C::kStageBytes;
        const uint32_t* words = reinterpret_cast<const uint32_t*>(st + L::kOffBRaw);  // [NT][8]
        const __nv_bfloat16* sc = reinterpret_cast<const __nv_bfloat16*>(st + L::kOffScale);
        const __nv_bfloat16* bi = reinterpret_cast<const __nv_bfloat16*>(st + L::kOffBias);
#pragma unroll
        for (int i = 0; i < C::kBRows / 32; ++i) {
          const int job = pt + 256 * i;
          const int rr = job >> 3;
          const int c = job & 7;
          const uint32_t w = words[rr * 8 + c];
          const __nv_bfloat162 s2 = __halves2bfloat162(sc[rr], sc[rr]);
          const __nv_bfloat162 b2 = __halves2bfloat162(bi[rr], bi[rr]);
          uint32_t o[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            // bf16 pair (128 + q[2jj], 128 + q[2jj + 1]): 0x4300 | nibble is 128 + nibble exactly
            const uint32_t pair = 0x43004300u | ((w >> (8 * jj)) & 0xFu) | (((w >> (8 * jj + 4)) & 0xFu) << 16);
            __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&pair);
            v = __hsub2(v, k128);      // exact: q
            v = __hfma2(s2, v, b2);    // scale * q + bias, one rounding
            o[jj] = *reinterpret_cast<const uint32_t*>(&v);
          }
          *reinterpret_cast<uint4*>(st + kAOp + sw128(rr, c)) = make_uint4(o[0], o[1], o[2], o[3]);
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
  if (P) {
    cluster_sync_all();  // no MMA, commit or remote arrival is in flight towards either CTA
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem_base, C::kTmemCols);
    }
  } else {
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem_base, C::kTmemCols);
    }
  }
}

// Adds the K ranges' partial sums of a split projection and applies its epilogue: out = y, or
// (EM) out = residual + (b10 + d10) y[m] + (b11 + d11) y[m - 1] with y[m - 1] = 0 at a block start.
// One thread per row and 8 columns (one group: gs >= 8).
template <int EM>
__global__ void __launch_bounds__(256) proj_reduce_kernel(const ProjArgs a) {
  pdl_trigger();
  pdl_wait();
  const int n8 = a.N / 8;
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<size_t>(a.M) * n8) return;
  const int m = static_cast<int>(idx / n8);
  const int c8 = static_cast<int>(idx % n8) * 8;
  const size_t plane = static_cast<size_t>(a.M) * a.N;
  float y[8] = {}, yp[8] = {};
  const bool prev = EM && (m % a.G) != 0;
  for (int s = 0; s < a.k_splits; ++s) {
    const float* p = a.part + s * plane + static_cast<size_t>(m) * a.N + c8;
    const float4 u0 = *reinterpret_cast<const float4*>(p);
    const float4 u1 = *reinterpret_cast<const float4*>(p + 4);
    y[0] += u0.x; y[1] += u0.y; y[2] += u0.z; y[3] += u0.w;
    y[4] += u1.x; y[5] += u1.y; y[6] += u1.z; y[7] += u1.w;
    if (prev) {
      const float4 v0 = *reinterpret_cast<const float4*>(p - a.N);
      const float4 v1 = *reinterpret_cast<const float4*>(p - a.N + 4);
      yp[0] += v0.x; yp[1] += v0.y; yp[2] += v0.z; yp[3] += v0.w;
      yp[4] += v1.x; yp[5] += v1.y; yp[6] += v1.z; yp[7] += v1.w;
    }
  }
  float o[8];
  if (EM) {
    const float d0 = __bfloat162float(a.coef1[(static_cast<size_t>(m) * 2 + 0) * a.groups + c8 / a.gs]);
    const float d1 = __bfloat162float(a.coef1[(static_cast<size_t>(m) * 2 + 1) * a.groups + c8 / a.gs]);
    float res[8] = {};
    if (a.residual != nullptr) bf16x8_to_f32(*reinterpret_cast<const uint4*>(a.residual + static_cast<size_t>(m) * a.N + c8), res);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float b0 = a.base[2 * static_cast<size_t>(a.N) + c8 + e];
      const float b1 = a.base[3 * static_cast<size_t>(a.N) + c8 + e];
      o[e] = res[e] + ((b0 + d0) * y[e] + (b1 + d1) * yp[e]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = y[e];
  }
  *reinterpret_cast<uint4*>(a.out + static_cast<size_t>(m) * a.N + c8) = f32x8_to_bf16(o);
}

// Sums the split-K partial sums of kernel_projection into the side-0 deltas (fp32, [tap][group][row],
// the layout the fused input projection loads) and the side-1 deltas (activation dtype,
// [row][tap][group], as prepare stores them): D[m, side, tap, g] = sum_s part[s][m][(side*2+tap)*groups + g].
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
  d0[(0 * static_cast<size_t>(groups) + g) * M + m] = d[0];
  d0[(1 * static_cast<size_t>(groups) + g) * M + m] = d[1];
  if (sizeof(T) == 2) {
    reinterpret_cast<__nv_bfloat16*>(coef1)[(m * 2 + 0) * groups + g] = __float2bfloat16_rn(d[2]);
    reinterpret_cast<__nv_bfloat16*>(coef1)[(m * 2 + 1) * groups + g] = __float2bfloat16_rn(d[3]);
  } else {
    reinterpret_cast<float*>(coef1)[(m * 2 + 0) * groups + g] = d[2];
    reinterpret_cast<float*>(coef1)[(m * 2 + 1) * groups + g] = d[3];
  }
}

}  // namespace

// CTA pairs of the projection kernel variant that the current device holds at once (0: unknown),
// cached per device.
template <typename K>
int proj_pair_capacity(K* kern, int threads, int smem) {
  constexpr int kMaxDev = 64;
  static int cached[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] != 0) return cached[dev] > 0 ? cached[dev] : 0;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  (void)cudaGetLastError();
  cached[dev] = n > 0 ? n : -1;
  return n > 0 ? n : 0;
}

template <int AM, int BM, int EM, int NT, int P>
static int launch_proj_t(const ProjSpec& p, int k_splits, int sk_ctas, cudaStream_t st) {
  using C = PCfg<AM, BM, EM, NT, P>;
  static_assert(C::kStages >= 2, "at least two pipeline stages");
  ProjMaps maps;
  const int a_rows = std::min(kPM, (p.M + 15) / 16 * 16);  // a small M loads only its own rows
  if (!make_tmap_sw128(&maps.a, p.a, static_cast<uint64_t>(p.M), static_cast<uint64_t>(p.K),
                       static_cast<uint32_t>(a_rows)))
    return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (projection A)");
  maps.b = maps.base = maps.d0 = maps.scales = maps.biases = maps.a;
  if (BM) {
    // packed codes [N][K / 8] 32-bit words: a box of 8 words (64 codes) x the CTA's weight rows;
    // scales and biases [K / 64][N] bf16: a box of those rows' values of one group
    const uint64_t dims[2] = {static_cast<uint64_t>(p.K / 8), static_cast<uint64_t>(p.N)};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.K / 8) * 4};
    const uint32_t box[2] = {8, static_cast<uint32_t>(C::kBRows)};
    const uint64_t sdims[2] = {static_cast<uint64_t>(p.N), static_cast<uint64_t>(p.K / kQGroup)};
    const uint64_t sstr[1] = {static_cast<uint64_t>(p.N) * 2};
    const uint32_t sbox[2] = {static_cast<uint32_t>(C::kBRows), 1};
    if (!make_tmap_plain(&maps.b, p.w, DFLASH2_F32, 2, dims, strides, box) ||
        !make_tmap_plain(&maps.scales, p.scales, DFLASH2_BF16, 2, sdims, sstr, sbox) ||
        !make_tmap_plain(&maps.biases, p.qbias, DFLASH2_BF16, 2, sdims, sstr, sbox))
      return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (4-bit weights)");
  } else if (!make_tmap_sw128(&maps.b, p.w, static_cast<uint64_t>(p.N), static_cast<uint64_t>(p.K), C::kBRows)) {
    return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (projection W)");
  }
  if (AM) {
    // base [2][2][K] fp32 as [4][K]: rows 0, 1 are side 0's taps, a box of 64 channels x 2 rows;
    // d0 [2][groups][M] fp32: a box of the A box's rows x the stage's 4 groups x 2 taps
    const uint64_t dims[2] = {static_cast<uint64_t>(p.K), 4};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.K) * 4};
    const uint32_t box[2] = {static_cast<uint32_t>(kPK), 2};
    const uint64_t ddims[3] = {static_cast<uint64_t>(p.M), static_cast<uint64_t>(p.groups), 2};
    const uint64_t dstr[2] = {static_cast<uint64_t>(p.M) * 4, static_cast<uint64_t>(p.M) * p.groups * 4};
    const uint32_t dbox[3] = {static_cast<uint32_t>(a_rows), static_cast<uint32_t>(kPK / 16), 2};
    if (!make_tmap_plain(&maps.base, p.base, DFLASH2_F32, 2, dims, strides, box) ||
        !make_tmap_plain(&maps.d0, p.d0, DFLASH2_F32, 3, ddims, dstr, dbox))
      return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (conv side 0)");
  }
  ProjArgs args{};
  args.M = p.M;
  args.N = p.N;
  args.K = p.K;
  args.k_splits = k_splits;
  args.stream_k = sk_ctas > 0 ? 1 : 0;
  args.part = p.part;
  args.a_rows = a_rows;
  args.tiles_m = (p.M + C::kTileM - 1) / C::kTileM;
  args.tiles_n = (p.N + NT - 1) / NT;
  args.G = p.G > 0 ? p.G : 1;
  args.gs = p.gs > 0 ? p.gs : 8;
  args.groups = p.groups > 0 ? p.groups : 1;
  args.coef1 = static_cast<const __nv_bfloat16*>(p.coef1);
  args.base = p.base;
  args.residual = static_cast<const __nv_bfloat16*>(p.residual);
  args.out = static_cast<__nv_bfloat16*>(p.out);
  args.err = device_error_word();
  const int items = args.tiles_m * args.tiles_n * k_splits;
  int grid = sk_ctas > 0 ? sk_ctas : std::min(items, sm_count());
  static unsigned done = 0;
  auto kern = proj_kernel<AM, BM, EM, NT, P>;
  if (!ensure_smem_attr(kern, C::kSmem, &done))
    return fail(DFLASH2_ERR_CUDA, "cudaFuncSetAttribute failed (projection)");
  cudaLaunchAttribute cl[1];
  if (P) {
    // every pair of the stream-K shares is resident at once (an owner waits for later pairs)
    const int cap = proj_pair_capacity(kern, C::kThreads, C::kSmem);
    if (cap > 0) grid = std::min(grid, 2 * cap);
    grid &= ~1;
    cl[0].id = cudaLaunchAttributeClusterDimension;
    cl[0].val.clusterDim.x = 2;
    cl[0].val.clusterDim.y = 1;
    cl[0].val.clusterDim.z = 1;
  }
  cudaError_t e = launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmem, st, P ? cl : nullptr, P ? 1 : 0, maps, args);
  if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "projection launch failed: %s", cudaGetErrorString(e));
  if (k_splits > 1) {
    const size_t n = static_cast<size_t>(p.M) * (p.N / 8);
    e = launch_pdl(proj_reduce_kernel<EM>, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, st, nullptr, 0,
                   args);
    if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "projection reduce launch failed: %s", cudaGetErrorString(e));
  }
  return DFLASH2_OK;
}

// Tiles and K splits of a projection. With enough rows every SM gets 256-column tiles. With few
// (the weight-streaming case) the K range is split so that about every SM streams a share of the
// weights through 256-column MMAs, the partial sums going through a workspace and a reduce pass;
// when K is too short to split, 64-column tiles spread the columns instead.
ProjPlan proj_plan(int M, int N, int K, int sms, bool epilogue_conv, bool producers) {
  const long long tiles256 = static_cast<long long>((M + kPM - 1) / kPM) * ((N + 255) / 256);
  const int k_stages = K / kPK;
  if (2 * tiles256 >= sms) {
    // stream-K: every SM gets the same number of k-blocks. Not with side 1 + residual in the
    // epilogue: every stream-K share ends in an owner epilogue that nothing overlaps, and the
    // conv epilogue's loads made that variant slower (103 against 93 us at 1024 x 5120 x 5120).
    if (epilogue_conv) return ProjPlan{256, 1, 0, 0};
    const int cap = std::min(sms, kSkMaxCtas);
    // CTA pairs over 256-row tiles (a third fewer operand bytes per MMA) for the plain projection. With
    // producer warps (side 0 in A, 4-bit dequant) the peer's warps would hand every stage over to the
    // leader with a remote mbarrier arrival: measured at 1024 x 5120 x 5120 that hand-off per stage
    // made the pair kernel twice as slow as single CTAs, so those variants keep single CTAs.
    if (M >= 256 && !producers && DFL_PROJ_PAIR) {
      const long long ptiles = static_cast<long long>((M + 255) / 256) * ((N + 255) / 256);
      return ProjPlan{256, 1, 2 * static_cast<int>(std::min<long long>(cap / 2, ptiles * k_stages)), 1};
    }
    return ProjPlan{256, 1, static_cast<int>(std::min<long long>(cap, tiles256 * k_stages)), 0};
  }
  const int ks = static_cast<int>(std::min<long long>(sms / std::max<long long>(tiles256, 1), k_stages / 4));
  if (ks >= 2) return ProjPlan{256, ks, 0, 0};
  return ProjPlan{64, 1, 0, 0};
}

// Above this many rows a 4-bit weight is dequantised once into the workspace and the projection
// runs on bf16 weights: each weight tile is otherwise dequantised again by every 128-row tile that
// reads it (8 times at 1024 rows), in shared memory the MMA operands also need. Likewise side 0 of
// the conv is applied once to the rows (into the workspace) instead of by every column tile's
// producer warps (20 times at N = 5120).
constexpr int kW4OnceRows = 384;
constexpr int kConvOnceRows = 384;

static size_t proj_w4_scratch_offset(int M, int N, int K, int sms) {
  const ProjPlan pl = proj_plan(M, N, K, sms, false, false);  // the largest workspace of the variants
  size_t b = 0;
  if (pl.ctas > 0)
    b = static_cast<size_t>(pl.ctas) * kPM * 256 * sizeof(float);  // one partial tile per CTA
  else if (pl.k_splits > 1)
    b = static_cast<size_t>(pl.k_splits) * M * N * sizeof(float);
  return (b + 255) & ~static_cast<size_t>(255);
}

// Workspace: [partial-sum slots][bf16 copy of a 4-bit weight (M > kW4OnceRows)][conv side 0 of
// the rows, M x K bf16, or the projection before side 1, M x N bf16 (M > kConvOnceRows)]; the
// query knows neither the weight format nor the fusion, so it counts every part the shape can use.
static size_t proj_conv_scratch_offset(int M, int N, int K, int sms) {
  size_t b = proj_w4_scratch_offset(M, N, K, sms);
  if (M > kW4OnceRows) b += static_cast<size_t>(N) * K * 2;
  return (b + 255) & ~static_cast<size_t>(255);
}

size_t proj_workspace(int M, int N, int K, int sms) {
  if (proj_small_eligible(M, N, K)) return 0;  // the small-row kernel reduces in shared memory
  const size_t off = proj_conv_scratch_offset(M, N, K, sms);
  return M > kConvOnceRows ? off + static_cast<size_t>(M) * std::max(K, N) * 2 : off;
}

// A[m, c] = (base[0][0][c] + d0[0][g][m]) n[m, c] + (base[0][1][c] + d0[1][g][m]) n[m - 1, c] with
// n[m - 1] = 0 at a block's first row (m % G == 0) and g = c / gs: the arithmetic of the conv
// producer warps, rounded once to bf16. Thread = 8 channels of one row.
static __global__ void __launch_bounds__(256) conv0_rows_kernel(const __nv_bfloat16* __restrict__ n,
                                                                const float* __restrict__ d0,
                                                                const float* __restrict__ base, int M, int K, int G,
                                                                int gs, int groups, __nv_bfloat16* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int vpr = K / 8;
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<size_t>(M) * vpr) return;
  const int m = static_cast<int>(idx / vpr);
  const int c = static_cast<int>(idx - static_cast<size_t>(m) * vpr) * 8;
  const int g = c / gs;
  float cur[8], prv[8] = {};
  bf16x8_to_f32(*reinterpret_cast<const uint4*>(n + static_cast<size_t>(m) * K + c), cur);
  if (m % G != 0) bf16x8_to_f32(*reinterpret_cast<const uint4*>(n + static_cast<size_t>(m - 1) * K + c), prv);
  const float dd0 = d0[static_cast<size_t>(g) * M + m];
  const float dd1 = d0[(static_cast<size_t>(groups) + g) * M + m];
  float o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = fmaf(base[c + e] + dd0, cur[e], (base[K + c + e] + dd1) * prv[e]);
  *reinterpret_cast<uint4*>(out + static_cast<size_t>(m) * K + c) = f32x8_to_bf16(o);
}

// W[n, k] = scale[k / 64][n] * q + bias[k / 64][n] as bf16, the same arithmetic as the dequant
// producer warps (0x4300 | q is 128 + q exactly, minus 128, one bf16 FMA). Thread = one 32-bit word
// (8 codes) of one row: reads 4 bytes of codes and writes 16 bytes of W.
static __global__ void __launch_bounds__(256) w4_dequant_kernel(const uint32_t* __restrict__ codes,
                                                         const __nv_bfloat16* __restrict__ scales,
                                                         const __nv_bfloat16* __restrict__ biases, int N, int K,
                                                         __nv_bfloat16* __restrict__ W) {
  pdl_trigger();
  pdl_wait();
  const int wpr = K / 8;  // words per row
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<size_t>(N) * wpr) return;
  const int n = static_cast<int>(idx / wpr);
  const int w = static_cast<int>(idx - static_cast<size_t>(n) * wpr);
  const int g = w >> 3;  // 64 codes per group: 8 words
  const uint32_t word = __ldg(codes + idx);
  const __nv_bfloat16 sc = scales[static_cast<size_t>(g) * N + n];
  const __nv_bfloat16 bi = biases[static_cast<size_t>(g) * N + n];
  const __nv_bfloat162 s2 = __halves2bfloat162(sc, sc);
  const __nv_bfloat162 b2 = __halves2bfloat162(bi, bi);
  const __nv_bfloat162 k128 = __floats2bfloat162_rn(128.f, 128.f);
  uint32_t o[4];
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const uint32_t pair = 0x43004300u | ((word >> (8 * jj)) & 0xFu) | (((word >> (8 * jj + 4)) & 0xFu) << 16);
    __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&pair);
    v = __hsub2(v, k128);    // exact: q
    v = __hfma2(s2, v, b2);  // scale * q + bias, one rounding
    o[jj] = *reinterpret_cast<const uint32_t*>(&v);
  }
  *reinterpret_cast<uint4*>(W + static_cast<size_t>(n) * K + 8 * w) = make_uint4(o[0], o[1], o[2], o[3]);
}

template <int AM, int BM, int EM>
static int launch_proj_nt(const ProjSpec& p, cudaStream_t st) {
  const ProjPlan pl = proj_plan(p.M, p.N, p.K, sm_count(), EM != 0, AM != 0 || BM != 0);
  if (pl.nt == 64) return launch_proj_t<AM, BM, EM, 64, 0>(p, 1, 0, st);
  constexpr int kPairOk = (AM || BM || EM) ? 0 : 1;  // only the plain projection is built in pairs
  if (kPairOk && pl.pair) return launch_proj_t<AM, BM, EM, 256, kPairOk>(p, 1, pl.ctas, st);
  return launch_proj_t<AM, BM, EM, 256, 0>(p, pl.k_splits, pl.ctas, st);
}

int launch_proj(const ProjSpec& p_in, cudaStream_t st) {
  if (proj_small_eligible(p_in.M, p_in.N, p_in.K)) return launch_proj_small(p_in, st);
  ProjSpec p = p_in;
  if (p.wbits == 4 && p.M > kW4OnceRows) {
    // dequantise once into the workspace (after the partial-sum slots), then a bf16 projection
    if (p.part == nullptr) return fail(DFLASH2_ERR_WORKSPACE, "the 4-bit projection at %d rows needs a workspace", p.M);
    __nv_bfloat16* W = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<uint8_t*>(p.part) +
                                                         proj_w4_scratch_offset(p.M, p.N, p.K, sm_count()));
    const size_t words = static_cast<size_t>(p.N) * (p.K / 8);
    const cudaError_t e = launch_pdl(w4_dequant_kernel, dim3(static_cast<unsigned>((words + 255) / 256)), dim3(256), 0,
                                     st, nullptr, 0, static_cast<const uint32_t*>(p.w),
                                     static_cast<const __nv_bfloat16*>(p.scales),
                                     static_cast<const __nv_bfloat16*>(p.qbias), p.N, p.K, W);
    if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "4-bit dequant launch failed: %s", cudaGetErrorString(e));
    p.w = W;
    p.wbits = 16;
    p.scales = p.qbias = nullptr;
  }
  if (p.d0 != nullptr && p.M > kConvOnceRows) {
    // side 0 applied once to the rows (into the workspace), then the projection of those rows
    if (p.part == nullptr) return fail(DFLASH2_ERR_WORKSPACE, "the fused projection at %d rows needs a workspace", p.M);
    __nv_bfloat16* A = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<uint8_t*>(p.part) +
                                                         proj_conv_scratch_offset(p.M, p.N, p.K, sm_count()));
    const size_t items = static_cast<size_t>(p.M) * (p.K / 8);
    const cudaError_t e = launch_pdl(conv0_rows_kernel, dim3(static_cast<unsigned>((items + 255) / 256)), dim3(256), 0,
                                     st, nullptr, 0, static_cast<const __nv_bfloat16*>(p.a), p.d0, p.base, p.M, p.K,
                                     p.G, p.gs, p.groups, A);
    if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "conv side-0 launch failed: %s", cudaGetErrorString(e));
    p.a = A;
    p.d0 = nullptr;
  }
  if (p.coef1 != nullptr && p.M > kConvOnceRows) {
    // the projection into the workspace, then side 1 + residual as the finish pass applies them:
    // the conv epilogue on whole persistent tiles exposes its loads after the last tile round
    if (p.part == nullptr) return fail(DFLASH2_ERR_WORKSPACE, "the fused projection at %d rows needs a workspace", p.M);
    ProjSpec q = p;
    q.coef1 = nullptr;
    q.residual = nullptr;
    q.out = reinterpret_cast<uint8_t*>(p.part) + proj_conv_scratch_offset(p.M, p.N, p.K, sm_count());
    const int rc = q.wbits == 4 ? launch_proj_nt<0, 1, 0>(q, st) : launch_proj_nt<0, 0, 0>(q, st);
    if (rc != DFLASH2_OK) return rc;
    const ConvShape s{p.M / p.G, p.G, p.N, p.gs, p.N / p.gs, DFLASH2_BF16};
    return launch_conv_side1(s, q.out, p.coef1, p.base, p.residual, p.out, nullptr, 0.f, nullptr, 0, st);
  }
  const bool am = p.d0 != nullptr, bm = p.wbits == 4, em = p.coef1 != nullptr;
  if (am && bm && em) return launch_proj_nt<1, 1, 1>(p, st);
  if (am && bm) return launch_proj_nt<1, 1, 0>(p, st);
  if (am && em) return launch_proj_nt<1, 0, 1>(p, st);
  if (bm && em) return launch_proj_nt<0, 1, 1>(p, st);
  if (am) return launch_proj_nt<1, 0, 0>(p, st);
  if (bm) return launch_proj_nt<0, 1, 0>(p, st);
  if (em) return launch_proj_nt<0, 0, 1>(p, st);
  return launch_proj_nt<0, 0, 0>(p, st);
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
