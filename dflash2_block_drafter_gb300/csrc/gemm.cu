// Tensor-core GEMM for sm_103a (tcgen05 + TMEM + TMA), with two epilogues:
//   * STORE: fp32 split-K partial sums (kernel_projection of the grouped conv);
//   * TOPK : per-row running top-16 of the logits (+bias), the extra columns written as z
//            (hidden_projection folded in as 64-row chunks after the vocabulary), optional
//            full logits. Full-vocabulary logits never reach memory unless asked for.
//
// C[m, n] = sum_k A[m, k] * W[n, k]: A = activations [M, K] (rows on the UMMA M axis, 128 per
// tile), W = weights [N, K] (columns on the UMMA N axis, 64-row TMA chunks, up to 256 per
// accumulator tile). Both operands are K-major, staged by TMA with 128-byte swizzle.
//
// Warp roles (one CTA per SM, persistent over its column range):
//   warp 0      : TMA producer (one elected lane)
//   warp 1      : TMEM allocator + MMA issuer (one elected lane)
//   warps 2..   : epilogue, 4 warps per 128-row M tile; warp w reads TMEM lanes 32*(w%4)..+31.
// Every wait is bounded (see mbar_wait_bounded); a timeout raises a CTA-wide abort flag, records
// DFLASH2_ERR_TIMEOUT, drains in-flight copies and MMAs and frees TMEM before returning.
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "warp_keys.cuh"

namespace dfl {
namespace {

// Bytes of K per operand row in one pipeline stage: 128 (128-byte swizzle) or 64 (64-byte
// swizzle, half-size stages, twice as many of them).
#ifndef DFL_GEMM_ROW_BYTES
#define DFL_GEMM_ROW_BYTES 128
#endif
constexpr int kRowBytes = DFL_GEMM_ROW_BYTES;
static_assert(kRowBytes == 128 || kRowBytes == 64, "row bytes per stage must be 64 or 128");
constexpr int kKSteps = kRowBytes / 32;            // 32-byte UMMA K steps per stage
constexpr int kChunk = 64;                         // W rows per TMA box (one column chunk)
constexpr int kMaxTileChunks = 4;                  // 256 accumulator columns per tile
constexpr int kATile = 128 * kRowBytes;            // one 128-row A tile
constexpr int kBChunkBytes = kChunk * kRowBytes;   // one 64-row W chunk
constexpr int kBTile = kMaxTileChunks * kBChunkBytes;
constexpr int kTopL = 16;                          // list length kept per row
constexpr uint64_t kDrainLimitNs = 100000000ull;   // 100 ms
constexpr int kSmemLimit = 232448;

template <int MT>
struct Cfg {
  static constexpr int kStageBytes = MT * kATile + kBTile;
  static constexpr int kEpiWarps = 4 * MT;
  static constexpr int kEpiThreads = 32 * kEpiWarps;
  static constexpr int kThreads = 64 + kEpiThreads;
  // One 128-row M tile fits twice in TMEM (2 x 256 columns): the accumulator is double-buffered
  // and the MMA of the next tile overlaps the epilogue of this one. Two M tiles fill TMEM.
  static constexpr int kAccBufs = MT == 1 ? 2 : 1;
  static constexpr int kTmemCols = 512;
  static constexpr int kBarBytes = 256;
  static constexpr int kBiasBytes = kEpiWarps * 256 * 4;  // one tile's bias per epilogue warp
  // STORE epilogue with one M tile: a 32x33 fp32 transpose tile per epilogue warp, so that partial
  // sums leave as full 128-byte row segments rather than 16-byte pieces of 32 different rows.
  static constexpr int kTransBytes = MT == 1 ? kEpiWarps * 32 * 33 * 4 : 0;
  static constexpr int kFit = (kSmemLimit - 1024 - kBarBytes - kBiasBytes - kTransBytes) / kStageBytes;
  static constexpr int kStages = kFit > 8 ? 8 : kFit;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes + kBiasBytes + kTransBytes;
};
static_assert(Cfg<2>::kStages >= 2 && Cfg<2>::kSmem <= kSmemLimit, "shared memory budget");
static_assert(Cfg<1>::kStages >= 2 && Cfg<1>::kSmem <= kSmemLimit, "shared memory budget");

struct GemmArgs {
  int M, K;
  int n_main, n_extra;
  int main_chunks, n_chunks;
  int main_units, n_units;  // pair head: 128-column units of the vocabulary / of all columns
  int m_groups, n_splits, k_splits, k_blocks;
  float* part;            // STORE: [k_splits][M][n_main]
  const float* bias;      // TOPK: [n_main] or null
  float* list_val;        // TOPK: [n_splits][M][16]
  int* list_idx;
  float* z;               // TOPK: [M][n_extra] or null
  float* logits;          // TOPK: [M][n_main] or null
  int* err;
};

// Next accumulator tile of the chunk range [c, c_end): up to 4 chunks, never straddling the
// boundary between the main and the extra operand.
__device__ __forceinline__ bool next_tile(int& c, int c_end, int main_chunks, int& t0, int& nch) {
  if (c >= c_end) return false;
  t0 = c;
  int e = min(c + kMaxTileChunks, c_end);
  if (t0 < main_chunks && e > main_chunks) e = main_chunks;
  nch = e - t0;
  c = e;
  return true;
}

__device__ __forceinline__ void raise_abort(volatile int* abort_flag, int* err) {
  *abort_flag = 1;
  if (err != nullptr) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_TIMEOUT));
}

// v[j] for a run-time j in [0, 32) without local memory: a 5-level select tree on the bits of j
// (depth 5 instead of a 31-long dependent chain).
__device__ __forceinline__ float select32(const float (&v)[32], int j) {
  float a[16], b[8], c[4], d[2];
#pragma unroll
  for (int k = 0; k < 16; ++k) a[k] = (j & 1) ? v[2 * k + 1] : v[2 * k];
#pragma unroll
  for (int k = 0; k < 8; ++k) b[k] = (j & 2) ? a[2 * k + 1] : a[2 * k];
#pragma unroll
  for (int k = 0; k < 4; ++k) c[k] = (j & 4) ? b[2 * k + 1] : b[2 * k];
#pragma unroll
  for (int k = 0; k < 2; ++k) d[k] = (j & 8) ? c[2 * k + 1] : c[2 * k];
  return (j & 16) ? d[1] : d[0];
}

// Insert (x, id) into a descending 16-entry list held in registers, dropping the last entry.
// Branch-free and fully unrolled; equal values stay behind earlier (lower-id) entries.
__device__ __forceinline__ void list_insert(float (&tv)[kTopL], int (&ti)[kTopL], float x, int id) {
#pragma unroll
  for (int i = kTopL - 1; i >= 1; --i) {
    const bool above = x > tv[i - 1];          // x lands before entry i-1: entry i-1 moves to i
    const bool here = !above && (x > tv[i]);   // x lands exactly at i
    tv[i] = above ? tv[i - 1] : (here ? x : tv[i]);
    ti[i] = above ? ti[i - 1] : (here ? id : ti[i]);
  }
  if (x > tv[0]) {
    tv[0] = x;
    ti[0] = id;
  }
}
// The hidden_projection columns r0..r0+31 of one row, written to z.
__device__ __forceinline__ void store_z32(const uint32_t (&r)[32], int r0, const GemmArgs& a, bool valid, int row) {
  if (valid && a.z != nullptr) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (r0 + j < a.n_extra) a.z[static_cast<size_t>(row) * a.n_extra + r0 + j] = __uint_as_float(r[j]);
  }
}

// Logits of the vocabulary columns col0..col0+31 of one row (accumulator + bias; columns past the
// vocabulary are -inf) into the row's running top-16 (tv, ti); optionally the full logits.
// `sb` holds the bias of these 32 columns in shared memory when col0 + 32 <= n_main.
// Candidates are the values above the row's current 16th: each lane walks its own candidate bits
// while any lane of the warp has one left, re-checking against the threshold as the list fills.
__device__ __forceinline__ void topk_cols32(const uint32_t (&r)[32], int col0, const float* sb, const GemmArgs& a,
                                            bool valid, int row, float (&tv)[kTopL], int (&ti)[kTopL]) {
  float v[32];
  if (col0 + 32 <= a.n_main) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    if (a.bias != nullptr) {
      const float4* bp = reinterpret_cast<const float4*>(sb);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 b4 = bp[q];
        v[4 * q] += b4.x;
        v[4 * q + 1] += b4.y;
        v[4 * q + 2] += b4.z;
        v[4 * q + 3] += b4.w;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int id = col0 + j;
      float x = __uint_as_float(r[j]);
      if (id < a.n_main) {
        if (a.bias != nullptr) x += __ldg(a.bias + id);
      } else {
        x = -INFINITY;
      }
      v[j] = x;
    }
  }
  if (a.logits != nullptr && valid) {
    float* dst = a.logits + static_cast<size_t>(row) * a.n_main;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (col0 + j < a.n_main) dst[col0 + j] = v[j];
  }
  float mx = fmaxf(v[0], v[1]);
#pragma unroll
  for (int j = 2; j < 32; ++j) mx = fmaxf(mx, v[j]);
  const bool any_cand = valid && mx > tv[kTopL - 1];
  if (!__any_sync(0xffffffffu, any_cand)) return;  // the common case once lists fill
  uint32_t cmask = 0u;
  if (any_cand) {
#pragma unroll
    for (int j = 0; j < 32; ++j) cmask |= (v[j] > tv[kTopL - 1] ? 1u : 0u) << j;
  }
  while (__any_sync(0xffffffffu, cmask != 0u)) {
    if (cmask != 0u) {
      const int jj = __ffs(cmask) - 1;
      cmask &= cmask - 1u;
      const float x = select32(v, jj);
      if (x > tv[kTopL - 1]) list_insert(tv, ti, x, col0 + jj);
    }
  }
}

// Stages the bias of the 256 columns from col0 in shared memory (one warp; zero past n_main).
__device__ __forceinline__ void stage_bias256(float* sb, const float* bias, int col0, int n_main, int lane) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i4 = lane + 32 * h;  // float4 index within the tile
    const int col = col0 + 4 * i4;
    float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col + 4 <= n_main) {
      b4 = __ldg(reinterpret_cast<const float4*>(bias + col));
    } else {
      if (col < n_main) b4.x = __ldg(bias + col);
      if (col + 1 < n_main) b4.y = __ldg(bias + col + 1);
      if (col + 2 < n_main) b4.z = __ldg(bias + col + 2);
    }
    reinterpret_cast<float4*>(sb)[i4] = b4;
  }
}

template <int MT, bool TF32, int MODE>
__global__ void __launch_bounds__(Cfg<MT>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmE, const GemmArgs a) {
  using C = Cfg<MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* bar_area = smem + C::kStages * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(bar_area);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;     // [kAccBufs]
  uint64_t* acc_empty = acc_full + C::kAccBufs;  // [kAccBufs]
  uint64_t* drain = acc_empty + C::kAccBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* sbias_all = reinterpret_cast<float*>(bar_area + C::kBarBytes);
  float* strans_all = reinterpret_cast<float*>(bar_area + C::kBarBytes + C::kBiasBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int bid = blockIdx.x;
  const int mg = bid % a.m_groups;
  bid /= a.m_groups;
  const int ns = bid % a.n_splits;
  const int ks = bid / a.n_splits;
  const int c_begin = static_cast<int>((static_cast<long long>(a.n_chunks) * ns) / a.n_splits);
  const int c_end = static_cast<int>((static_cast<long long>(a.n_chunks) * (ns + 1)) / a.n_splits);
  const int kb0 = static_cast<int>((static_cast<long long>(a.k_blocks) * ks) / a.k_splits);
  const int kb1 = static_cast<int>((static_cast<long long>(a.k_blocks) * (ks + 1)) / a.k_splits);
  const int row0 = mg * 128 * MT;
  const int mt_valid = min(MT, (a.M - row0 + 127) / 128);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), C::kEpiWarps);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (a.n_extra > 0) prefetch_tmap(&tmE);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();
  // The weight tiles of the first stages are requested before the wait on the preceding kernel
  // (weights are never an output of the kernels this one overlaps); the activations follow.
  int w_pre = 0;
  const uint64_t pol_keep = policy_evict_last();    // activations: re-read by every column tile
  const uint64_t pol_stream = policy_evict_first(); // weights: streamed
  if (warp == 0 && lane == 0) {
    int c = c_begin, t0 = 0, nch = 0;
    if (next_tile(c, c_end, a.main_chunks, t0, nch)) {
      w_pre = min(C::kStages, kb1 - kb0);
      for (int i = 0; i < w_pre; ++i) {
        const uint32_t fb = smem_u32(&full[i]);
        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(mt_valid * kATile + nch * kBChunkBytes));
        uint8_t* sb = smem + i * C::kStageBytes + MT * kATile;
        const int kx = (kb0 + i) * (kRowBytes / (TF32 ? 4 : 2));
        for (int j = 0; j < nch; ++j) {
          const int ch = t0 + j;
          if (ch < a.main_chunks)
            tma_load_2d(smem_u32(sb + j * kBChunkBytes), &tmB, fb, kx, ch * kChunk, pol_stream);
          else
            tma_load_2d(smem_u32(sb + j * kBChunkBytes), &tmE, fb, kx, (ch - a.main_chunks) * kChunk, pol_keep);
        }
      }
    }
  }
  pdl_wait();  // no global memory but the weights is touched above this line

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      int c = c_begin, t0 = 0, nch = 0;
      while (ok && next_tile(c, c_end, a.main_chunks, t0, nch)) {
        for (int kb = kb0; kb < kb1; ++kb) {
          // the first tile's first w_pre stages: fresh barriers, byte count and weights already set
          const bool pre = issued < w_pre;
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          if (!pre) mbar_arrive_expect_tx(fb, static_cast<uint32_t>(mt_valid * kATile + nch * kBChunkBytes));
          uint8_t* sa = smem + stage * C::kStageBytes;
          uint8_t* sb = sa + MT * kATile;
          const int kx = kb * (kRowBytes / (TF32 ? 4 : 2));
          for (int mt = 0; mt < mt_valid; ++mt)
            tma_load_2d(smem_u32(sa + mt * kATile), &tmA, fb, kx, row0 + mt * 128, pol_keep);
          for (int j = 0; !pre && j < nch; ++j) {
            const int ch = t0 + j;
            if (ch < a.main_chunks)
              tma_load_2d(smem_u32(sb + j * kBChunkBytes), &tmB, fb, kx, ch * kChunk, pol_stream);
            else
              tma_load_2d(smem_u32(sb + j * kBChunkBytes), &tmE, fb, kx, (ch - a.main_chunks) * kChunk, pol_keep);
          }
          ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        raise_abort(abort_flag, a.err);
        // Wait for the copies still in flight (the last min(issued, stages) fills).
        int s = stage;
        uint32_t ph = phase;
        const int n = min(issued, C::kStages);
        for (int i = 0; i < n; ++i) {
          if (s == 0) {
            s = C::kStages - 1;
            ph ^= 1u;
          } else {
            --s;
          }
          mbar_wait_bounded(smem_u32(&full[s]), ph, nullptr, kDrainLimitNs);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int tile_i = 0;
      bool ok = true, any = false;
      int c = c_begin, t0 = 0, nch = 0;
      while (ok && next_tile(c, c_end, a.main_chunks, t0, nch)) {
        const int ab = tile_i % C::kAccBufs;                       // accumulator buffer of this tile
        const uint32_t acc_par = static_cast<uint32_t>(tile_i / C::kAccBufs) & 1u;
        const uint32_t acc_col = static_cast<uint32_t>(ab * 256);
        if (!mbar_wait_bounded(smem_u32(&acc_empty[ab]), acc_par ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t idesc = make_idesc(TF32, 128, nch * kChunk);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
          const uint64_t bdesc = desc_kmajor_swizzled<kRowBytes>(sa + MT * kATile);
#pragma unroll
          for (int k = 0; k < kKSteps; ++k) {  // 32-byte K steps along the swizzled row
            for (int mt = 0; mt < mt_valid; ++mt) {
              const uint64_t adesc = desc_kmajor_swizzled<kRowBytes>(sa + mt * kATile) + static_cast<uint64_t>(2 * k);
              const uint32_t acc = (kb > kb0 || k > 0) ? 1u : 0u;
              if (TF32)
                mma_tf32(tmem_base + acc_col + static_cast<uint32_t>(mt * 256), adesc, bdesc + static_cast<uint64_t>(2 * k),
                         idesc, acc);
              else
                mma_f16(tmem_base + acc_col + static_cast<uint32_t>(mt * 256), adesc, bdesc + static_cast<uint64_t>(2 * k),
                        idesc, acc);
            }
          }
          mma_commit(smem_u32(&empty[stage]));  // frees the stage once these MMAs have read it
          any = true;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&acc_full[ab]));  // accumulator complete
        ++tile_i;
      }
      if (!ok) {
        raise_abort(abort_flag, a.err);
        if (any) {
          mma_commit(smem_u32(drain));
          mbar_wait_bounded(smem_u32(drain), 0, nullptr, kDrainLimitNs);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    const int e = warp - 2;
    const int q = warp & 3;
    const int mt = e >> 2;
    const int row = row0 + mt * 128 + q * 32 + lane;
    const bool tile_ok = mt < mt_valid;
    const bool valid = tile_ok && row < a.M;
    int tile_i = 0;
    float tv[kTopL];  // this row's running top-16 (descending), tv[15] is the admission threshold
    int ti[kTopL];
#pragma unroll
    for (int i = 0; i < kTopL; ++i) {
      tv[i] = -INFINITY;
      ti[i] = -1;
    }
    float* sbias = sbias_all + e * 256;  // this warp's copy of the tile's bias
    int c = c_begin, t0 = 0, nch = 0;
    while (next_tile(c, c_end, a.main_chunks, t0, nch)) {
      const int ab = tile_i % C::kAccBufs;
      const uint32_t acc_par = static_cast<uint32_t>(tile_i / C::kAccBufs) & 1u;
      const uint32_t acc_col = static_cast<uint32_t>(ab * 256);
      // Stage the tile's bias in shared memory before waiting for the accumulator, so its global
      // load latency hides behind the mainloop (each 32-column chunk would otherwise miss L1).
      if (MODE == 1 && a.bias != nullptr && t0 < a.main_chunks) {
        __syncwarp();
        stage_bias256(sbias, a.bias, t0 * kChunk, a.n_main, lane);
        __syncwarp();
      }
      if (!mbar_wait_bounded(smem_u32(&acc_full[ab]), acc_par, abort_flag, kWaitLimitNs)) {
        if (lane == 0) raise_abort(abort_flag, a.err);
        break;
      }
      tc_fence_after();
      if (tile_ok) {
        const bool extra = t0 >= a.main_chunks;
        for (int cc = 0; cc < nch * 2; ++cc) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(
              tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc_col + static_cast<uint32_t>(mt * 256 + cc * 32), r);
          tmem_ld_wait();
          const int col0 = t0 * kChunk + cc * 32;
          if (MODE == 0 && MT == 1) {
            // lane l holds row (row - lane + l); transpose through shared memory and write each
            // row's 32 columns as one 128-byte segment
            float* tr = strans_all + e * (32 * 33);
#pragma unroll
            for (int j = 0; j < 32; ++j) tr[lane * 33 + j] = __uint_as_float(r[j]);
            __syncwarp();
            const int rbase = row - lane;
            const int col = col0 + lane;
            float* base_ptr = a.part + static_cast<size_t>(ks) * a.M * a.n_main;
#pragma unroll 8
            for (int rr = 0; rr < 32; ++rr) {
              const int rrow = rbase + rr;
              if (tile_ok && rrow < a.M && col < a.n_main)
                base_ptr[static_cast<size_t>(rrow) * a.n_main + col] = tr[rr * 33 + lane];
            }
            __syncwarp();
          } else if (MODE == 0) {
            if (valid) {
              float* dst = a.part + (static_cast<size_t>(ks) * a.M + row) * a.n_main + col0;
              if (col0 + 32 <= a.n_main && (a.n_main & 3) == 0) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                  *reinterpret_cast<float4*>(dst + j) =
                      make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                                  __uint_as_float(r[j + 3]));
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (col0 + j < a.n_main) dst[j] = __uint_as_float(r[j]);
              }
            }
          } else if (extra) {
            store_z32(r, col0 - a.main_chunks * kChunk, a, valid, row);
          } else {
            topk_cols32(r, col0, sbias + cc * 32, a, valid, row, tv, ti);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
      ++tile_i;
    }
    if (MODE == 1 && valid && *abort_flag == 0) {
      const size_t o = (static_cast<size_t>(ns) * a.M + row) * kTopL;
      for (int i = 0; i < kTopL; ++i) {
        a.list_val[o + i] = tv[i];
        a.list_idx[o + i] = ti[i];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------------------------ CTA-pair GEMM
// The GEMM on pairs of CTAs: a two-CTA cluster computes 256 rows x up to 256 columns per tile
// with one pair MMA (cta_group::2, M = 256). Each CTA stages its own 128 activation rows and half
// of the tile's weight rows, so a 32 KB stage per SM feeds the work a 64 KB stage fed a
// two-M-tile CTA, and each CTA's accumulator (its 128 rows x 256 columns) fits in TMEM twice: the
// epilogue of one tile overlaps the MMAs of the next. Epilogues as in tc_gemm_kernel: TOPK (the
// head) and STORE (split-K fp32 partials of kernel_projection, written by TMA from swizzled
// shared-memory tiles).
//
// Columns go in 128-column units (two 64-row TMA chunks of one operand); a tile is one or two
// units of the same operand. Of a tile of n units the leader loads the first n chunks and the
// peer the next n (the pair MMA takes B's first half from the leader, the second from the peer).
//
// Barriers: full[s] is the leader's (armed by the leader with both CTAs' bytes; the peer's copies
// complete on it across the cluster); empty[s] and acc_full[b] exist in both CTAs (the leader's
// commits arrive on both); acc_empty[b] is the leader's (4 epilogue warps from each CTA).

// L2 policy of the weight stream (0: evict_first, 1: evict_normal, 2: evict_last) and where the
// head epilogue reads the bias from (1: a per-warp copy in shared memory, 0: global memory
// through L1, which leaves room for a seventh stage).
#ifndef DFL_PAIR_WPOL
#define DFL_PAIR_WPOL 1
#endif
#ifndef DFL_PAIR_SMEM_BIAS
#define DFL_PAIR_SMEM_BIAS 1
#endif

template <int MODE>
struct PairCfg {
  static constexpr int kStageBytes = kATile + 2 * kBChunkBytes;
  static constexpr int kEpiWarps = 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kAccBufs = 2;
  static constexpr int kTmemCols = 512;
  static constexpr int kBarBytes = 256;
  static constexpr int kBiasBytes = (MODE == 1 && DFL_PAIR_SMEM_BIAS) ? kEpiWarps * 256 * 4 : 0;
  // STORE: 32x32 fp32 staging tiles (128-byte swizzled rows), eight per epilogue warp (one per
  // 32-column chunk of a two-unit tile), carved out of the stage ring once the accumulator is ready
  static constexpr int kOutTile = 32 * 32 * 4;
  static constexpr int kOutPerWarp = 8;
  static constexpr int kFit = (kSmemLimit - 1024 - kBarBytes - kBiasBytes) / kStageBytes;
  static constexpr int kStages = kFit > 8 ? 8 : kFit;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes + kBiasBytes;
};
static_assert(PairCfg<1>::kStages >= 2 && PairCfg<1>::kSmem <= kSmemLimit, "shared memory budget (pair, head)");
static_assert(PairCfg<0>::kStageBytes % 1024 == 0 && PairCfg<0>::kOutTile % 1024 == 0, "staging tile alignment");
static_assert(PairCfg<0>::kEpiWarps * PairCfg<0>::kOutPerWarp * PairCfg<0>::kOutTile <=
                  PairCfg<0>::kStages * PairCfg<0>::kStageBytes,
              "STORE staging tiles fit in the stage ring");
static_assert(PairCfg<0>::kStages >= 2 && PairCfg<0>::kSmem <= kSmemLimit, "shared memory budget (pair, store)");
static_assert((2 * PairCfg<1>::kStages + 2 * PairCfg<1>::kAccBufs + 1) * 8 + 8 <= PairCfg<1>::kBarBytes, "barriers");
static_assert((2 * PairCfg<0>::kStages + 2 * PairCfg<0>::kAccBufs + 1) * 8 + 8 <= PairCfg<0>::kBarBytes, "barriers");

// Next tile of the unit range [u, u_end): up to 2 units, never straddling the operand boundary.
__device__ __forceinline__ bool next_unit_tile(int& u, int u_end, int main_units, int& u0, int& nu) {
  if (u >= u_end) return false;
  u0 = u;
  int e = min(u + 2, u_end);
  if (u0 < main_units && e > main_units) e = main_units;
  nu = e - u0;
  u = e;
  return true;
}

__device__ __forceinline__ void raise_abort_pair(volatile int* abort_flag, uint32_t peer_flag, int* err) {
  *abort_flag = 1;
  st_shared_cluster_u32(peer_flag, 1u);
  if (err != nullptr) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_TIMEOUT));
}

template <bool TF32, int MODE>
__global__ void __launch_bounds__(PairCfg<MODE>::kThreads, 1)
    tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmE, const __grid_constant__ CUtensorMap tmD, const GemmArgs a) {
  using C = PairCfg<MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  // layout: stages | barriers | bias. STORE stages its output tiles in the stage ring: a STORE pair
  // computes exactly one tile (the launcher checks), so once that accumulator is complete every
  // stage has been consumed by the MMAs and no further load is issued.
  uint8_t* bar_area = smem + C::kStages * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(bar_area);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + C::kAccBufs;
  uint64_t* drain = acc_empty + C::kAccBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* sbias_all = reinterpret_cast<float*>(bar_area + C::kBarBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: leader (issues the MMAs), 1: peer
  const uint32_t peer_abort = mapa_shared(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u);
  int pair = static_cast<int>(blockIdx.x >> 1);
  const int mg = pair % a.m_groups;
  pair /= a.m_groups;
  const int ns = pair % a.n_splits;
  const int ks = pair / a.n_splits;
  const int u_begin = static_cast<int>((static_cast<long long>(a.n_units) * ns) / a.n_splits);
  const int u_end = static_cast<int>((static_cast<long long>(a.n_units) * (ns + 1)) / a.n_splits);
  const int kb0 = static_cast<int>((static_cast<long long>(a.k_blocks) * ks) / a.k_splits);
  const int kb1 = static_cast<int>((static_cast<long long>(a.k_blocks) * (ks + 1)) / a.k_splits);
  const int rowA = mg * 256 + static_cast<int>(rank) * 128;  // this CTA's 128 activation rows

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 2 * C::kEpiWarps);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (a.n_extra > 0) prefetch_tmap(&tmE);
    if (MODE == 0) prefetch_tmap(&tmD);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers are initialised before anything arrives on them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();
  // The weight tiles of the first stages are requested before the wait on the preceding kernel:
  // weights are never an output of the kernels this one overlaps, and their loads (from HBM) then
  // run under that kernel's tail. The activation tiles follow after the wait.
  int w_pre = 0;
  const uint64_t pol_keep = policy_evict_last();  // activations: re-read by every column tile
  // weights: streamed, but read by the pairs of every row group
  const uint64_t pol_stream = DFL_PAIR_WPOL == 0 ? policy_evict_first()
                              : DFL_PAIR_WPOL == 1 ? policy_evict_normal() : policy_evict_last();
  if (warp == 0 && lane == 0) {
    int u = u_begin, u0 = 0, nu = 0;
    if (next_unit_tile(u, u_end, a.main_units, u0, nu)) {
      const bool extra = u0 >= a.main_units;
      const CUtensorMap* mw = extra ? &tmE : &tmB;
      const int wrow0 = (extra ? u0 - a.main_units : u0) * 128 + static_cast<int>(rank) * nu * kChunk;
      const uint32_t cta_bytes = static_cast<uint32_t>(kATile + nu * kBChunkBytes);
      w_pre = min(C::kStages, kb1 - kb0);
      for (int i = 0; i < w_pre; ++i) {
        const uint32_t fb_own = smem_u32(&full[i]);
        const uint32_t fb = mapa_shared(fb_own, 0);  // the leader's full barrier
        if (rank == 0) mbar_arrive_expect_tx(fb_own, 2 * cta_bytes);
        uint8_t* sb = smem + i * C::kStageBytes + kATile;
        const int kx = (kb0 + i) * (kRowBytes / (TF32 ? 4 : 2));
        for (int j = 0; j < nu; ++j)
          tma_load_2d_pair(smem_u32(sb + j * kBChunkBytes), mw, fb, kx, wrow0 + j * kChunk, extra ? pol_keep : pol_stream);
      }
    }
  }
  pdl_wait();  // no global memory but the weights is touched above this line

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      int u = u_begin, u0 = 0, nu = 0;
      while (ok && next_unit_tile(u, u_end, a.main_units, u0, nu)) {
        const bool extra = u0 >= a.main_units;
        const CUtensorMap* mw = extra ? &tmE : &tmB;
        const uint64_t pol_w = extra ? pol_keep : pol_stream;
        const int wrow0 = (extra ? u0 - a.main_units : u0) * 128 + static_cast<int>(rank) * nu * kChunk;
        const uint32_t cta_bytes = static_cast<uint32_t>(kATile + nu * kBChunkBytes);
        for (int kb = kb0; kb < kb1; ++kb) {
          // the first tile's first w_pre stages: fresh barriers, byte count and weights already set
          const bool pre = issued < w_pre;
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t fb_own = smem_u32(&full[stage]);
          const uint32_t fb = mapa_shared(fb_own, 0);  // the leader's full barrier
          if (rank == 0 && !pre) mbar_arrive_expect_tx(fb_own, 2 * cta_bytes);
          uint8_t* sa = smem + stage * C::kStageBytes;
          uint8_t* sb = sa + kATile;
          const int kx = kb * (kRowBytes / (TF32 ? 4 : 2));
          tma_load_2d_pair(smem_u32(sa), &tmA, fb, kx, rowA, pol_keep);
          if (!pre)
            for (int j = 0; j < nu; ++j)
              tma_load_2d_pair(smem_u32(sb + j * kBChunkBytes), mw, fb, kx, wrow0 + j * kChunk, pol_w);
          ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every stage released: all of the leader's commits towards this CTA have landed.
      for (int i = 0; ok && i < C::kStages; ++i) {
        if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) ok = false;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        raise_abort_pair(abort_flag, peer_abort, a.err);
        if (rank == 0) {
          // Wait for the fills still in flight (they count both CTAs' bytes).
          int s = stage;
          uint32_t ph = phase;
          const int n = min(issued, C::kStages);
          for (int i = 0; i < n; ++i) {
            if (s == 0) {
              s = C::kStages - 1;
              ph ^= 1u;
            } else {
              --s;
            }
            mbar_wait_bounded(smem_u32(&full[s]), ph, nullptr, kDrainLimitNs);
          }
        } else {
          // The peer's copies complete on the leader's barriers: give them a fixed bounded time.
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 2000000ull) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ pair MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int tile_i = 0;
      bool ok = true, any = false;
      int u = u_begin, u0 = 0, nu = 0;
      while (ok && next_unit_tile(u, u_end, a.main_units, u0, nu)) {
        const int ab = tile_i & 1;
        const uint32_t acc_par = static_cast<uint32_t>(tile_i >> 1) & 1u;
        const uint32_t acc_col = static_cast<uint32_t>(ab * 256);
        if (!mbar_wait_bounded(smem_u32(&acc_empty[ab]), acc_par ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t idesc = make_idesc(TF32, 256, nu * 128);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
          const uint64_t adesc = desc_kmajor_swizzled<kRowBytes>(sa);
          const uint64_t bdesc = desc_kmajor_swizzled<kRowBytes>(sa + kATile);
#pragma unroll
          for (int k = 0; k < kKSteps; ++k) {  // 32-byte K steps along the swizzled row
            const uint32_t acc = (kb > kb0 || k > 0) ? 1u : 0u;
            if (TF32)
              mma_tf32_pair(tmem_base + acc_col, adesc + static_cast<uint64_t>(2 * k),
                            bdesc + static_cast<uint64_t>(2 * k), idesc, acc);
            else
              mma_f16_pair(tmem_base + acc_col, adesc + static_cast<uint64_t>(2 * k),
                           bdesc + static_cast<uint64_t>(2 * k), idesc, acc);
          }
          mma_commit_pair(smem_u32(&empty[stage]), 0x3);  // frees the stage in both CTAs
          any = true;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(smem_u32(&acc_full[ab]), 0x3);  // accumulator complete in both CTAs
        ++tile_i;
      }
      if (!ok) {
        raise_abort_pair(abort_flag, peer_abort, a.err);
        if (any) {
          mma_commit_pair(smem_u32(drain), 0x1);
          mbar_wait_bounded(smem_u32(drain), 0, nullptr, kDrainLimitNs);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int e = warp - 2;
    const int q = warp & 3;
    const int row = rowA + q * 32 + lane;
    const bool valid = row < a.M;
    float tv[kTopL];
    int ti[kTopL];
#pragma unroll
    for (int i = 0; i < kTopL; ++i) {
      tv[i] = -INFINITY;
      ti[i] = -1;
    }
    float* sbias = sbias_all + e * 256;
    uint8_t* sout = smem + e * C::kOutPerWarp * C::kOutTile;  // STORE: this warp's staging tiles
    int tile_i = 0;
    int u = u_begin, u0 = 0, nu = 0;
    while (next_unit_tile(u, u_end, a.main_units, u0, nu)) {
      const int ab = tile_i & 1;
      const uint32_t acc_par = static_cast<uint32_t>(tile_i >> 1) & 1u;
      const uint32_t acc_col = static_cast<uint32_t>(ab * 256);
      const bool extra = u0 >= a.main_units;
      if (MODE == 1 && DFL_PAIR_SMEM_BIAS && a.bias != nullptr && !extra) {
        __syncwarp();
        stage_bias256(sbias, a.bias, u0 * 128, a.n_main, lane);
        __syncwarp();
      }
      if (!mbar_wait_bounded(smem_u32(&acc_full[ab]), acc_par, abort_flag, kWaitLimitNs)) {
        if (lane == 0) raise_abort_pair(abort_flag, peer_abort, a.err);
        break;
      }
      tc_fence_after();
      for (int cc = 0; cc < nu * 4; ++cc) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc_col + static_cast<uint32_t>(cc * 32),
                           r);
        tmem_ld_wait();
        if (MODE == 0) {
          // This warp's 32 rows x 32 columns of the partial sum: into a staging tile laid out as
          // the tensor map's 128-byte swizzle expects (16-byte unit j of row i at unit j ^ (i % 8),
          // so the eight lanes of a store phase hit eight different units), then one TMA store.
          // Boxes that start past the last row or column are not stored (warp-uniform test). Each
          // chunk has a staging tile of its own, so no store waits for an earlier one.
          const int col0 = u0 * 128 + cc * 32;
          const int row0 = rowA + q * 32;
          if (row0 < a.M && col0 < a.n_main) {
            uint8_t* tile = sout + cc * C::kOutTile;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<float4*>(tile + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                  make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                              __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmD, smem_u32(tile), col0, row0, ks);
              bulk_commit_group();
            }
          }
        } else if (extra) {
          store_z32(r, (u0 - a.main_units) * 128 + cc * 32, a, valid, row);
        } else {
          topk_cols32(r, u0 * 128 + cc * 32, DFL_PAIR_SMEM_BIAS ? sbias + cc * 32 : a.bias + u0 * 128 + cc * 32, a,
                      valid, row, tv, ti);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[ab]), 0));
      ++tile_i;
    }
    if (MODE == 0) {
      if (lane == 0) bulk_wait_group_all();  // partial sums written before the CTA retires
      __syncwarp();
    }
    if (MODE == 1 && valid && *abort_flag == 0) {
      const size_t o = (static_cast<size_t>(ns) * a.M + row) * kTopL;
      for (int i = 0; i < kTopL; ++i) {
        a.list_val[o + i] = tv[i];
        a.list_idx[o + i] = ti[i];
      }
    }
  }

  // Nothing is in flight towards either CTA past this point (stages released, accumulators read,
  // remote arrivals made before the barrier), so the pair can free TMEM and exit.
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------------------------ top-K merge


// The list of split `s` for `row` (sorted, value desc / id asc) into a lane's registers; empty slots
// (id -1) become (-inf, INT_MAX) so that they lose every tie.
__device__ __forceinline__ void load_list(const float* lv, const int* li, int s, int M, int row, float (&tv)[kTopL],
                                          int (&ti)[kTopL]) {
  const size_t o = (static_cast<size_t>(s) * M + row) * kTopL;
#pragma unroll
  for (int q = 0; q < kTopL / 4; ++q) {  // the whole sorted list in 8 vector loads
    const float4 f = __ldg(reinterpret_cast<const float4*>(lv + o) + q);
    const int4 n = __ldg(reinterpret_cast<const int4*>(li + o) + q);
    const float fv[4] = {f.x, f.y, f.z, f.w};
    const int nv[4] = {n.x, n.y, n.z, n.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      tv[4 * q + e] = nv[e] >= 0 ? fv[e] : -INFINITY;
      ti[4 * q + e] = nv[e] >= 0 ? nv[e] : INT_MAX;
    }
  }
}

__device__ __forceinline__ void empty_list(float (&tv)[kTopL], int (&ti)[kTopL]) {
#pragma unroll
  for (int i = 0; i < kTopL; ++i) {
    tv[i] = -INFINITY;
    ti[i] = INT_MAX;
  }
}

// K-way merge of the lanes' sorted lists (one per lane; ids unique across lanes): round k takes the
// best head over the warp (value desc, id asc) with two warp reductions and its owner pops it.
// Every lane sees the K results in order through `emit(k, value, id)`.
template <typename Emit>
__device__ __forceinline__ void warp_merge_lists(float (&tv)[kTopL], int (&ti)[kTopL], int K, Emit emit) {
  for (int k = 0; k < K; ++k) {
    // best head: the warp's largest value key, then the smallest id among the lanes holding it
    const uint32_t key = float_key(tv[0]);
    uint32_t kmax, imin;
    warp_max_min_index(key, true, static_cast<uint32_t>(ti[0]), kmax, imin);
    const int bi = static_cast<int>(imin);
    emit(k, key_float(kmax), bi);
    if (key == kmax && ti[0] == bi) {
#pragma unroll
      for (int j = 0; j < kTopL - 1; ++j) {
        tv[j] = tv[j + 1];
        ti[j] = ti[j + 1];
      }
      tv[kTopL - 1] = -INFINITY;
      ti[kTopL - 1] = INT_MAX;
    }
  }
}

// Up to 32 splits: one warp per row, lane s holding split s's list.
// `ids_map` (nullable): token id of each column when the head ran over a draft vocabulary.
__global__ void __launch_bounds__(256) topk_merge_kernel(const float* __restrict__ lv, const int* __restrict__ li,
                                                         int n_splits, int M, int K, const int32_t* __restrict__ ids_map,
                                                         int32_t* __restrict__ cand, float* __restrict__ unary) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  float tv[kTopL];
  int ti[kTopL];
  if (lane < n_splits)
    load_list(lv, li, lane, M, row, tv, ti);
  else
    empty_list(tv, ti);
  warp_merge_lists(tv, ti, K, [&](int k, float v, int id) {
    if (lane == 0) {
      cand[static_cast<size_t>(row) * K + k] = ids_map != nullptr ? __ldg(ids_map + id) : id;
      unary[static_cast<size_t>(row) * K + k] = v;
    }
  });
}

// 33 to 512 splits: one CTA of W <= 16 warps per row. Warp w merges splits w, w + W, ... (at most 32)
// into its top-16 in shared memory; warp 0 then merges the W lists into the row's top-K.
__global__ void __launch_bounds__(512) topk_merge_wide_kernel(const float* __restrict__ lv,
                                                               const int* __restrict__ li, int n_splits, int M, int K,
                                                               const int32_t* __restrict__ ids_map,
                                                               int32_t* __restrict__ cand, float* __restrict__ unary) {
  __shared__ float sv[32][kTopL];
  __shared__ int si[32][kTopL];
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x;
  const int W = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  float tv[kTopL];
  int ti[kTopL];
  const int s = warp + W * lane;
  if (s < n_splits)
    load_list(lv, li, s, M, row, tv, ti);
  else
    empty_list(tv, ti);
  warp_merge_lists(tv, ti, kTopL, [&](int k, float v, int id) {
    if (lane == 0) {
      sv[warp][k] = v;
      si[warp][k] = id;
    }
  });
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int i = 0; i < kTopL; ++i) {
    tv[i] = lane < W ? sv[lane][i] : -INFINITY;
    ti[i] = lane < W ? si[lane][i] : INT_MAX;
  }
  warp_merge_lists(tv, ti, K, [&](int k, float v, int id) {
    if (lane == 0) {
      cand[static_cast<size_t>(row) * K + k] = ids_map != nullptr ? __ldg(ids_map + id) : id;
      unary[static_cast<size_t>(row) * K + k] = v;
    }
  });
}

// One thread waits on an mbarrier that nothing completes; the bounded wait gives up.
__global__ void wait_selftest_kernel(uint64_t limit_ns, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  if (!mbar_wait_bounded(smem_u32(&bar), 0, nullptr, limit_ns)) atomicCAS(err, 0, static_cast<int>(DFLASH2_ERR_TIMEOUT));
}

// ------------------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Row-major [rows, cols] operand, box = kRowBytes of K x box_rows rows, swizzled to match.
bool make_map(CUtensorMap* m, const void* ptr, int dtype, int rows, int cols, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const int es = dtype == DFLASH2_F32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * es};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kRowBytes / es), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, dtype == DFLASH2_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         kRowBytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Split-K partial sums [k_splits][rows][cols] fp32 as a 3D map for TMA stores of 32 x 32 boxes
// with 128-byte swizzle (the pair GEMM's STORE epilogue). Rows past `rows` in a box are clipped
// per split.
bool make_part_map(CUtensorMap* m, float* part, int k_splits, int rows, int cols) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(k_splits)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 4, static_cast<cuuint64_t>(rows) * cols * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, part, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int MT, bool TF32, int MODE>
int launch_tc(const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mE, const GemmArgs& args, int grid,
              cudaStream_t st) {
  static unsigned done = 0;
  auto kern = tc_gemm_kernel<MT, TF32, MODE>;
  if (!ensure_smem_attr(kern, Cfg<MT>::kSmem, &done))
    return fail(DFLASH2_ERR_CUDA, "cudaFuncSetAttribute failed: %s", cudaGetErrorString(cudaGetLastError()));
  const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(Cfg<MT>::kThreads), Cfg<MT>::kSmem, st, nullptr, 0, mA, mB,
                                   mE, args);
  if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "tc_gemm launch failed: %s", cudaGetErrorString(e));
  return DFLASH2_OK;
}

template <bool TF32, int MODE>
cudaLaunchConfig_t pair_config(int pairs, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.blockDim = dim3(PairCfg<MODE>::kThreads);
  cfg.dynamicSmemBytes = PairCfg<MODE>::kSmem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <bool TF32, int MODE>
int launch_pair(const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mE, const CUtensorMap& mD,
                const GemmArgs& args, int pairs, cudaStream_t st) {
  static unsigned done = 0;
  auto kern = tc_pair_kernel<TF32, MODE>;
  if (!ensure_smem_attr(kern, PairCfg<MODE>::kSmem, &done))
    return fail(DFLASH2_ERR_CUDA, "cudaFuncSetAttribute failed: %s", cudaGetErrorString(cudaGetLastError()));
  cudaLaunchAttribute cluster[1];
  cluster[0].id = cudaLaunchAttributeClusterDimension;
  cluster[0].val.clusterDim.x = 2;
  cluster[0].val.clusterDim.y = 1;
  cluster[0].val.clusterDim.z = 1;
  const cudaError_t e = launch_pdl(kern, dim3(2 * pairs), dim3(PairCfg<MODE>::kThreads), PairCfg<MODE>::kSmem, st,
                                   cluster, 1, mA, mB, mE, mD, args);
  if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "pair GEMM launch failed: %s", cudaGetErrorString(e));
  return DFLASH2_OK;
}

// Two-CTA clusters of the pair GEMM that can be resident at once on the current device (0 if the
// query fails: the GEMMs then run on single CTAs). Both epilogues fit one CTA per SM.
int pair_capacity() {
  constexpr int kMaxDev = 64;
  static int cached[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] != 0) return cached[dev] > 0 ? cached[dev] : 0;
  int n = 0;
  static unsigned done1 = 0, done0 = 0;
  auto k1 = tc_pair_kernel<false, 1>;
  auto k0 = tc_pair_kernel<false, 0>;
  if (ensure_smem_attr(k1, PairCfg<1>::kSmem, &done1) && ensure_smem_attr(k0, PairCfg<0>::kSmem, &done0)) {
    cudaLaunchAttribute attr[1];
    int n1 = 0, n0 = 0;
    cudaLaunchConfig_t cfg = pair_config<false, 1>(1, nullptr, attr);
    if (cudaOccupancyMaxActiveClusters(&n1, k1, &cfg) != cudaSuccess) n1 = 0;
    cfg = pair_config<false, 0>(1, nullptr, attr);
    if (cudaOccupancyMaxActiveClusters(&n0, k0, &cfg) != cudaSuccess) n0 = 0;
    n = std::min(n1, n0);
  }
  (void)cudaGetLastError();
  cached[dev] = n > 0 ? n : -1;
  return n > 0 ? n : 0;
}

template <int MODE>
int dispatch_tc(int mt, bool tf32, const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mE,
                const GemmArgs& args, int grid, cudaStream_t st) {
  if (mt == 1) return tf32 ? launch_tc<1, true, MODE>(mA, mB, mE, args, grid, st)
                           : launch_tc<1, false, MODE>(mA, mB, mE, args, grid, st);
  return tf32 ? launch_tc<2, true, MODE>(mA, mB, mE, args, grid, st)
              : launch_tc<2, false, MODE>(mA, mB, mE, args, grid, st);
}

int prepare_args(const GemmProblem& p, const GemmPlan& plan, CUtensorMap* mA, CUtensorMap* mB, CUtensorMap* mE,
                 GemmArgs* args) {
  if (!make_map(mA, p.A, p.dtype, p.M, p.K, 128)) return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (A)");
  if (!make_map(mB, p.Bw, p.dtype, p.n_main, p.K, kChunk)) return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (W)");
  if (p.E != nullptr && p.n_extra > 0) {
    if (!make_map(mE, p.E, p.dtype, p.n_extra, p.K, kChunk))
      return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (extra)");
  } else {
    *mE = *mB;
  }
  const int bk = kRowBytes / (p.dtype == DFLASH2_F32 ? 4 : 2);
  GemmArgs& a = *args;
  a = GemmArgs{};
  a.M = p.M;
  a.K = p.K;
  a.n_main = p.n_main;
  a.n_extra = (p.E != nullptr) ? p.n_extra : 0;
  a.main_chunks = (p.n_main + kChunk - 1) / kChunk;
  a.n_chunks = plan.n_chunks;
  a.main_units = (p.n_main + 127) / 128;
  a.n_units = plan.n_chunks;
  a.m_groups = plan.m_groups;
  a.n_splits = plan.n_splits;
  a.k_splits = plan.k_splits;
  a.k_blocks = (p.K + bk - 1) / bk;
  a.err = device_error_word();
  return DFLASH2_OK;
}

}  // namespace

bool make_tmap_sw128(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_sw128_3d(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint64_t planes,
                        uint64_t plane_stride_bytes, uint32_t box_rows, uint32_t box_planes) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, static_cast<cuuint64_t>(plane_stride_bytes)};
  cuuint32_t box[3] = {64, box_rows, box_planes};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Largest M-tile count per CTA the head uses (2: one weight tile feeds 256 rows, single-buffered
// accumulator; 1: 128 rows, double-buffered accumulator).
#ifndef DFL_HEAD_MAX_MT
#define DFL_HEAD_MAX_MT 2
#endif

// 1: heads of more than 128 rows run on CTA pairs (cta_group::2) when the device can host them.
#ifndef DFL_HEAD_PAIR
#define DFL_HEAD_PAIR 1
#endif

GemmPlan head_plan(int M, int K, int n_main, int n_extra, int sms) {
  (void)K;
  GemmPlan p{};
  const int pairs = (DFL_HEAD_PAIR && M > 128) ? std::min(pair_capacity(), sms / 2) : 0;
  if (pairs > 0) {
    p.pair = 1;
    p.mt = 2;
    p.m_groups = (M + 255) / 256;
    p.n_chunks = (n_main + 127) / 128 + (n_extra + 127) / 128;  // 128-column units
    p.n_splits = std::max(1, std::min(p.n_chunks, pairs / p.m_groups));
    p.k_splits = 1;
    return p;
  }
  p.mt = (M > 128 && DFL_HEAD_MAX_MT >= 2) ? 2 : 1;
  p.m_groups = (M + 128 * p.mt - 1) / (128 * p.mt);
  p.n_chunks = (n_main + kChunk - 1) / kChunk + (n_extra + kChunk - 1) / kChunk;
  p.n_splits = std::max(1, std::min(p.n_chunks, sms / p.m_groups));
  p.k_splits = 1;
  return p;
}

size_t head_workspace(int M, int V, int K, int R, int sms) {
  (void)K;
  const GemmPlan p = head_plan(M, 0, V, R, sms);
  const size_t lists = static_cast<size_t>(p.n_splits) * M * kTopL;
  return lists * (sizeof(float) + sizeof(int)) + 256;
}

int gemm_pair_capacity() { return pair_capacity(); }

bool make_tmap_plain(CUtensorMap* m, const void* ptr, int dtype, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
  const CUresult r = enc(m, dtype == DFLASH2_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), d, st, b, e,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int launch_gemm_store(const GemmProblem& p, const GemmPlan& plan, float* part, cudaStream_t st) {
  CUtensorMap mA, mB, mE;
  GemmArgs a;
  int rc = prepare_args(p, plan, &mA, &mB, &mE, &a);
  if (rc != DFLASH2_OK) return rc;
  a.part = part;
  const int grid = plan.m_groups * plan.n_splits * plan.k_splits;
  if (plan.pair) {
    if (p.n_main % 4 != 0) return fail(DFLASH2_ERR_INVALID_ARG, "pair GEMM store needs N %% 4 == 0 (N=%d)", p.n_main);
    // one tile (at most two 128-column units) per pair: its output is staged in the stage ring
    if ((a.n_units + plan.n_splits - 1) / plan.n_splits > 2)
      return fail(DFLASH2_ERR_INVALID_ARG, "pair GEMM store: %d column units over %d splits is more than one tile",
                  a.n_units, plan.n_splits);
    CUtensorMap mD;
    if (!make_part_map(&mD, part, plan.k_splits, p.M, p.n_main))
      return fail(DFLASH2_ERR_CUDA, "tensor map encode failed (partials)");
    return p.dtype == DFLASH2_F32 ? launch_pair<true, 0>(mA, mB, mE, mD, a, grid, st)
                                  : launch_pair<false, 0>(mA, mB, mE, mD, a, grid, st);
  }
  return dispatch_tc<0>(plan.mt, p.dtype == DFLASH2_F32, mA, mB, mE, a, grid, st);
}

int launch_head_topk(const GemmProblem& p, const GemmPlan& plan, const float* bias, int K, int32_t* cand,
                     float* unary, float* z, float* logits, void* workspace, cudaStream_t st, const int32_t* ids_map) {
  CUtensorMap mA, mB, mE;
  GemmArgs a;
  int rc = prepare_args(p, plan, &mA, &mB, &mE, &a);
  if (rc != DFLASH2_OK) return rc;
  const size_t lists = static_cast<size_t>(plan.n_splits) * p.M * kTopL;
  a.list_val = static_cast<float*>(workspace);
  a.list_idx = reinterpret_cast<int*>(a.list_val + lists);
  a.bias = bias;
  a.z = z;
  a.logits = logits;
  const int grid = plan.m_groups * plan.n_splits;
  if (plan.pair)
    rc = p.dtype == DFLASH2_F32 ? launch_pair<true, 1>(mA, mB, mE, mA, a, grid, st)
                                : launch_pair<false, 1>(mA, mB, mE, mA, a, grid, st);
  else
    rc = dispatch_tc<1>(plan.mt, p.dtype == DFLASH2_F32, mA, mB, mE, a, grid, st);
  if (rc != DFLASH2_OK) return rc;
  cudaError_t e;
  if (plan.n_splits <= 32) {
    const int rows_per_block = 8;
    e = launch_pdl(topk_merge_kernel, dim3((p.M + rows_per_block - 1) / rows_per_block), dim3(32 * rows_per_block), 0,
                   st, nullptr, 0, static_cast<const float*>(a.list_val), static_cast<const int*>(a.list_idx),
                   plan.n_splits, p.M, K, ids_map, cand, unary);
  } else {
    const int W = (plan.n_splits + 31) / 32;  // warps per row, each merging at most 32 lists
    if (W > 16) return fail(DFLASH2_ERR_INVALID_ARG, "top-K merge: %d column ranges exceed 512", plan.n_splits);
    e = launch_pdl(topk_merge_wide_kernel, dim3(p.M), dim3(32 * W), 0, st, nullptr, 0,
                   static_cast<const float*>(a.list_val), static_cast<const int*>(a.list_idx), plan.n_splits, p.M, K,
                   ids_map, cand, unary);
  }
  if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "topk_merge launch failed: %s", cudaGetErrorString(e));
  return DFLASH2_OK;
}

int launch_wait_selftest(int limit_us, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(static_cast<uint64_t>(limit_us) * 1000ull, device_error_word());
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "selftest launch failed: %s", cudaGetErrorString(e));
  return DFLASH2_OK;
}

}  // namespace dfl
