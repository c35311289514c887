// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "dflash2.h"

namespace dfl {

// Device error word of the current device (defined in abi.cu): first error wins.
int* device_error_word();

// Wall-time limit of every bounded wait inside the GEMM pipeline.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Records a message for dflash2_last_error_message() and returns `status`.
int fail(int status, const char* fmt, ...);

int sm_count();  // multiprocessors of the current device (cached per device)

// Raises a kernel's dynamic shared-memory limit once per (kernel, device), outside any stream
// work, so that later calls can be captured into a CUDA graph.
template <typename F>
bool ensure_smem_attr(F* kern, int bytes, unsigned* done_mask) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned bit = 1u << (dev & 31);
  if (*done_mask & bit) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  *done_mask |= bit;
  return true;
}

// Programmatic dependent launch: every library kernel is launched with programmatic stream
// serialization, lets its successor's CTAs be scheduled as soon as its own are all running
// (griddepcontrol.launch_dependents at entry) and waits for its predecessor to complete, with
// memory visible (griddepcontrol.wait), before its first global-memory access. The successor's
// launch and prologue then overlap this kernel's last wave instead of following it.
#ifndef DFL_PDL
#define DFL_PDL 1
#endif

// cudaLaunchKernelEx with the programmatic-serialization attribute (and optional extra attributes).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       const cudaLaunchAttribute* extra, int n_extra, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[4];
  int n = 0;
  for (int i = 0; i < n_extra && n < 3; ++i) attr[n++] = extra[i];
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = DFL_PDL ? 1 : 0;
  ++n;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Encodes a tiled, non-swizzled tensor map: dims / box innermost first, strides in bytes for
// dims 1.. (rank - 1 of them). dtype is DFLASH2_BF16 or DFLASH2_F32. False on failure.
bool make_tmap_plain(CUtensorMap* m, const void* ptr, int dtype, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box);

// ---------------------------------------------------------------- conv (conv.cu)
struct ConvShape {
  int B, G, H, gs, groups, dtype;
  int rows() const { return B * G; }
};
struct GemmPlan;
size_t conv_prepare_workspace(const ConvShape& s, int sms);
int launch_rmsnorm(const void* x, const void* w, float eps, void* n, int rows, int H, int dtype, cudaStream_t st);
int launch_conv_side0(const ConvShape& s, const void* n, const float* part, int k_splits, const float* base,
                      void* out, void* coef1, float* d_full, cudaStream_t st);
// kernel_projection and the side-0 pass in one kernel for at most 128 bf16 rows (kp_small.cu);
// with out = null and d0 given, the coefficients only (d0 [2][groups][M] fp32, coef1).
bool kp_small_eligible(const ConvShape& s, int sms);
int launch_kp_small(const ConvShape& s, const void* n, const void* w_kp, const float* base, void* out, void* coef1,
                    float* d_full, cudaStream_t st, float* d0 = nullptr);
// Kernels one prepare call launches (the optional first RMSNorm, kernel_projection, the side-0
// pass) and one finish call (the fused finish + next norm, or the side-1 pass and the norm).
int conv_prepare_kernels(const ConvShape& s, bool with_norm);
int conv_finish_kernels(const ConvShape& s, bool with_next_norm);
// row_off (nullable): the next norm's output rows of block b are the first row_off[b + 1] -
// row_off[b] rows from next_row0 on, written at rows row_off[b] .. of an m_out-row output.
int launch_conv_side1(const ConvShape& s, const void* y, const void* coef1, const float* base, const void* residual,
                      void* out, const void* next_w, float eps, void* next_n, int next_row0, cudaStream_t st,
                      const int32_t* row_off = nullptr, int m_out = 0);

// ---------------------------------------------------------------- tensor-core GEMM (gemm.cu)
// C[m, n] = sum_k A[m, k] * Bw[n, k] over rows m < M of A ([M, K]) and the virtual column range
// [0, n_main) of Bw ([n_main, K]) followed by [pad64(n_main), pad64(n_main) + n_extra) of E ([n_extra, K]).
struct GemmProblem {
  const void* A;
  const void* Bw;
  const void* E;  // extra operand rows (hidden_projection) or nullptr
  int M, K, n_main, n_extra, dtype;
};
struct GemmPlan {
  int mt;        // 128-row M tiles per CTA (1 or 2); per CTA pair when `pair`
  int m_groups;  // ceil(M / (128 * mt))
  int n_splits;  // column ranges (balanced over 64-column chunks, or 128-column units when `pair`)
  int k_splits;  // reduction ranges (STORE mode only)
  int n_chunks;  // 64-column chunks (128-column units when `pair`) over the virtual range
  int pair;      // head on two-CTA clusters (cta_group::2): grid = 2 * m_groups * n_splits CTAs
};
// Split-K plan of the kernel_projection GEMM; shared by the workspace query and the launch.
GemmPlan kp_plan(const ConvShape& s, int sms);
GemmPlan head_plan(int M, int K, int n_main, int n_extra, int sms);
// Two-CTA clusters of the pair GEMM that fit the current device at once (0: pairs unavailable).
int gemm_pair_capacity();
size_t head_workspace(int M, int V, int K, int R, int sms);
// mode 0: write fp32 partial sums part[k_split][M][n_main].
int launch_gemm_store(const GemmProblem& p, const GemmPlan& plan, float* part, cudaStream_t st);
// mode 1: per-row running top-16 over the main columns (+bias), z for the extra columns,
// optional full logits; then a merge into cand/unary.
// ids_map (nullable): token id of each weight row when the head runs over a draft vocabulary.
int launch_head_topk(const GemmProblem& p, const GemmPlan& plan, const float* bias, int K, int32_t* cand,
                     float* unary, float* z, float* logits, void* workspace, cudaStream_t st,
                     const int32_t* ids_map = nullptr);
int launch_wait_selftest(int limit_us, cudaStream_t st);

// bf16 row-major [rows, cols] operand for tcgen05: box of 64 elements (128 bytes) x box_rows rows,
// 128-byte swizzle (defined in gemm.cu).
bool make_tmap_sw128(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);
// The same over `planes` planes of [rows, cols] (plane_stride_bytes apart): box of 64 elements x
// box_rows rows x box_planes planes, landing as box_planes consecutive [box_rows][128 B] tiles.
bool make_tmap_sw128_3d(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint64_t planes,
                        uint64_t plane_stride_bytes, uint32_t box_rows, uint32_t box_planes);

// ---------------------------------------------------------------- sublayer projections (proj.cu)
// out[M, N] = A[M, K] W[N, K]^T (bf16 in and out, fp32 accumulation), with optional fusions:
//   d0 (non-null): A = Conv_0(a) with side-0 deltas d0 [2 taps][groups][M] fp32 and base [2][2][K];
//   coef1 (non-null): out = residual + Conv_1(A W^T) with side-1 deltas coef1 [M][2][groups] bf16 and
//                     base [2][2][N] (residual may be null);
//   wbits = 4: w is packed affine 4-bit [N][K / 8] 32-bit words (value k at bits 4 (k % 8) of word
//              k / 8), scales / qbias [N][K / 64] bf16; wbits = 16: w is bf16 [N][K].
struct ProjSpec {
  const void* a;
  const void* w;
  const void* scales;
  const void* qbias;
  int wbits;
  int M, N, K;
  const float* d0;
  const float* base;
  int G, gs, groups;
  const void* coef1;
  const void* residual;
  void* out;
  float* part;  // split-K partial sums or stream-K slots (proj_workspace bytes), or null when the plan needs none
};
struct ProjPlan {
  int nt;        // columns per tile (64 or 256)
  int k_splits;  // K ranges summed by a reduce pass (1: none)
  int ctas;      // > 0: stream-K over this many CTAs (equal shares of the tiles' k-blocks)
  int pair;      // 1: CTA pairs (cta_group::2) over 256-row tiles; the stream-K units are the pairs
};
ProjPlan proj_plan(int M, int N, int K, int sms, bool epilogue_conv, bool producers);
// At most 128 rows: the weight rows on the MMA's 128-row side, K split over a cluster and reduced in
// shared memory, no workspace (proj_small.cu).
bool proj_small_eligible(int M, int N, int K);
int launch_proj_small(const ProjSpec& p, cudaStream_t st);
size_t proj_workspace(int M, int N, int K, int sms);
int launch_proj(const ProjSpec& p, cudaStream_t st);
// D from kernel_projection's split-K partials: d0 = side 0's deltas (fp32), coef1 = side 1's (dtype).
int launch_conv_coefficients(const float* part, int k_splits, int M, int groups, int dtype, float* d0, void* coef1,
                             cudaStream_t st);

// ---------------------------------------------------------------- selector (selector.cu)
// depths (nullable): per-block draft length of a mixed-depth batch; slots past it get path -1.
// row_off (nullable): a ragged batch, block b's slots are rows row_off[b] .. row_off[b + 1] - 1 of
// the m_rows-row inputs (cand, unary, z, S); path stays [B, steps] with -1 past each block's rows.
int launch_score_edges(const int32_t* cand, const float* unary, const float* z, const int32_t* anchors,
                       const void* pred, const void* succ, int B, int steps, int K, int R, int V, int dtype,
                       float* S, int32_t* path, cudaStream_t st, const int32_t* depths = nullptr,
                       const int32_t* row_off = nullptr, int m_rows = 0);
int launch_select_path(const float* S, const int32_t* cand, int B, int steps, int K, int32_t* path,
                       cudaStream_t st, const int32_t* depths = nullptr);

}  // namespace dfl
