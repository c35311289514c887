// C ABI entry points: host-side validation, workspace carving and dispatch to the kernels.
// Nothing here allocates device memory; every failure returns a status before any launch.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace dfl {

namespace {
__device__ int g_error_word = 0;  // first device-side error of the current device, 0 if none

thread_local char g_msg[512] = "";

constexpr int kMaxDevices = 64;
int g_err_ptr_ready[kMaxDevices];
int* g_err_ptr[kMaxDevices];
int g_sms[kMaxDevices];
std::mutex g_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return status;
}

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_err_ptr_ready[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(p);
    g_err_ptr_ready[dev] = 1;
  }
  return g_err_ptr[dev];
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

}  // namespace dfl

using namespace dfl;

#define REQUIRE(cond, ...)                                  \
  do {                                                      \
    if (!(cond)) return fail(DFLASH2_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

static int check_conv_shape(int B, int G, int H, int gs, int taps, int dtype) {
  if (taps != 2) return fail(DFLASH2_ERR_UNSUPPORTED, "taps=%d: only the two-tap conv is implemented", taps);
  REQUIRE(dtype == DFLASH2_BF16 || dtype == DFLASH2_F32, "dtype=%d is not DFLASH2_BF16 or DFLASH2_F32", dtype);
  REQUIRE(B >= 1, "B=%d must be >= 1", B);
  REQUIRE(G >= 2 && G <= 64, "G=%d must be in [2, 64] (a block needs at least one draft row)", G);
  REQUIRE(H >= 64 && H % 64 == 0, "H=%d must be a positive multiple of 64", H);
  REQUIRE(gs >= 8 && gs % 8 == 0 && H % gs == 0, "group_size=%d must be a multiple of 8 dividing H=%d", gs, H);
  return DFLASH2_OK;
}

extern "C" {

int dflash2_version(void) { return 100; }

const char* dflash2_status_string(int status) {
  switch (status) {
    case DFLASH2_OK: return "DFLASH2_OK";
    case DFLASH2_ERR_INVALID_ARG: return "DFLASH2_ERR_INVALID_ARG";
    case DFLASH2_ERR_UNSUPPORTED: return "DFLASH2_ERR_UNSUPPORTED";
    case DFLASH2_ERR_CUDA: return "DFLASH2_ERR_CUDA";
    case DFLASH2_ERR_WORKSPACE: return "DFLASH2_ERR_WORKSPACE";
    case DFLASH2_ERR_TIMEOUT: return "DFLASH2_ERR_TIMEOUT";
    case DFLASH2_ERR_BAD_INDEX: return "DFLASH2_ERR_BAD_INDEX";
    default: return "DFLASH2_ERR_UNKNOWN";
  }
}

const char* dflash2_last_error_message(void) { return g_msg; }

int dflash2_poll_error(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "stream synchronize failed: %s", cudaGetErrorString(e));
  int* p = device_error_word();
  if (p == nullptr) return fail(DFLASH2_ERR_CUDA, "no device error word");
  int v = 0;
  e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "reading the error word failed: %s", cudaGetErrorString(e));
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail(DFLASH2_ERR_CUDA, "clearing the error word failed: %s", cudaGetErrorString(e));
    fail(v, "a kernel recorded %s", dflash2_status_string(v));
  }
  return v;
}

size_t dflash2_conv_prepare_workspace_bytes(int B, int G, int H, int group_size, int dtype) {
  if (check_conv_shape(B, G, H, group_size, 2, dtype) != DFLASH2_OK) return 0;
  const ConvShape s{B, G, H, group_size, H / group_size, dtype};
  return conv_prepare_workspace(s, sm_count());
}

int dflash2_conv_prepare_launches(int B, int G, int H, int group_size, int dtype, int with_norm) {
  if (check_conv_shape(B, G, H, group_size, 2, dtype) != DFLASH2_OK) return -1;
  return conv_prepare_kernels(ConvShape{B, G, H, group_size, H / group_size, dtype}, with_norm != 0);
}

int dflash2_conv_finish_launches(int B, int G, int H, int group_size, int dtype, int with_next_norm) {
  if (check_conv_shape(B, G, H, group_size, 2, dtype) != DFLASH2_OK) return -1;
  return conv_finish_kernels(ConvShape{B, G, H, group_size, H / group_size, dtype}, with_next_norm != 0);
}

int dflash2_conv_prepare(const void* x, const void* norm_w, float eps, const void* w_kp, const float* base, int B,
                         int G, int H, int group_size, int taps, int dtype, void* out, void* coef1, float* d_full,
                         void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_conv_shape(B, G, H, group_size, taps, dtype);
  if (rc != DFLASH2_OK) return rc;
  REQUIRE(x && w_kp && base && out && coef1 && workspace, "a required pointer is NULL");
  REQUIRE(aligned16(x) && aligned16(w_kp) && aligned16(base) && aligned16(out) && (!norm_w || aligned16(norm_w)),
          "x, norm_w, w_kp, base and out must be 16-byte aligned");
  REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, "workspace must be 256-byte aligned");
  const ConvShape s{B, G, H, group_size, H / group_size, dtype};
  const int sms = sm_count();
  const size_t need = conv_prepare_workspace(s, sms);
  if (workspace_bytes < need)
    return fail(DFLASH2_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", workspace_bytes,
                need);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const GemmPlan plan = kp_plan(s, sms);
  const size_t es = dtype == DFLASH2_F32 ? 4 : 2;
  size_t n_bytes = static_cast<size_t>(s.rows()) * H * es;
  n_bytes = (n_bytes + 255) & ~static_cast<size_t>(255);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const void* n = x;
  if (norm_w != nullptr) {
    rc = launch_rmsnorm(x, norm_w, eps, ws, s.rows(), H, dtype, st);
    if (rc != DFLASH2_OK) return rc;
    n = ws;
  }
  if (kp_small_eligible(s, sms)) return launch_kp_small(s, n, w_kp, base, out, coef1, d_full, st);
  float* part = reinterpret_cast<float*>(ws + n_bytes);
  const GemmProblem gp{n, w_kp, nullptr, s.rows(), H, 4 * s.groups, 0, dtype};
  rc = launch_gemm_store(gp, plan, part, st);
  if (rc != DFLASH2_OK) return rc;
  return launch_conv_side0(s, n, part, plan.k_splits, base, out, coef1, d_full, st);
}

int dflash2_conv_finish(const void* y, const void* coef1, const float* base, int B, int G, int H, int group_size,
                        int taps, int dtype, const void* residual, void* out, const void* next_norm_w, float eps,
                        void* next_n, int next_row0, void* stream) {
  int rc = check_conv_shape(B, G, H, group_size, taps, dtype);
  if (rc != DFLASH2_OK) return rc;
  REQUIRE(y && coef1 && base && out, "a required pointer is NULL");
  REQUIRE((next_norm_w == nullptr) == (next_n == nullptr), "next_norm_w and next_n must be both set or both NULL");
  REQUIRE(aligned16(y) && aligned16(base) && aligned16(out) && (!residual || aligned16(residual)) &&
              (!next_norm_w || aligned16(next_norm_w)) && (!next_n || aligned16(next_n)),
          "y, base, residual, out, next_norm_w and next_n must be 16-byte aligned");
  if (next_n != nullptr) {
    REQUIRE(next_row0 >= 0 && next_row0 < G, "next_row0=%d must be in [0, G)", next_row0);
    REQUIRE(H / 8 <= 1024, "H=%d: the fused norm needs H <= 8192", H);
  }
  const ConvShape s{B, G, H, group_size, H / group_size, dtype};
  return launch_conv_side1(s, y, coef1, base, residual, out, next_norm_w, eps, next_n, next_row0,
                           static_cast<cudaStream_t>(stream));
}

int dflash2_conv_finish_ragged(const void* y, const void* coef1, const float* base, int B, int G, int H,
                               int group_size, int taps, int dtype, const void* residual, void* out,
                               const void* next_norm_w, float eps, void* next_n, int next_row0,
                               const int32_t* row_offsets, int m_rows, void* stream) {
  REQUIRE(row_offsets != nullptr, "row_offsets is NULL (use dflash2_conv_finish for dense rows)");
  REQUIRE(next_norm_w != nullptr && next_n != nullptr, "the ragged finish needs next_norm_w and next_n");
  REQUIRE(m_rows >= 1, "m_rows=%d must be >= 1", m_rows);
  int rc = check_conv_shape(B, G, H, group_size, taps, dtype);
  if (rc != DFLASH2_OK) return rc;
  REQUIRE(y && coef1 && base && out, "a required pointer is NULL");
  REQUIRE(aligned16(y) && aligned16(base) && aligned16(out) && (!residual || aligned16(residual)) &&
              aligned16(next_norm_w) && aligned16(next_n),
          "y, base, residual, out, next_norm_w and next_n must be 16-byte aligned");
  REQUIRE(next_row0 >= 0 && next_row0 < G, "next_row0=%d must be in [0, G)", next_row0);
  REQUIRE(H / 8 <= 1024, "H=%d: the fused norm needs H <= 8192", H);
  const ConvShape s{B, G, H, group_size, H / group_size, dtype};
  return launch_conv_side1(s, y, coef1, base, residual, out, next_norm_w, eps, next_n, next_row0,
                           static_cast<cudaStream_t>(stream), row_offsets, m_rows);
}

int dflash2_conv_coefficients(const void* x, const void* norm_w, float eps, const void* w_kp, int B, int G, int H,
                              int group_size, int taps, int dtype, void* n_out, float* d0, void* coef1,
                              void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_conv_shape(B, G, H, group_size, taps, dtype);
  if (rc != DFLASH2_OK) return rc;
  REQUIRE(x && w_kp && d0 && coef1 && workspace, "a required pointer is NULL");
  REQUIRE(norm_w == nullptr || n_out != nullptr, "n_out is required when norm_w is given");
  REQUIRE(aligned16(x) && aligned16(w_kp) && (!norm_w || aligned16(norm_w)) && (!n_out || aligned16(n_out)),
          "x, norm_w, w_kp and n_out must be 16-byte aligned");
  REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, "workspace must be 256-byte aligned");
  const ConvShape s{B, G, H, group_size, H / group_size, dtype};
  const int sms = sm_count();
  const size_t need = conv_prepare_workspace(s, sms);
  if (workspace_bytes < need)
    return fail(DFLASH2_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", workspace_bytes,
                need);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const GemmPlan plan = kp_plan(s, sms);
  const size_t es = dtype == DFLASH2_F32 ? 4 : 2;
  size_t n_bytes = static_cast<size_t>(s.rows()) * H * es;
  n_bytes = (n_bytes + 255) & ~static_cast<size_t>(255);
  const void* n = x;
  if (norm_w != nullptr) {
    rc = launch_rmsnorm(x, norm_w, eps, n_out, s.rows(), H, dtype, st);
    if (rc != DFLASH2_OK) return rc;
    n = n_out;
  }
  if (kp_small_eligible(s, sms)) return launch_kp_small(s, n, w_kp, nullptr, nullptr, coef1, nullptr, st, d0);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + n_bytes);
  const GemmProblem gp{n, w_kp, nullptr, s.rows(), H, 4 * s.groups, 0, dtype};
  rc = launch_gemm_store(gp, plan, part, st);
  if (rc != DFLASH2_OK) return rc;
  return launch_conv_coefficients(part, plan.k_splits, s.rows(), s.groups, dtype, d0, coef1, st);
}

static int check_proj(const void* a, int M, int K, const void* w, const void* w_scales, const void* w_biases, int wbits,
                      int N, int dtype, void* out) {
  if (dtype != DFLASH2_BF16) return fail(DFLASH2_ERR_UNSUPPORTED, "the projections run in bf16 only (dtype=%d)", dtype);
  REQUIRE(a && w && out, "a required pointer is NULL");
  REQUIRE(M >= 1, "M=%d must be >= 1", M);
  REQUIRE(K >= 64 && K % 64 == 0, "K=%d must be a positive multiple of 64", K);
  REQUIRE(N >= 8 && N % 8 == 0, "N=%d must be a positive multiple of 8", N);
  REQUIRE(wbits == 16 || wbits == 4, "wbits=%d must be 16 (bf16) or 4 (affine 4-bit, groups of 64)", wbits);
  if (wbits == 4)
    REQUIRE(w_scales && w_biases && aligned16(w_scales) && aligned16(w_biases),
            "4-bit weights need 16-byte aligned w_scales and w_biases");
  REQUIRE(aligned16(a) && aligned16(w) && aligned16(out), "a, w and out must be 16-byte aligned");
  return DFLASH2_OK;
}

size_t dflash2_proj_workspace_bytes(int M, int N, int K) {
  if (M < 1 || N < 8 || K < 64) return 0;
  return proj_workspace(M, N, K, sm_count());
}

static int proj_ws(int M, int N, int K, void* workspace, size_t workspace_bytes, float** part) {
  const size_t need = proj_workspace(M, N, K, sm_count());
  *part = nullptr;
  if (need == 0) return DFLASH2_OK;
  if (workspace == nullptr || workspace_bytes < need)
    return fail(DFLASH2_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", workspace_bytes,
                need);
  REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, "workspace must be 256-byte aligned");
  *part = static_cast<float*>(workspace);
  return DFLASH2_OK;
}

int dflash2_proj(const void* a, int M, int K, const void* w, const void* w_scales, const void* w_biases, int wbits,
                 int N, int dtype, void* out, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_proj(a, M, K, w, w_scales, w_biases, wbits, N, dtype, out);
  if (rc != DFLASH2_OK) return rc;
  float* part = nullptr;
  if ((rc = proj_ws(M, N, K, workspace, workspace_bytes, &part)) != DFLASH2_OK) return rc;
  ProjSpec p{};
  p.part = part;
  p.a = a; p.w = w; p.scales = w_scales; p.qbias = w_biases; p.wbits = wbits;
  p.M = M; p.N = N; p.K = K; p.out = out;
  return launch_proj(p, static_cast<cudaStream_t>(stream));
}

int dflash2_proj_conv_in(const void* n, const float* d0, const float* base, int G, int group_size, int M, int K,
                         const void* w, const void* w_scales, const void* w_biases, int wbits, int N, int dtype,
                         void* out, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_proj(n, M, K, w, w_scales, w_biases, wbits, N, dtype, out);
  if (rc != DFLASH2_OK) return rc;
  float* part = nullptr;
  REQUIRE(d0 && base, "d0 and base are required");
  REQUIRE(G >= 2 && G <= 64 && 128 % G == 0, "G=%d must divide 128 (blocks must not straddle a 128-row tile)", G);
  REQUIRE(M % G == 0, "M=%d must be a whole number of %d-row blocks", M, G);
  REQUIRE(group_size == 16, "group_size=%d: the fused side 0 is built for groups of 16 channels", group_size);
  REQUIRE(M % 4 == 0, "M=%d must be a multiple of 4 (rows of the side-0 deltas are loaded in 16-byte units)", M);
  REQUIRE(aligned16(base) && aligned16(d0), "base and d0 must be 16-byte aligned");
  if ((rc = proj_ws(M, N, K, workspace, workspace_bytes, &part)) != DFLASH2_OK) return rc;
  ProjSpec p{};
  p.part = part;
  p.a = n; p.w = w; p.scales = w_scales; p.qbias = w_biases; p.wbits = wbits;
  p.M = M; p.N = N; p.K = K; p.out = out;
  p.d0 = d0; p.base = base; p.G = G; p.gs = group_size; p.groups = K / group_size;
  return launch_proj(p, static_cast<cudaStream_t>(stream));
}

int dflash2_proj_conv_out(const void* a, int M, int K, const void* w, const void* w_scales, const void* w_biases,
                          int wbits, int N, const void* coef1, const float* base, int G, int group_size,
                          const void* residual, int dtype, void* out, void* workspace, size_t workspace_bytes,
                          void* stream) {
  int rc = check_proj(a, M, K, w, w_scales, w_biases, wbits, N, dtype, out);
  if (rc != DFLASH2_OK) return rc;
  float* part = nullptr;
  REQUIRE(coef1 && base, "coef1 and base are required");
  REQUIRE(G >= 2 && G <= 32 && 32 % G == 0, "G=%d must divide 32 (a block's rows must share a warp)", G);
  REQUIRE(M % G == 0, "M=%d must be a whole number of %d-row blocks", M, G);
  REQUIRE(group_size == 8 || group_size == 16 || group_size == 32, "group_size=%d must be 8, 16 or 32", group_size);
  REQUIRE(N % group_size == 0 && N % 32 == 0, "N=%d must be a multiple of 32 and of group_size", N);
  REQUIRE(aligned16(base) && (!residual || aligned16(residual)), "base and residual must be 16-byte aligned");
  if ((rc = proj_ws(M, N, K, workspace, workspace_bytes, &part)) != DFLASH2_OK) return rc;
  ProjSpec p{};
  p.part = part;
  p.a = a; p.w = w; p.scales = w_scales; p.qbias = w_biases; p.wbits = wbits;
  p.M = M; p.N = N; p.K = K; p.out = out;
  p.coef1 = coef1; p.base = base; p.residual = residual; p.G = G; p.gs = group_size; p.groups = N / group_size;
  return launch_proj(p, static_cast<cudaStream_t>(stream));
}

size_t dflash2_head_topk_workspace_bytes(int M, int H, int V, int K, int R) {
  if (M < 1 || H < 64 || V < 1 || K < 1 || R < 0) return 0;
  return head_workspace(M, V, K, R, sm_count());
}

int dflash2_head_topk(const void* h, int M, int H, const void* w_head, int V, const float* bias, const void* w_proj,
                      int R, int K, int dtype, int32_t* cand, float* unary, float* z, float* logits, void* workspace,
                      size_t workspace_bytes, void* stream) {
  REQUIRE(dtype == DFLASH2_BF16 || dtype == DFLASH2_F32, "dtype=%d is not DFLASH2_BF16 or DFLASH2_F32", dtype);
  REQUIRE(M >= 1, "M=%d must be >= 1", M);
  REQUIRE(H >= 64 && H % 64 == 0, "H=%d must be a positive multiple of 64", H);
  REQUIRE(K >= 1 && K <= 16 && K <= V, "K=%d must be in [1, min(16, V)]", K);
  REQUIRE(h && w_head && cand && unary && workspace, "a required pointer is NULL");
  REQUIRE((w_proj == nullptr) == (z == nullptr), "w_proj and z must be both set or both NULL");
  if (w_proj != nullptr) REQUIRE(R >= 16 && R <= 256 && R % 16 == 0, "R=%d must be a multiple of 16 in [16, 256]", R);
  REQUIRE(aligned16(h) && aligned16(w_head) && (!w_proj || aligned16(w_proj)) && (!bias || aligned16(bias)),
          "h, w_head, w_proj and bias must be 16-byte aligned");
  REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, "workspace must be 256-byte aligned");
  const int r_eff = w_proj != nullptr ? R : 0;
  const int sms = sm_count();
  const size_t need = head_workspace(M, V, K, r_eff, sms);
  if (workspace_bytes < need)
    return fail(DFLASH2_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", workspace_bytes,
                need);
  const GemmPlan plan = head_plan(M, H, V, r_eff, sms);
  const GemmProblem gp{h, w_head, w_proj, M, H, V, r_eff, dtype};
  return launch_head_topk(gp, plan, bias, K, cand, unary, z, logits, workspace, static_cast<cudaStream_t>(stream));
}

int dflash2_head_topk_vocab(const void* h, int M, int H, const void* w_listed, int V_listed, const int32_t* vocab_ids,
                            const float* bias_listed, const void* w_proj, int R, int K, int dtype, int32_t* cand,
                            float* unary, float* z, float* logits, void* workspace, size_t workspace_bytes,
                            void* stream) {
  REQUIRE(vocab_ids != nullptr, "vocab_ids is NULL (use dflash2_head_topk for the full vocabulary)");
  REQUIRE(dtype == DFLASH2_BF16 || dtype == DFLASH2_F32, "dtype=%d is not DFLASH2_BF16 or DFLASH2_F32", dtype);
  REQUIRE(M >= 1, "M=%d must be >= 1", M);
  REQUIRE(H >= 64 && H % 64 == 0, "H=%d must be a positive multiple of 64", H);
  REQUIRE(K >= 1 && K <= 16 && K <= V_listed, "K=%d must be in [1, min(16, V_listed)]", K);
  REQUIRE(h && w_listed && cand && unary && workspace, "a required pointer is NULL");
  REQUIRE((w_proj == nullptr) == (z == nullptr), "w_proj and z must be both set or both NULL");
  if (w_proj != nullptr) REQUIRE(R >= 16 && R <= 256 && R % 16 == 0, "R=%d must be a multiple of 16 in [16, 256]", R);
  REQUIRE(aligned16(h) && aligned16(w_listed) && (!w_proj || aligned16(w_proj)) && (!bias_listed || aligned16(bias_listed)),
          "h, w_listed, w_proj and bias_listed must be 16-byte aligned");
  REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, "workspace must be 256-byte aligned");
  const int r_eff = w_proj != nullptr ? R : 0;
  const int sms = sm_count();
  const size_t need = head_workspace(M, V_listed, K, r_eff, sms);
  if (workspace_bytes < need)
    return fail(DFLASH2_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", workspace_bytes,
                need);
  const GemmPlan plan = head_plan(M, H, V_listed, r_eff, sms);
  const GemmProblem gp{h, w_listed, w_proj, M, H, V_listed, r_eff, dtype};
  return launch_head_topk(gp, plan, bias_listed, K, cand, unary, z, logits, workspace,
                          static_cast<cudaStream_t>(stream), vocab_ids);
}

int dflash2_score_edges(const int32_t* cand, const float* unary, const float* z, const int32_t* anchors,
                        const void* pred_book, const void* succ_book, int B, int steps, int K, int R, int V, int dtype,
                        float* S, int32_t* path, void* stream) {
  REQUIRE(dtype == DFLASH2_BF16 || dtype == DFLASH2_F32, "dtype=%d is not DFLASH2_BF16 or DFLASH2_F32", dtype);
  REQUIRE(B >= 1 && steps >= 1 && steps <= 63, "B=%d, steps=%d: need B >= 1 and 1 <= steps <= 63", B, steps);
  REQUIRE(K >= 1 && K <= 32, "K=%d must be in [1, 32]", K);
  REQUIRE(R >= 8 && R <= 128 && R % 8 == 0, "R=%d must be a multiple of 8 in [8, 128]", R);
  REQUIRE(V >= 1, "V=%d must be >= 1", V);
  REQUIRE(cand && unary && z && anchors && pred_book && succ_book, "a required pointer is NULL");
  REQUIRE(S != nullptr || path != nullptr, "at least one of S and path must be non-NULL");
  REQUIRE(aligned16(z) && aligned16(pred_book) && aligned16(succ_book), "z and the codebooks must be 16-byte aligned");
  return launch_score_edges(cand, unary, z, anchors, pred_book, succ_book, B, steps, K, R, V, dtype, S, path,
                            static_cast<cudaStream_t>(stream));
}

int dflash2_score_edges_depths(const int32_t* cand, const float* unary, const float* z, const int32_t* anchors,
                               const void* pred_book, const void* succ_book, const int32_t* depths, int B, int steps,
                               int K, int R, int V, int dtype, float* S, int32_t* path, void* stream) {
  REQUIRE(depths != nullptr, "depths is NULL (use dflash2_score_edges for full-depth blocks)");
  REQUIRE(dtype == DFLASH2_BF16 || dtype == DFLASH2_F32, "dtype=%d is not DFLASH2_BF16 or DFLASH2_F32", dtype);
  REQUIRE(B >= 1 && steps >= 1 && steps <= 63, "B=%d, steps=%d: need B >= 1 and 1 <= steps <= 63", B, steps);
  REQUIRE(K >= 1 && K <= 32, "K=%d must be in [1, 32]", K);
  REQUIRE(R >= 8 && R <= 128 && R % 8 == 0, "R=%d must be a multiple of 8 in [8, 128]", R);
  REQUIRE(V >= 1, "V=%d must be >= 1", V);
  REQUIRE(cand && unary && z && anchors && pred_book && succ_book && path, "a required pointer is NULL");
  REQUIRE(aligned16(z) && aligned16(pred_book) && aligned16(succ_book), "z and the codebooks must be 16-byte aligned");
  return launch_score_edges(cand, unary, z, anchors, pred_book, succ_book, B, steps, K, R, V, dtype, S, path,
                            static_cast<cudaStream_t>(stream), depths);
}

int dflash2_score_edges_ragged(const int32_t* cand, const float* unary, const float* z, const int32_t* anchors,
                               const void* pred_book, const void* succ_book, const int32_t* row_offsets, int B,
                               int steps, int K, int R, int V, int m_rows, int dtype, float* S, int32_t* path,
                               void* stream) {
  REQUIRE(row_offsets != nullptr, "row_offsets is NULL (use dflash2_score_edges for dense blocks)");
  REQUIRE(dtype == DFLASH2_BF16 || dtype == DFLASH2_F32, "dtype=%d is not DFLASH2_BF16 or DFLASH2_F32", dtype);
  REQUIRE(B >= 1 && steps >= 1 && steps <= 63, "B=%d, steps=%d: need B >= 1 and 1 <= steps <= 63", B, steps);
  REQUIRE(m_rows >= 1, "m_rows=%d must be >= 1", m_rows);
  REQUIRE(K == 16 && (R == 16 || R == 32 || (R == 64 && dtype == DFLASH2_BF16)),
          "ragged rows need K = 16 and R in {16, 32, 64} (bf16) or {16, 32} (f32); got K=%d, R=%d", K, R);
  REQUIRE(V >= 1, "V=%d must be >= 1", V);
  REQUIRE(cand && unary && z && anchors && pred_book && succ_book && path, "a required pointer is NULL");
  REQUIRE(aligned16(z) && aligned16(pred_book) && aligned16(succ_book), "z and the codebooks must be 16-byte aligned");
  return launch_score_edges(cand, unary, z, anchors, pred_book, succ_book, B, steps, K, R, V, dtype, S, path,
                            static_cast<cudaStream_t>(stream), nullptr, row_offsets, m_rows);
}

int dflash2_select_path_depths(const float* S, const int32_t* cand, const int32_t* depths, int B, int steps, int K,
                               int32_t* path, void* stream) {
  REQUIRE(depths != nullptr, "depths is NULL (use dflash2_select_path for full-depth blocks)");
  REQUIRE(B >= 1 && steps >= 1, "B=%d, steps=%d must be >= 1", B, steps);
  REQUIRE(K >= 1 && K <= 32, "K=%d must be in [1, 32]", K);
  REQUIRE(S && cand && path, "a required pointer is NULL");
  return launch_select_path(S, cand, B, steps, K, path, static_cast<cudaStream_t>(stream), depths);
}

int dflash2_select_path(const float* S, const int32_t* cand, int B, int steps, int K, int32_t* path, void* stream) {
  REQUIRE(B >= 1 && steps >= 1, "B=%d, steps=%d must be >= 1", B, steps);
  REQUIRE(K >= 1 && K <= 32, "K=%d must be in [1, 32]", K);
  REQUIRE(S && cand && path, "a required pointer is NULL");
  return launch_select_path(S, cand, B, steps, K, path, static_cast<cudaStream_t>(stream));
}

int dflash2_selftest_bounded_wait(int limit_us, void* stream) {
  REQUIRE(limit_us >= 1 && limit_us <= 1000000, "limit_us=%d must be in [1, 1000000]", limit_us);
  return launch_wait_selftest(limit_us, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
