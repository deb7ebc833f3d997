// extern "C" device entry points of libqfmt: argument validation, kernel
// selection by batch size, and launch on the caller's stream.
//
// Kernel selection (the pages pick kernels by batch size as well: the
// metaltile qmm selector routes 4 <= m <= 12 to its two-row variant, and the
// rlx-cpu matmuls switch on m > 1): M <= 16 runs the decode GEMV, M > 16 the
// tensor-core GEMM, float32 activations the CUDA-core path.
#include <atomic>
#include <cmath>
#include <cstdint>

#include <cuda_runtime.h>

#include "kernels.h"
#include "qfmt_internal.h"

using namespace qfmt;

namespace {

std::atomic<int> g_sms[64];

// SM count of the current device (cached per device).
int device_sms(int* err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { *err = fail(QFMT_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e)); return 0; }
  if (dev < 0 || dev >= 64) { *err = fail(QFMT_ECUDA, "device index %d out of range", dev); return 0; }
  int v = g_sms[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) { *err = fail(QFMT_ECUDA, "device query: %s", cudaGetErrorString(e)); return 0; }
  g_sms[dev].store(v, std::memory_order_relaxed);
  return v;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return QFMT_OK;
  return fail(QFMT_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Code rows the kernels stream for N outputs: mxfp4x2 keeps two residual
// planes per output row, which the kernels treat as rows 2n and 2n + 1.
int64_t weight_rows(int fmt, int64_t N) { return fmt == QFMT_MXFP4X2 ? 2 * N : N; }

int check_common(int fmt, const void* codes, const void* scales, float glob, int group) {
  int st = check_group(fmt, group);
  if (st) return st;
  if ((st = check_ptr(codes, 16, "codes"))) return st;
  if ((st = check_ptr(scales, 4, "scales"))) return st;
  if (fmt == QFMT_NVFP4 && !(std::isfinite(glob) && glob > 0.0f))
    return fail(QFMT_EINVAL, "nvfp4 global_scale must be finite and > 0");
  return QFMT_OK;
}

}  // namespace

extern "C" {

int qfmt_dequant(int fmt, const void* codes, const void* scales, float global_scale, void* out,
                 int out_dtype, int64_t N, int64_t K, int group, void* stream) {
  clear_error();
  int st = check_group(fmt, group);
  if (st) return st;
  if ((st = check_shape(fmt, 0, N, K))) return st;
  if (out_dtype != QFMT_F32 && out_dtype != QFMT_BF16) return fail(QFMT_EINVAL, "bad out_dtype %d", out_dtype);
  if (N == 0 || K == 0) return QFMT_OK;
  if ((st = check_common(fmt, codes, scales, global_scale, group))) return st;
  if ((st = check_ptr(out, 16, "out"))) return st;
  int err = QFMT_OK;
  const int sms = device_sms(&err);
  if (err) return err;
  if (qfmt_dev::is_sub_byte(fmt))
    return cuda_status(qfmt_dev::launch_dequant_sub(fmt, codes, scales, out, out_dtype == QFMT_BF16, N, K,
                                                    static_cast<cudaStream_t>(stream), sms),
                       "dequant launch");
  return cuda_status(qfmt_dev::launch_dequant(fmt, codes, scales, global_scale, out, out_dtype == QFMT_BF16,
                                              N, K, static_cast<cudaStream_t>(stream), sms),
                     "dequant launch");
}

int qmm_ex(int fmt, const void* codes, const void* scales, float global_scale, const void* x, int x_dtype,
           void* out, int out_dtype, int64_t M, int64_t N, int64_t K, int group, void* workspace,
           size_t workspace_bytes, void* stream) {
  clear_error();
  int st = check_group(fmt, group);
  if (st) return st;
  if ((st = check_shape(fmt, M, N, K))) return st;
  if (x_dtype != QFMT_F32 && x_dtype != QFMT_BF16) return fail(QFMT_EINVAL, "bad x_dtype %d", x_dtype);
  if (out_dtype != QFMT_F32 && out_dtype != QFMT_BF16) return fail(QFMT_EINVAL, "bad out_dtype %d", out_dtype);
  if (M == 0 || N == 0) return QFMT_OK;
  if ((st = check_ptr(out, 16, "out"))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool out_f32 = out_dtype == QFMT_F32;
  if (K == 0)
    return cuda_status(cudaMemsetAsync(out, 0, size_t(M) * size_t(N) * (out_f32 ? 4 : 2), s), "memset");
  if ((st = check_common(fmt, codes, scales, global_scale, group))) return st;
  if ((st = check_ptr(x, 16, "x"))) return st;
  // the GEMM's 128-row tiles run along the grid's y dimension (at most 65535)
  if (x_dtype == QFMT_BF16 && M > 16 && (M + 127) / 128 > 65535)
    return fail(QFMT_ESHAPE, "M=%lld: more than 65535 row tiles of 128", (long long)M);
  int err = QFMT_OK;
  const int sms = device_sms(&err);
  if (err) return err;
  if (qfmt_dev::is_sub_byte(fmt))   // the 2/3/5/6-bit codes: one CUDA-core kernel for every M and X dtype
    return cuda_status(qfmt_dev::launch_qmm_sub(fmt, codes, scales, x, x_dtype == QFMT_F32, out, out_f32, M, N, K, s),
                       "qmm (sub-byte codes) launch");
  if (x_dtype == QFMT_F32)
    return cuda_status(qfmt_dev::launch_qmm_f32x(fmt, codes, scales, global_scale, static_cast<const float*>(x),
                                                 out, out_f32, M, N, K, s, sms),
                       "qmm (f32 activations) launch");
  if (M <= 16) {
    // the MX formats the block-scaled MMA reads as stored: the tensor-core
    // decode GEMV (no ALU decode); the rest: the mma.sync decode GEMVs
    if (qfmt_dev::qgemv_mx_supported(fmt, M, N, K, codes, sms))
      return cuda_status(qfmt_dev::launch_qgemv_mx(fmt, codes, scales, x, out, out_f32, M, N, K, s, sms),
                         "block-scaled qgemv launch");
    return cuda_status(qfmt_dev::launch_qgemv(fmt, codes, scales, global_scale, x, out, out_f32, M,
                                              weight_rows(fmt, N), K, s, sms),
                       "qgemv launch");
  }
  // With a workspace, the MX formats the block-scaled MMA reads as stored take
  // it (the E2M1 codes' tensor map needs a 32-byte aligned base).
  if (workspace && qfmt_dev::qgemm_mx_supported(fmt, M, K) &&
      !(fmt == QFMT_MXFP4 && (reinterpret_cast<uintptr_t>(codes) & 31u))) {
    const size_t need = qfmt_dev::qgemm_mx_workspace_bytes(M, K);
    if (workspace_bytes < need)
      return fail(QFMT_ENOSPACE, "workspace of %zu bytes, the block-scaled GEMM needs %zu", workspace_bytes, need);
    if ((st = check_ptr(workspace, 128, "workspace"))) return st;
    return cuda_status(qfmt_dev::launch_qgemm_mx(fmt, codes, scales, x, out, out_f32, M, N, K, workspace, s, sms),
                       "block-scaled qgemm launch");
  }
  // the GEMM decodes both mxfp4x2 planes of an output row together: N output rows
  return cuda_status(qfmt_dev::launch_qgemm_tc(fmt, codes, scales, global_scale, x, out, out_f32, M, N, K, s, sms),
                     "qgemm launch");
}

int qmm(int fmt, const void* codes, const void* scales, float global_scale, const void* x, void* out,
        int64_t M, int64_t N, int64_t K, int group, void* stream) {
  return qmm_ex(fmt, codes, scales, global_scale, x, QFMT_BF16, out, QFMT_BF16, M, N, K, group, nullptr, 0,
                stream);
}

// The fused decode forms run on the mma.sync decode GEMV, which takes the
// byte- and nibble-aligned formats; the 2/3/5/6-bit ones take qmm.
static int refuse_sub_byte(int fmt, const char* name) {
  if (!qfmt_dev::is_sub_byte(fmt)) return QFMT_OK;
  return fail(QFMT_EUNSUPPORTED, "%s: the 2/3/5/6-bit formats run through qmm / qmm_ex only", name);
}

int qmm_gather(int fmt, const void* codes, const void* scales, float global_scale, const void* x,
               const int32_t* expert_idx, void* out, int64_t M, int64_t N, int64_t K, int64_t E, int group,
               void* stream) {
  clear_error();
  int st = check_group(fmt, group);
  if (st) return st;
  if ((st = refuse_sub_byte(fmt, "qmm_gather"))) return st;
  if ((st = check_shape(fmt, M, N, K))) return st;
  if (E < 1) return fail(QFMT_EINVAL, "expert count E=%lld must be >= 1", (long long)E);
  if (E * weight_rows(fmt, N) >= (int64_t(1) << 31)) return fail(QFMT_ESHAPE, "E*N code rows of 2^31 or more");
  if (M > 65535) return fail(QFMT_ESHAPE, "M=%lld above 65535 rows", (long long)M);
  if (M == 0 || N == 0) return QFMT_OK;
  if ((st = check_ptr(out, 16, "out"))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return cuda_status(cudaMemsetAsync(out, 0, size_t(M) * size_t(N) * 2, s), "memset");
  if ((st = check_common(fmt, codes, scales, global_scale, group))) return st;
  if ((st = check_ptr(x, 16, "x"))) return st;
  if ((st = check_ptr(expert_idx, 4, "expert_idx"))) return st;
  if (!qfmt_dev::qgemv_m2_fits(fmt, 1, K))
    return fail(QFMT_EUNSUPPORTED, "K=%lld too long for the expert-routed GEMV", (long long)K);
  return cuda_status(qfmt_dev::launch_qgemv_gather(fmt, codes, scales, global_scale, x, expert_idx, out, false, M,
                                                    weight_rows(fmt, N), K, E, s),
                     "qmm_gather launch");
}

int qmm_batched(int fmt, int count, const void* const* codes, const void* const* scales,
                const float* global_scales, const int64_t* N, const void* x, void* const* out, int64_t M,
                int64_t K, int group, void* stream) {
  clear_error();
  int st = check_group(fmt, group);
  if (st) return st;
  if ((st = refuse_sub_byte(fmt, "qmm_batched"))) return st;
  if (count < 1 || count > 4) return fail(QFMT_EINVAL, "count=%d must be 1..4", count);
  if (!codes || !scales || !global_scales || !N || !out) return fail(QFMT_EINVAL, "NULL pointer array");
  for (int i = 0; i < count; ++i) {
    if ((st = check_shape(fmt, M, N[i], K))) return st;
    if ((st = check_ptr(out[i], 16, "out"))) return st;
  }
  if (M == 0) return QFMT_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    for (int i = 0; i < count; ++i)
      if ((st = cuda_status(cudaMemsetAsync(out[i], 0, size_t(M) * size_t(N[i]) * 2, s), "memset"))) return st;
    return QFMT_OK;
  }
  for (int i = 0; i < count; ++i)
    if ((st = check_common(fmt, codes[i], scales[i], global_scales[i], group))) return st;
  if ((st = check_ptr(x, 16, "x"))) return st;
  bool any = false;
  for (int i = 0; i < count; ++i) any |= N[i] > 0;
  if (!any) return QFMT_OK;
  if (M <= 2 && qfmt_dev::qgemv_m2_fits(fmt, M, K)) {
    // one launch over every matrix's row tiles (a matrix with N = 0 has none)
    const void* c[4];
    const void* sc[4];
    float g[4];
    int64_t n[4];
    void* o[4];
    int live = 0;
    for (int i = 0; i < count; ++i) {
      if (N[i] == 0) continue;
      c[live] = codes[i];
      sc[live] = scales[i];
      g[live] = global_scales[i];
      n[live] = weight_rows(fmt, N[i]);
      o[live] = out[i];
      ++live;
    }
    return cuda_status(qfmt_dev::launch_qgemv_multi(fmt, live, c, sc, g, n, x, nullptr, 0.0f, o, false, M, K, s),
                       "qmm_batched launch");
  }
  for (int i = 0; i < count; ++i)   // larger batches: one qmm per matrix
    if ((st = qmm(fmt, codes[i], scales[i], global_scales[i], x, out[i], M, N[i], K, group, stream))) return st;
  return QFMT_OK;
}

// The fused RMSNorm (gate == nullptr) and gated-RMSNorm decode GEMVs.
static int rmsnorm_form(int fmt, const void* codes, const void* scales, float global_scale, const void* x,
                 const void* gate, const void* norm_weight, float eps, void* out, int64_t M, int64_t N, int64_t K,
                 int group, void* stream, const char* name) {
  clear_error();
  int st = check_group(fmt, group);
  if (st) return st;
  if ((st = refuse_sub_byte(fmt, name))) return st;
  if ((st = check_shape(fmt, M, N, K))) return st;
  if (M > 2) return fail(QFMT_EUNSUPPORTED, "%s is the decode form: M=%lld above 2", name, (long long)M);
  if (!(std::isfinite(eps) && eps >= 0.0f)) return fail(QFMT_EINVAL, "eps must be finite and >= 0");
  if (M == 0 || N == 0) return QFMT_OK;
  if (K == 0) return fail(QFMT_ESHAPE, "the RMS of an empty row is undefined (K = 0)");
  if ((st = check_ptr(out, 16, "out"))) return st;
  if ((st = check_common(fmt, codes, scales, global_scale, group))) return st;
  if ((st = check_ptr(x, 16, "x"))) return st;
  if ((st = check_ptr(norm_weight, 16, "norm_weight"))) return st;
  if (gate && (st = check_ptr(gate, 16, "gate"))) return st;
  if (!qfmt_dev::qgemv_m2_fits(fmt, M, K))
    return fail(QFMT_EUNSUPPORTED, "K=%lld too long for the fused decode GEMV", (long long)K);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float g = global_scale;
  const int64_t nw = weight_rows(fmt, N);
  return cuda_status(qfmt_dev::launch_qgemv_multi(fmt, 1, &codes, &scales, &g, &nw, x, norm_weight, eps, &out, false,
                                                   M, K, s, gate),
                     name);
}

int qmm_rmsnorm(int fmt, const void* codes, const void* scales, float global_scale, const void* x,
                const void* norm_weight, float eps, void* out, int64_t M, int64_t N, int64_t K, int group,
                void* stream) {
  return rmsnorm_form(fmt, codes, scales, global_scale, x, nullptr, norm_weight, eps, out, M, N, K, group, stream,
                      "qmm_rmsnorm");
}

int qmm_gated_rmsnorm(int fmt, const void* codes, const void* scales, float global_scale, const void* x,
                      const void* gate, const void* norm_weight, float eps, void* out, int64_t M, int64_t N,
                      int64_t K, int group, void* stream) {
  if (!gate) {
    clear_error();
    return fail(QFMT_EINVAL, "gate is NULL");
  }
  return rmsnorm_form(fmt, codes, scales, global_scale, x, gate, norm_weight, eps, out, M, N, K, group, stream,
                      "qmm_gated_rmsnorm");
}

int qfmt_device_status(void* stream) {
  clear_error();
  int st = cuda_status(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream sync");
  if (st) return st;
  unsigned int word = 0, gw = 0;
  if ((st = cuda_status(qfmt_dev::read_and_clear_device_status(&word), "device status"))) return st;
  if ((st = cuda_status(qfmt_dev::read_and_clear_gemv_status(&gw), "device status"))) return st;
  unsigned int gx = 0, mw = 0, rb = 0;
  if ((st = cuda_status(qfmt_dev::read_and_clear_gather_status(&gx), "device status"))) return st;
  if ((st = cuda_status(qfmt_dev::read_and_clear_rb_status(&rb), "device status"))) return st;
  if ((st = cuda_status(qfmt_dev::read_and_clear_mx_status(&mw), "device status"))) return st;
  if (word) return fail(QFMT_ETIMEOUT, "a tensor-core GEMM pipeline wait expired (status 0x%x)", word);
  if (mw & 1u) return fail(QFMT_ETIMEOUT, "a block-scaled GEMM pipeline wait expired (status 0x%x)", mw);
  if (gw) return fail(QFMT_ETIMEOUT, "a GEMV weight-copy wait expired (status 0x%x)", gw);
  if (gx & 2u) return fail(QFMT_ETIMEOUT, "a decode GEMV weight-copy wait expired (status 0x%x)", gx);
  if (rb) return fail(QFMT_ETIMEOUT, "a batch decode GEMV activation-copy wait expired (status 0x%x)", rb);
  if ((gx & 1u) || (mw & 2u))
    return fail(QFMT_EINDEX, "qmm_gather / qmm_grouped: an expert index outside [0, E) (its output row was zeroed)");
  return QFMT_OK;
}

int qfmt_debug_set(int key, int64_t value) {
  clear_error();
  if (key == 1) {
    qfmt_dev::set_wait_limit_ns(value > 0 ? uint64_t(value) : 2000000000ull);
    qfmt_dev::set_mx_wait_limit_ns(value > 0 ? uint64_t(value) : 2000000000ull);
    return QFMT_OK;
  }
  if (key == 2) {
    qfmt_dev::set_drop_arrivals(value ? 1 : 0);
    qfmt_dev::set_mx_drop_arrivals(value ? 1 : 0);
    return QFMT_OK;
  }
  if (key == 3 || key == 4) {   // the block-scaled GEMM's tile width (224, 256) / K split (1-4); 0 = planner
    static std::atomic<int> bn{0}, sk{0};
    (key == 3 ? bn : sk).store(int(value));
    qfmt_dev::set_mx_plan(bn.load(), sk.load());
    return QFMT_OK;
  }
  if (key == 5 || key == 6) {   // decode GEMV of the MX formats: 5 = use the mma.sync GEMVs; 6 = K split
    static std::atomic<int> off{0}, sk{0};
    (key == 5 ? off : sk).store(int(value));
    qfmt_dev::set_mx_gemv(off.load(), sk.load());
    return QFMT_OK;
  }
  if (key == 7) {   // the batch decode GEMV (3 <= M <= 16): 1 = the K-split kernel instead of the one-decode one
    qfmt_dev::set_gemv_rb(value ? 1 : 0);
    return QFMT_OK;
  }
  if (key == 9) {   // the quantized-activation GEMM's tall tiles: 0 = its plan, 1 = never, 2 = wherever allowed
    if (value < 0 || value > 2) return fail(QFMT_EINVAL, "debug key 9 takes 0, 1 or 2");
    qfmt_dev::set_mx_tall(int(value));
    return QFMT_OK;
  }
  if (key == 8) {   // the bf16-decode GEMM's tile order: 0 = the host's choice, 1 = N tiles first, 2 = M tiles first
    if (value < 0 || value > 2) return fail(QFMT_EINVAL, "debug key 8 takes 0, 1 or 2");
    qfmt_dev::set_tc_order(int(value));
    return QFMT_OK;
  }
  return fail(QFMT_EINVAL, "unknown debug key %d", key);
}

size_t qmm_grouped_workspace_bytes(int fmt, int64_t M, int64_t K, int64_t E) {
  clear_error();
  if (fmt != QFMT_MXFP4 && fmt != QFMT_MXFP8_E4M3 && fmt != QFMT_MXFP8_E5M2) return 0;
  if (M <= 0 || K <= 0 || K % 128 || E < 1 || E > qfmt_dev::qgemm_grouped_max_experts()) return 0;
  return qfmt_dev::qgemm_grouped_workspace_bytes(M, K, E);
}

int qmm_grouped(int fmt, const void* codes, const void* scales, const void* x, const int32_t* expert_idx, void* out,
                int out_dtype, int64_t M, int64_t N, int64_t K, int64_t E, void* workspace, size_t workspace_bytes,
                void* stream) {
  clear_error();
  int st = check_group(fmt, 0);
  if (st) return st;
  if (fmt != QFMT_MXFP4 && fmt != QFMT_MXFP8_E4M3 && fmt != QFMT_MXFP8_E5M2)
    return fail(QFMT_EUNSUPPORTED, "qmm_grouped takes mxfp4, mxfp8 E4M3 or E5M2 weights (format %d)", fmt);
  if ((st = check_shape(fmt, M, N, K))) return st;
  if (E < 1 || E > qfmt_dev::qgemm_grouped_max_experts())
    return fail(QFMT_EINVAL, "expert count E=%lld must be in 1..%d", (long long)E, qfmt_dev::qgemm_grouped_max_experts());
  if (E * N >= (int64_t(1) << 31)) return fail(QFMT_ESHAPE, "E*N weight rows of 2^31 or more");
  if (out_dtype != QFMT_F32 && out_dtype != QFMT_BF16) return fail(QFMT_EINVAL, "bad out_dtype %d", out_dtype);
  if (M == 0 || N == 0) return QFMT_OK;
  if (K % 128) return fail(QFMT_ESHAPE, "qmm_grouped: K=%lld must be a multiple of 128", (long long)K);
  if (M > 65535LL * 128 / 2) return fail(QFMT_ESHAPE, "M=%lld too large for the grouped tile grid", (long long)M);
  const size_t need = qfmt_dev::qgemm_grouped_workspace_bytes(M, K, E);
  if (!workspace || workspace_bytes < need)
    return fail(QFMT_ENOSPACE, "workspace of %zu bytes, qmm_grouped needs %zu", workspace_bytes, need);
  if ((st = check_ptr(codes, fmt == QFMT_MXFP4 ? 32 : 16, "codes"))) return st;
  if ((st = check_ptr(scales, 4, "scales"))) return st;
  if ((st = check_ptr(x, 16, "x"))) return st;
  if ((st = check_ptr(out, 16, "out"))) return st;
  if ((st = check_ptr(expert_idx, 4, "expert_idx"))) return st;
  if ((st = check_ptr(workspace, 128, "workspace"))) return st;
  int err = QFMT_OK;
  const int sms = device_sms(&err);
  if (err) return err;
  return cuda_status(qfmt_dev::launch_qgemm_grouped(fmt, codes, scales, x, expert_idx, out, out_dtype == QFMT_F32, M, N,
                                                    K, E, workspace, static_cast<cudaStream_t>(stream), sms),
                     "qmm_grouped launch");
}

int qfmt_quantize(int fmt, const void* x, int x_dtype, void* codes, void* scales, int64_t M, int64_t K,
                  void* stream) {
  clear_error();
  int st = check_group(fmt, 0);
  if (st) return st;
  if (fmt != QFMT_MXFP4 && fmt != QFMT_MXFP8_E4M3 && fmt != QFMT_MXFP8_E5M2)
    return fail(QFMT_EUNSUPPORTED, "qfmt_quantize takes mxfp4, mxfp8 E4M3 or E5M2 (format %d)", fmt);
  if ((st = check_shape(fmt, 0, M, K))) return st;
  if (x_dtype != QFMT_F32 && x_dtype != QFMT_BF16) return fail(QFMT_EINVAL, "bad x_dtype %d", x_dtype);
  if (M == 0 || K == 0) return QFMT_OK;
  if ((st = check_ptr(x, 16, "x"))) return st;
  if ((st = check_ptr(codes, 16, "codes"))) return st;
  if ((st = check_ptr(scales, 1, "scales"))) return st;
  return cuda_status(qfmt_dev::launch_quantize(fmt, x, x_dtype == QFMT_F32, codes, scales, M, K,
                                               static_cast<cudaStream_t>(stream)),
                     "quantize launch");
}

size_t qmm_a8_workspace_bytes(int fmt, int64_t M, int64_t K) {
  clear_error();
  if (fmt != QFMT_MXFP4 && fmt != QFMT_MXFP8_E4M3 && fmt != QFMT_MXFP8_E5M2) return 0;
  if (M <= 0 || K <= 0 || K % 128) return 0;
  return qfmt_dev::qgemm_a8_workspace_bytes(M, K);
}

int qmm_a8(int fmt, const void* codes, const void* scales, const void* x, void* out, int out_dtype, int64_t M,
           int64_t N, int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  int st = check_group(fmt, 0);
  if (st) return st;
  if (fmt != QFMT_MXFP4 && fmt != QFMT_MXFP8_E4M3 && fmt != QFMT_MXFP8_E5M2)
    return fail(QFMT_EUNSUPPORTED, "qmm_a8 takes mxfp4, mxfp8 E4M3 or E5M2 weights (format %d)", fmt);
  if ((st = check_shape(fmt, M, N, K))) return st;
  if (out_dtype != QFMT_F32 && out_dtype != QFMT_BF16) return fail(QFMT_EINVAL, "bad out_dtype %d", out_dtype);
  if (M == 0 || N == 0) return QFMT_OK;
  if (K % 128) return fail(QFMT_ESHAPE, "qmm_a8: K=%lld must be a multiple of 128", (long long)K);
  if (M > 65535LL * 128) return fail(QFMT_ESHAPE, "M=%lld: more than 65535 row tiles of 128", (long long)M);
  const size_t need = qfmt_dev::qgemm_a8_workspace_bytes(M, K);
  if (!workspace || workspace_bytes < need)
    return fail(QFMT_ENOSPACE, "workspace of %zu bytes, qmm_a8 needs %zu", workspace_bytes, need);
  if ((st = check_ptr(codes, fmt == QFMT_MXFP4 ? 32 : 16, "codes"))) return st;
  if ((st = check_ptr(scales, 4, "scales"))) return st;
  if ((st = check_ptr(x, 16, "x"))) return st;
  if ((st = check_ptr(out, 16, "out"))) return st;
  if ((st = check_ptr(workspace, 128, "workspace"))) return st;
  int err = QFMT_OK;
  const int sms = device_sms(&err);
  if (err) return err;
  return cuda_status(qfmt_dev::launch_qgemm_a8(fmt, codes, scales, x, out, out_dtype == QFMT_F32, M, N, K, workspace,
                                               static_cast<cudaStream_t>(stream), sms),
                     "qmm_a8 launch");
}

size_t qmm_a4_workspace_bytes(int fmt, int64_t M, int64_t K) {
  clear_error();
  if (fmt != QFMT_MXFP4 && fmt != QFMT_NVFP4) return 0;
  if (M <= 0 || K <= 0 || K % 256) return 0;
  return qfmt_dev::qgemm_a4_workspace_bytes(fmt, M, K);
}

int qmm_a4(int fmt, const void* codes, const void* scales, float global_scale, const void* x, void* out,
           int out_dtype, int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  int st = check_group(fmt, 0);
  if (st) return st;
  if (fmt != QFMT_MXFP4 && fmt != QFMT_NVFP4)
    return fail(QFMT_EUNSUPPORTED, "qmm_a4 takes mxfp4 or nvfp4 weights (format %d)", fmt);
  if ((st = check_shape(fmt, M, N, K))) return st;
  if (out_dtype != QFMT_F32 && out_dtype != QFMT_BF16) return fail(QFMT_EINVAL, "bad out_dtype %d", out_dtype);
  if (M == 0 || N == 0) return QFMT_OK;
  if (K % 256) return fail(QFMT_ESHAPE, "qmm_a4: K=%lld must be a multiple of 256", (long long)K);
  if (M > 65535LL * 128) return fail(QFMT_ESHAPE, "M=%lld: more than 65535 row tiles of 128", (long long)M);
  const size_t need = qfmt_dev::qgemm_a4_workspace_bytes(fmt, M, K);
  if (!workspace || workspace_bytes < need)
    return fail(QFMT_ENOSPACE, "workspace of %zu bytes, qmm_a4 needs %zu", workspace_bytes, need);
  if ((st = check_ptr(codes, 16, "codes"))) return st;
  if ((st = check_ptr(scales, fmt == QFMT_NVFP4 ? 16 : 8, "scales"))) return st;
  if ((st = check_ptr(x, 16, "x"))) return st;
  if ((st = check_ptr(out, 16, "out"))) return st;
  if ((st = check_ptr(workspace, 128, "workspace"))) return st;
  int err = QFMT_OK;
  const int sms = device_sms(&err);
  if (err) return err;
  return cuda_status(qfmt_dev::launch_qgemm_a4(fmt, codes, scales, global_scale, x, out, out_dtype == QFMT_F32, M, N,
                                               K, workspace, static_cast<cudaStream_t>(stream), sms),
                     "qmm_a4 launch");
}

size_t qmm_workspace_bytes(int fmt, int64_t M, int64_t K) {
  clear_error();
  if (!valid_format(fmt) || M < 0 || K < 0) return 0;
  return qfmt_dev::qgemm_mx_supported(fmt, M, K) ? qfmt_dev::qgemm_mx_workspace_bytes(M, K) : 0;
}

}  // extern "C"
