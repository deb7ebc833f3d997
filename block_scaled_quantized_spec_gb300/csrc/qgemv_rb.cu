// Batch decode GEMV (3 <= M <= 16): routes each format to the translation unit
// that instantiates its kernels (the kernel itself is in qgemv_rb.cuh).
#include "qgemv_rb.cuh"

namespace qfmt_dev {

static std::atomic<int> g_rb_off{0};

void set_gemv_rb(int off) { g_rb_off.store(off); }

// K in whole 32-code blocks, at least one a warp; the staged activations
// within a CTA's shared memory; and enough 16-row tiles for one CTA on at
// least half of the SMs (smaller launches take the K-split batch GEMV).  The
// (scale, bias) int4 formats stay on the K-split kernel: measured faster there
// (int4 affine, decode chains of 4096 x 4096 and 11008 x 4096 layers: 9.6
// against 10.5 us at M = 8, 22.2 against 28.6 us at M = 16).
bool qgemv_rb_fits(int fmt, int64_t M, int64_t N, int64_t K, int sms) {
  return !g_rb_off.load() && !fmt_is_i4(fmt) && M >= 3 && M <= 16 && K % 32 == 0 && K / 32 >= gemv_rb::WARPS &&
         K <= (int64_t(1) << 20) &&
         gemv_rb::smem_bytes(fmt, int(M), int(K)) <= size_t(227 * 1024) && (N + 15) / 16 >= int64_t(sms / 2);
}

cudaError_t launch_qgemv_rb(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                            bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st, int sms) {
  using namespace gemv_rb;
  const int m = int(M), n = int(N), k = int(K);
  if (fmt == MXFP4 || fmt == NVFP4 || fmt == MXFP4X2 || fmt == MXINT4 || fmt == FP4 || fmt == FP4_F16)
    return e2m1_launch(fmt, codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
  if (fmt == INT4_AFFINE || fmt == INT4 || fmt == INT4_F16 || fmt == MXINT8 || fmt == INT8 || fmt == INT8_F16)
    return intg_launch(fmt, codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
  return fp8_launch(fmt, codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
}

// A batch GEMV of any group whose activation copy did not land in time.
cudaError_t read_and_clear_rb_status(unsigned int* status) {
  unsigned int a = 0, b = 0, c = 0;
  cudaError_t e = gemv_rb::e2m1_status(&a);
  if (e == cudaSuccess) e = gemv_rb::intg_status(&b);
  if (e == cudaSuccess) e = gemv_rb::fp8_status(&c);
  *status = a | b | c;
  return e;
}

}  // namespace qfmt_dev
