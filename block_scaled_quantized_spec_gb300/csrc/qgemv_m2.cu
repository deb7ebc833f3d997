// Decode GEMV for M <= 2: routes each format to the translation unit that
// instantiates its kernels (the kernel itself is in qgemv_m2.cuh).
#include "qgemv_m2.cuh"

namespace qfmt_dev {

bool qgemv_m2_fits(int fmt, int64_t M, int64_t K) {
  return M >= 1 && M <= 2 && K <= (int64_t(1) << 20) && gemv_m2::smem_bytes(fmt, int(M), int(K)) <= gemv_m2::SMEM_LIMIT;
}

cudaError_t launch_qgemv_m2(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                            bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st, int sms) {
  using namespace gemv_m2;
  const int m = int(M), n = int(N), k = int(K);
  if (GroupE2M1::has(fmt)) return e2m1_launch(fmt, codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
  if (GroupFp8::has(fmt)) return fp8_launch(fmt, codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
  return intg_launch(fmt, codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
}

cudaError_t launch_qgemv_gather(int fmt, const void* codes, const void* scales, float glob, const void* x,
                                const int32_t* eidx, void* out, bool out_f32, int64_t M, int64_t N, int64_t K,
                                int64_t E, cudaStream_t st) {
  using namespace gemv_m2;
  const int m = int(M), n = int(N), k = int(K), e = int(E);
  if (GroupE2M1::has(fmt)) return e2m1_gather(fmt, codes, scales, glob, x, eidx, out, out_f32, m, n, k, e, st);
  if (GroupFp8::has(fmt)) return fp8_gather(fmt, codes, scales, glob, x, eidx, out, out_f32, m, n, k, e, st);
  return intg_gather(fmt, codes, scales, glob, x, eidx, out, out_f32, m, n, k, e, st);
}

// The expert-routed kernels of every group: a set bit in any of them.
cudaError_t read_and_clear_gather_status(unsigned int* status) {
  unsigned int a = 0, b = 0, c = 0;
  cudaError_t e = gemv_m2::e2m1_status(&a);
  if (e == cudaSuccess) e = gemv_m2::intg_status(&b);
  if (e == cudaSuccess) e = gemv_m2::fp8_status(&c);
  *status = a | b | c;
  return e;
}

cudaError_t launch_qgemv_multi(int fmt, int count, const void* const* codes, const void* const* scales,
                               const float* globs, const int64_t* Ns, const void* x, const void* gamma, float eps,
                               void* const* outs, bool out_f32, int64_t M, int64_t K, cudaStream_t st,
                               const void* gate) {
  using namespace gemv_m2;
  Extra ex{};
  ex.count = count;
  int tiles = 0;
  for (int i = 0; i < 4; ++i) {
    const int j = i < count ? i : count - 1;   // unused slots repeat the last matrix
    ex.codes[i] = static_cast<const uint8_t*>(codes[j]);
    ex.scales[i] = static_cast<const uint8_t*>(scales[j]);
    ex.glob[i] = globs[j];
    ex.out[i] = outs[j];
    ex.n[i] = int(Ns[j]);
    ex.tile0[i] = tiles;
    if (i < count) tiles += int((Ns[i] + 15) / 16);
  }
  ex.tile0[4] = tiles;
  ex.gamma = static_cast<const uint16_t*>(gamma);
  ex.eps = eps;
  ex.gate = static_cast<const uint16_t*>(gate);
  const int m = int(M), k = int(K);
  const bool rms = gamma != nullptr, batch = count > 1;
  const int mode = gate != nullptr ? (RMS | GATE) : rms ? (batch ? (BATCH | RMS) : RMS) : BATCH;
  if (GroupE2M1::has(fmt)) return e2m1_multi(fmt, mode, ex, x, out_f32, m, k, tiles, st);
  if (GroupFp8::has(fmt)) return fp8_multi(fmt, mode, ex, x, out_f32, m, k, tiles, st);
  return intg_multi(fmt, mode, ex, x, out_f32, m, k, tiles, st);
}

}  // namespace qfmt_dev
