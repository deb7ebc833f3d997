// Batch decode GEMV (3 <= M <= 16) kernels of the 8-bit float formats: mxfp8 E4M3 / E5M2, nvfp8 and its twin, the legacy fp8.
#include "qgemv_rb.cuh"

namespace qfmt_dev {
namespace gemv_rb {
cudaError_t fp8_launch(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                        bool out_f32, int M, int N, int K, cudaStream_t st, int sms) {
  return GroupFp8::launch(fmt, codes, scales, glob, x, out, out_f32, M, N, K, st, sms);
}
cudaError_t fp8_status(unsigned int* status) { return GroupFp8::read_status(status); }
}  // namespace gemv_rb
}  // namespace qfmt_dev
