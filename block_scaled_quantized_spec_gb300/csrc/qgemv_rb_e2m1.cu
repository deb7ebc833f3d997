// Batch decode GEMV (3 <= M <= 16) kernels of the E2M1 and signed-nibble formats: mxfp4, nvfp4, mxfp4x2, mxint4, fp4, fp4_f16.
#include "qgemv_rb.cuh"

namespace qfmt_dev {
namespace gemv_rb {
cudaError_t e2m1_launch(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                        bool out_f32, int M, int N, int K, cudaStream_t st, int sms) {
  return GroupE2M1::launch(fmt, codes, scales, glob, x, out, out_f32, M, N, K, st, sms);
}
cudaError_t e2m1_status(unsigned int* status) { return GroupE2M1::read_status(status); }
}  // namespace gemv_rb
}  // namespace qfmt_dev
