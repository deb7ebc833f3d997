// Batch decode GEMV (3 <= M <= 16) kernels of the integer formats: int4 affine, int4, int4_f16, mxint8, int8, int8_f16.
#include "qgemv_rb.cuh"

namespace qfmt_dev {
namespace gemv_rb {
cudaError_t intg_launch(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                        bool out_f32, int M, int N, int K, cudaStream_t st, int sms) {
  return GroupInt::launch(fmt, codes, scales, glob, x, out, out_f32, M, N, K, st, sms);
}
cudaError_t intg_status(unsigned int* status) { return GroupInt::read_status(status); }
}  // namespace gemv_rb
}  // namespace qfmt_dev
