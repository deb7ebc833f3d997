// Prefill dequantizing GEMM, M > 16.  (Placeholder: 16-row slices through the
// decode GEMV; replaced by the tcgen05 kernel.)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace qfmt_dev {

cudaError_t launch_qgemm_tc(int fmt, const void* codes, const void* scales, float glob, const void* x,
                            void* out, bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st,
                            int sms) {
  for (int64_t m0 = 0; m0 < M; m0 += 16) {
    const int64_t mm = M - m0 < 16 ? M - m0 : 16;
    const void* xs = static_cast<const __nv_bfloat16*>(x) + m0 * K;
    void* os = out_f32 ? static_cast<void*>(static_cast<float*>(out) + m0 * N)
                       : static_cast<void*>(static_cast<__nv_bfloat16*>(out) + m0 * N);
    cudaError_t e = launch_qgemv(fmt, codes, scales, glob, xs, os, out_f32, mm, N, K, st, sms);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace qfmt_dev
