// Decode GEMV (M <= 2) kernels of the 8-bit float formats: mxfp8 E4M3 / E5M2, nvfp8, nvfp8_f16.
#include "qgemv_m2.cuh"

namespace qfmt_dev {
namespace gemv_m2 {
QFMT_M2_GROUP_DEF(fp8, GroupFp8)
}  // namespace gemv_m2
}  // namespace qfmt_dev
