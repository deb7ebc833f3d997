// Decode GEMV (M <= 2) kernels of the E2M1 and signed-nibble formats under E8M0 / E4M3 / float32 scales: mxfp4, nvfp4, mxfp4x2, mxint4.
#include "qgemv_m2.cuh"

namespace qfmt_dev {
namespace gemv_m2 {
QFMT_M2_GROUP_DEF(e2m1, GroupE2M1)
}  // namespace gemv_m2
}  // namespace qfmt_dev
