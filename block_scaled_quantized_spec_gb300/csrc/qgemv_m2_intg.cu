// Decode GEMV (M <= 2) kernels of the integer formats: int4 affine, int4, int4_f16, mxint8, int8, int8_f16.
#include "qgemv_m2.cuh"

namespace qfmt_dev {
namespace gemv_m2 {
QFMT_M2_GROUP_DEF(intg, GroupInt)
}  // namespace gemv_m2
}  // namespace qfmt_dev
