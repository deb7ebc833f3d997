// qmm_noalloc: the block-scaled tensor-core GEMM with its scratch in a fixed
// array of this library instead of a caller workspace.
//
// Some callers cannot allocate device memory for an op's scratch: an
// inference engine whose plugin interface hands the op only its input and
// output buffers (the engine owns every other byte of device memory), or a
// latency-critical path that cannot afford cudaMalloc's implicit
// device-wide synchronisation.  For them qmm_noalloc runs the same
// activation split and block-scaled GEMM as qmm_ex with a workspace, keeping
// the split activations in g_noalloc_scratch, a file-scope device array of
// QMM_NOALLOC_SCRATCH_BYTES.  That array exists on every GPU that loads this
// library, for as long as the process runs.
//
// Host code cannot pass the array's name to a kernel: on the host it stands
// for a host-side shadow, not a device address.  The first call on each
// device therefore asks the runtime for the device address
// (cudaGetSymbolAddress, with that device current) and keeps it.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"
#include "qfmt_internal.h"

using namespace qfmt;

namespace {

constexpr size_t SCRATCH_BYTES = size_t(QMM_NOALLOC_SCRATCH_BYTES);

// The split activations of one call (two E4M3 code planes and their scale
// atoms).  Every call overwrites what it reads before reading it, so nothing
// here needs to start at zero; calls that run at the same time on the GPU
// (on different streams) share it and race.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SCRATCH_BYTES];

std::mutex g_mu;
void* g_addr[64];   // device address of g_noalloc_scratch per device, once looked up

// Device address of the scratch array on the current device (looked up on the
// first call there); nullptr with the failure recorded on error.
void* scratch_address(int* st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *st = fail(QFMT_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    return nullptr;
  }
  if (dev < 0 || dev >= 64) {
    *st = fail(QFMT_ECUDA, "device index %d out of range", dev);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      *st = fail(QFMT_ECUDA, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
      return nullptr;
    }
    g_addr[dev] = p;
  }
  return g_addr[dev];
}

}  // namespace

extern "C" int qmm_noalloc(int fmt, const void* codes, const void* scales, float global_scale, const void* x,
                           void* out, int64_t M, int64_t N, int64_t K, int group, void* stream) {
  clear_error();
  (void)global_scale;   // the MX formats have no global scale
  int st = check_group(fmt, group);
  if (st) return st;
  if ((st = check_shape(fmt, M, N, K))) return st;
  if (M == 0 || N == 0) return QFMT_OK;
  if (!qfmt_dev::qgemm_mx_supported(fmt, M, K))
    return fail(QFMT_EUNSUPPORTED,
                "qmm_noalloc takes mxfp4 / mxfp8 E4M3 / E5M2 with M > 16 and K a multiple of 128 "
                "(format %d, M=%lld, K=%lld)", fmt, (long long)M, (long long)K);
  const size_t need = qfmt_dev::qgemm_mx_workspace_bytes(M, K);
  if (need > SCRATCH_BYTES)
    return fail(QFMT_ENOSPACE, "M=%lld, K=%lld needs %zu bytes of scratch; the static scratch holds %zu",
                (long long)M, (long long)K, need, SCRATCH_BYTES);
  if ((st = check_ptr(codes, fmt == QFMT_MXFP4 ? 32 : 16, "codes"))) return st;
  if ((st = check_ptr(scales, 4, "scales"))) return st;
  if ((st = check_ptr(x, 16, "x"))) return st;
  if ((st = check_ptr(out, 16, "out"))) return st;
  void* ws = scratch_address(&st);
  if (!ws) return st;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(QFMT_ECUDA, "device query: %s", cudaGetErrorString(e));
  e = qfmt_dev::launch_qgemm_mx(fmt, codes, scales, x, out, false, M, N, K, ws, static_cast<cudaStream_t>(stream), sms);
  if (e != cudaSuccess) return fail(QFMT_ECUDA, "qmm_noalloc launch: %s", cudaGetErrorString(e));
  return QFMT_OK;
}
