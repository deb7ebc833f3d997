/*
 * qfmt.h -- C ABI of libqfmt: block-scaled weight formats and the fused
 * dequantizing matmul  out[M,N] = X[M,K] . dequant(W[N,K])^T  on one GB300 GPU.
 *
 * Formats (metaltile PR #250, "spec-conformant nvfp4/mxfp4/mxfp8/nvfp8"
 * format list and codec commit; metaltile-std tests/qmm_gpu_correctness.rs
 * for the MLX-style int4 affine format):
 *
 *   fmt                 element            block  scale per block
 *   QFMT_MXFP4          E2M1 (4-bit)       32     E8M0 byte, 2^(b-127)
 *   QFMT_NVFP4          E2M1 (4-bit)       16     E4M3 byte x one FP32 global
 *   QFMT_MXFP8_E4M3     E4M3 (8-bit)       32     E8M0 byte
 *   QFMT_MXFP8_E5M2     E5M2 (8-bit)       32     E8M0 byte
 *   QFMT_NVFP8          E4M3 (8-bit)       16     FP32 (4 bytes)
 *   QFMT_INT4_AFFINE    unsigned 4-bit q   64     bf16 scale + bf16 bias (4 bytes)
 *   QFMT_NVFP8_F16      E4M3 (8-bit)       16     IEEE half (2 bytes): the fp16-scale
 *                                                 twin of nvfp8 (PR #250: the same element
 *                                                 and block, the scale stored as a 2-byte
 *                                                 half, rounded to nearest even with
 *                                                 subnormals kept)
 *   QFMT_MXINT8         signed int8 q      32     E8M0 byte: w = q * 2^(b-127), q the
 *                                                 two's-complement byte (PR #250, the MXINT
 *                                                 axis: a symmetric integer element; the
 *                                                 packer clamps q to +-127 and rounds half
 *                                                 away from zero; a stored -128 decodes as
 *                                                 -128)
 *   QFMT_MXINT4         signed 4-bit q     32     E8M0 byte: w = q * 2^(b-127), q the
 *                                                 two's-complement nibble (PR #250's MXINT4;
 *                                                 the packer clamps to +-7)
 *   QFMT_INT8           signed int8 q      64     FP32 (4 bytes): w = q * scale (PR #250's
 *                                                 symmetric int8, scale-only, +-127)
 *   QFMT_INT8_F16       signed int8 q      64     IEEE half (2 bytes): the fp16-scale twin
 *                                                 of QFMT_INT8
 *   QFMT_INT4           signed 4-bit q     64     FP32 (4 bytes): w = q * scale, q the
 *                                                 two's-complement nibble (PR #250's symmetric
 *                                                 intN, sign-extended from bit 3, +-7)
 *   QFMT_INT4_F16       signed 4-bit q     64     IEEE half (2 bytes): the fp16-scale twin
 *                                                 of QFMT_INT4
 *   QFMT_FP4            E2M1 (4-bit)       32     FP32 (4 bytes): PR #250's legacy float format,
 *                                                 s = amax/6 unsnapped
 *   QFMT_FP8_E4M3       E4M3 (8-bit)       32     FP32 (4 bytes): legacy, s = amax/448
 *   QFMT_FP8_E5M2       E5M2 (8-bit)       32     FP32 (4 bytes): legacy, s = amax/57344
 *   QFMT_FP4_F16, QFMT_FP8_E4M3_F16, QFMT_FP8_E5M2_F16: their fp16-scale twins
 *                                                 (the scale an IEEE half, 2 bytes)
 *   QFMT_INT2/3/5/6     signed N-bit q     64     FP32 (4 bytes): w = q * scale (PR #250's symmetric
 *                                                 intN, sign-extended from bit N-1, +-(2^(N-1)-1))
 *   QFMT_INT2/3/5/6_F16                     64     IEEE half (2 bytes): their fp16-scale twins
 *   QFMT_MXINT2/3/5/6   signed N-bit q     32     E8M0 byte: w = q * 2^(b-127) (PR #250's MXINT axis)
 *   QFMT_MXFP4X2        two E2M1 planes    32     two FP32 (8 bytes): the two-level residual
 *                                                 weight w = s0 e2m1(q0) + s1 e2m1(q1) (rlx-cpu
 *                                                 dequant_matmul_mxfp4x2); level 0 packs w with
 *                                                 s0 = amax/6, level 1 the float32 residual
 *                                                 w - s0 e2m1(q0) with s1 = amax(residual)/6
 *
 * Memory layouts (all row-major, no padding, little-endian):
 *   codes   [N, K/2] bytes for 4-bit formats (mxfp4, nvfp4, int4 affine, int4, mxint4, fp4): element k of a row sits in byte
 *           k/2, low nibble for even k (LSB-first; 8 codes per u32 word);
 *           [N, K] bytes for 8-bit formats;
 *           [N, K N_bits / 8] bytes for the 2/3/5/6-bit formats: one LSB-first
 *           bit stream per row, code k at bits [k N, k N + N) of the row's
 *           little-endian bit sequence (PR #250's sub-byte packing; K a
 *           multiple of 32 makes every row whole 32-bit words).
 *   scales  [N, ceil(K/block)] entries of the sizes above; int4 affine stores
 *           the (scale, bias) bf16 pair of each group adjacently:
 *           [N, ceil(K/64), 2].  K is a multiple of 32 for every format, so
 *           only the group-64 formats (int4 affine, int8, int4 and twins) can end in
 *           a ragged group (of 32 values, with its own scale and bias; PR
 *           #250: a ragged trailing block, the block count rounded up).
 *           mxfp4x2: codes [N, 2, K/2] (a row's plane-0 nibbles, then its
 *           plane-1 nibbles), scales [N, 2, K/32] float32 (a row's s0 of every
 *           block, then its s1 of every block).
 *   X       [M, K] bf16 (or f32 through qmm_ex), out [M, N] bf16 (or f32).
 *
 * Element values: E2M1 {0,.5,1,1.5,2,3,4,6} with sign bit 3; E4M3 bias 7,
 * subnormal m*2^-9, only S.1111.111 is NaN (max 448, no infinity); E5M2 is
 * the high byte of an IEEE half; E8M0 code b is 2^(b-127) (b = 0 gives the
 * float32 subnormal 2^-127, b = 255 NaN).
 *
 * Ownership and synchronisation: the caller allocates and frees every
 * buffer.  qfmt_pack works on host memory and is synchronous.  qfmt_dequant,
 * qmm and qmm_ex take device pointers, enqueue work on `stream` (a
 * cudaStream_t; NULL = the legacy default stream) and return without
 * waiting; their status reports argument and launch errors only.  They
 * launch with programmatic dependent launch: X is read and `out` written only
 * after every preceding kernel in the stream has completed, but the weight
 * codes and scales may be read while a preceding kernel that signals early
 * completion (griddepcontrol.launch_dependents, as this library's kernels do)
 * is still running, so such a kernel must not write them.  The
 * library keeps no handle and allocates no device memory.  Its global state
 * is a per-thread error message, one status word per device (written only
 * when a kernel's bounded wait expires; see qfmt_device_status) and the
 * process-wide test settings of qfmt_debug_set.
 *
 * Errors: every function returns a qfmt_status (or a size; see each), never
 * aborts and never throws.  qfmt_last_error() describes the last failure on
 * the calling thread.
 */
#ifndef QFMT_H
#define QFMT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QFMT_MXFP4 = 1,
  QFMT_NVFP4 = 2,
  QFMT_MXFP8_E4M3 = 3,
  QFMT_MXFP8_E5M2 = 4,
  QFMT_NVFP8 = 5,
  QFMT_INT4_AFFINE = 6,
  QFMT_NVFP8_F16 = 7,
  QFMT_MXINT8 = 8,
  QFMT_INT8 = 9,
  QFMT_INT8_F16 = 10,
  QFMT_INT4 = 11,
  QFMT_INT4_F16 = 12,
  QFMT_MXFP4X2 = 13,
  QFMT_MXINT4 = 14,
  QFMT_FP4 = 15,
  QFMT_FP4_F16 = 16,
  QFMT_FP8_E4M3 = 17,
  QFMT_FP8_E4M3_F16 = 18,
  QFMT_FP8_E5M2 = 19,
  QFMT_FP8_E5M2_F16 = 20,
  QFMT_INT2 = 21,
  QFMT_INT3 = 22,
  QFMT_INT5 = 23,
  QFMT_INT6 = 24,
  QFMT_INT2_F16 = 25,
  QFMT_INT3_F16 = 26,
  QFMT_INT5_F16 = 27,
  QFMT_INT6_F16 = 28,
  QFMT_MXINT2 = 29,
  QFMT_MXINT3 = 30,
  QFMT_MXINT5 = 31,
  QFMT_MXINT6 = 32
} qfmt_format;

typedef enum { QFMT_F32 = 0, QFMT_BF16 = 1 } qfmt_dtype;

typedef enum {
  QFMT_OK = 0,
  QFMT_EINVAL = -1,        /* unknown format/dtype, NULL pointer, bad global scale */
  QFMT_ESHAPE = -2,        /* negative size, or K not a multiple of 32 */
  QFMT_EALIGN = -3,        /* a device pointer not 16-byte aligned (scales: 4-byte) */
  QFMT_EUNSUPPORTED = -4,  /* a group size other than the format's block */
  QFMT_ECUDA = -5,         /* a CUDA launch or device query failed */
  QFMT_ETIMEOUT = -6,      /* a kernel's bounded pipeline wait expired (see qfmt_device_status) */
  QFMT_ENONFINITE = -7,    /* qfmt_pack: NaN/Inf weight, or a block scale overflowing float32 */
  QFMT_ENOSPACE = -8,      /* a caller workspace smaller than qmm_workspace_bytes() */
  QFMT_EINDEX = -9         /* qmm_gather met an expert index outside [0, E) (see qfmt_device_status) */
} qfmt_status;

/* Block (group) size along K of format `fmt` packed with `group` (0 = the
 * format's default; the only other accepted value is that default itself):
 * 16 for the nv formats, 64 for the int4 affine / int8 / int4 groups, 32 for
 * the rest (metaltile PR #250 format table).  0 for an unknown format or a
 * group the format does not take (qfmt_last_error says which). */
int qfmt_block_size(int fmt, int group);

/* Bytes of the codes / scales buffers of an [N, K] weight packed with `group`
 * (codes: K/2 or K bytes a row, mxfp4x2 K; scales: ceil(K/block) entries a
 * row of the entry size in the table).  SIZE_MAX on an unknown format, a
 * group the format does not take, or a shape qfmt_pack rejects (negative
 * size, K not a multiple of 32, 2^31 or more code rows); qfmt_last_error
 * says which. */
size_t qfmt_codes_bytes(int fmt, int64_t N, int64_t K, int group);
size_t qfmt_scales_bytes(int fmt, int64_t N, int64_t K, int group);

/*
 * qfmt_pack -- host packer: float32 W [N, K] (host) -> codes, scales (host
 * buffers of the sizes above) and *global_scale (nvfp4; 1.0f otherwise).
 * Per row and block along K (metaltile PR #250, commit "Foundation for the
 * spec-conformant ... formats"; rlx-cpu thunk/ops/quant.rs
 * lowp_compute_scales / lowp_snap_scale / lowp_quantize):
 *   amax -> raw scale amax/max_finite (1.0 for an all-zero block) -> snapped
 *   stored scale (E8M0 = the smallest power of two >= the raw scale; nvfp4:
 *   global = amax(W)/2688, micro = E4M3(amax_b/6/global); nvfp8: float32)
 *   -> codes = encode(w / effective scale), round to nearest, ties to the
 *   even code, saturating to the largest finite value.  int4 affine: scale =
 *   bf16((max-min)/15), bias = bf16(min), q = clamp(round_half_away((w-bias)/
 *   scale), 0, 15).  All arithmetic is float32 with one rounding per op.
 * `group` must be 0 (format default) or the format's block.  Returns
 * QFMT_ENONFINITE on NaN/Inf weights.  Multi-threaded, synchronous.
 */
int qfmt_pack(int fmt, const float* W, int64_t N, int64_t K, int group,
              void* codes, void* scales, float* global_scale);

/*
 * qfmt_dequant -- device: out[n,k] = dequant(W)[n,k] for all N*K elements
 * (metaltile PR #250, standalone dequant kernels: out[i] =
 * elem(code) * scale(block)).  out_dtype QFMT_F32 is bit-exact: the exact
 * value elem * scale (nvfp4: (e2m1 * e4m3) * global; int4 affine:
 * fmaf(scale, q, bias)) rounded once to float32, subnormals kept, overflow
 * to +-inf.  QFMT_BF16 rounds that float32 to bf16 (nearest even).
 * codes/out 16-byte aligned, scales 4-byte aligned.
 */
int qfmt_dequant(int fmt, const void* codes, const void* scales, float global_scale,
                 void* out, int out_dtype, int64_t N, int64_t K, int group,
                 void* stream);

/*
 * qmm -- device: out[M,N] (bf16) = X[M,K] (bf16) . dequant(W[N,K])^T with
 * float32 accumulation (metaltile PR #250 qgemv/qmm/qmm-MMA commits:
 * output[m,n] = sum_k dequant(weight[n,k]) * x[m,k]; rlx-cpu
 * dequant_matmul_nvfp4 for the nvfp4 value).  M <= 16 runs a decode GEMV
 * (for mxfp4 / mxfp8 with K a multiple of 128 up to 1024, on the
 * block-scaled tensor cores; otherwise the HBM-streaming mma.sync GEMV);
 * larger M the tensor-core GEMM that decodes the weights to bf16.  Result
 * within 2e-3 * sum_k |x||w| + 1e-6 of the exact value, before the final
 * rounding of the bf16 output.  M == 0 or N == 0 is a no-op; K == 0 writes
 * zeros.  No workspace is needed.
 */
int qmm(int fmt, const void* codes, const void* scales, float global_scale,
        const void* x, void* out, int64_t M, int64_t N, int64_t K, int group,
        void* stream);

/*
 * qmm_ex -- qmm with explicit activation and output dtypes (QFMT_BF16 or
 * QFMT_F32 each) and an optional device workspace.  A float32 X takes a
 * CUDA-core float32 path (exact products, float32 accumulation) at any M.
 * With bf16 X, M > 16, a format the block-scaled MMA reads as stored (mxfp4,
 * mxfp8 E4M3 / E5M2), K a multiple of 128 and a workspace of at least
 * qmm_workspace_bytes(fmt, M, K) bytes (128-byte aligned; mxfp4 codes 32-byte
 * aligned), the product runs on tcgen05.mma kind::mxf8f6f4 (rlx-cpu
 * thunk/ops/quant.rs lowp_scaled_matmul, acc += (a_s b_s) sum dec(a) dec(b);
 * metaltile PR #250's "Blackwell tcgen05 scaled-MMA (MXFP)"): X is first
 * split into two MXFP8 E4M3 terms in the workspace (exact for every
 * activation within 2^14 of its block's largest).  A smaller workspace there
 * is QFMT_ENOSPACE; NULL (or any other case) takes the paths of qmm.  The
 * workspace is scratch: its contents are not kept between calls, and calls
 * sharing one must be ordered on one stream.
 */
int qmm_ex(int fmt, const void* codes, const void* scales, float global_scale,
           const void* x, int x_dtype, void* out, int out_dtype,
           int64_t M, int64_t N, int64_t K, int group,
           void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes qmm_ex uses for the block-scaled GEMM at this format and
 * shape: 2 M K (the two E4M3 code planes of X) plus 2 M' K / 32 (their E8M0
 * scales, M' = M rounded up to 128), each part 1 KiB aligned; 0 where qmm_ex
 * takes no workspace (another format, M <= 16, K not a multiple of 128). */
size_t qmm_workspace_bytes(int fmt, int64_t M, int64_t K);

/*
 * qfmt_quantize -- device: an activation X [M, K] (bf16 or float32, per
 * x_dtype; 16-byte aligned) packed as a weight of `fmt` (QFMT_MXFP4,
 * QFMT_MXFP8_E4M3 or QFMT_MXFP8_E5M2): codes [M, K] bytes (mxfp4: [M, K/2],
 * 16-byte aligned) and E8M0 scales [M, K/32], the same bytes qfmt_pack gives
 * for that matrix (rlx-cpu thunk/ops/quant.rs lowp_compute_scales /
 * lowp_snap_scale / lowp_quantize, the activation side of lowp_scaled_matmul:
 * per block of 32, s = amax / max_finite in float32, 1.0 for a zero block;
 * the scale the smallest power of two >= s; codes the nearest-even,
 * saturating encoding of x / scale).  A block holding an infinity or a NaN
 * gets the scale 255 (NaN).  K a multiple of 32.  Asynchronous on `stream`.
 */
int qfmt_quantize(int fmt, const void* x, int x_dtype, void* codes, void* scales, int64_t M, int64_t K,
                  void* stream);

/*
 * qmm_a8 -- device, both operands quantized (rlx-cpu thunk/ops/quant.rs
 * lowp_scaled_matmul: acc += (a_s * b_s) * sum_k dec(a) dec(b)):
 *   out[M, N] = Q(X) . dequant(W)^T
 * with Q(X) the activation packed to MXFP8 E4M3 as qfmt_quantize packs it,
 * W mxfp4 / mxfp8 E4M3 / E5M2, one tcgen05.mma kind::mxf8f6f4 per block of
 * 32 (the FP8 rate; qmm_ex's exact path takes two).  This is a different
 * product from qmm's: the activation carries E4M3's rounding (up to 2^-4 of
 * each value).  Result within 2^-12 * sum_k |q(x)||w| + 1e-6 of the exact
 * Q(X) . W^T (float32 accumulation).  x bf16 [M, K]; out bf16 or float32
 * per out_dtype; K a multiple of 128; workspace of at least
 * qmm_a8_workspace_bytes(fmt, M, K) bytes, 128-byte aligned, else
 * QFMT_ENOSPACE (scratch: ordered on one stream between calls); mxfp4 codes
 * 32-byte aligned.  Any M >= 1.
 */
int qmm_a8(int fmt, const void* codes, const void* scales, const void* x, void* out, int out_dtype, int64_t M,
           int64_t N, int64_t K, void* workspace, size_t workspace_bytes, void* stream);
/* Workspace bytes of qmm_a8: align(M K) + align(M' K / 32), M' = M rounded
 * up to 128, each part 1 KiB aligned; 0 for another format or K not a
 * positive multiple of 128. */
size_t qmm_a8_workspace_bytes(int fmt, int64_t M, int64_t K);

/*
 * qmm_a4 -- device, the all-FP4 product (rlx-cpu thunk/ops/quant.rs
 * lowp_quantize on the activation, then lowp_scaled_matmul; metaltile PR
 * #250 names Blackwell tcgen05 scaled MMA over its MXFP / NVFP formats):
 *   out[M, N] = Q4(X) . dequant(W)^T
 * with Q4(X) the activation packed in W's FP4 family by the packer's rule:
 *   - W mxfp4: X as MXFP4 (E2M1 codes, E8M0 scale per 32, as qfmt_quantize
 *     packs it); one tcgen05.mma kind::mxf4 per 64 K;
 *   - W nvfp4 (global_scale its global): X as NVFP4 over the whole X as one
 *     tensor (its own global amax(X) / (6 * 448), an E4M3 scale per 16, E2M1
 *     codes); one kind::mxf4nvf4 per 64 K, the output times both globals.
 *     A non-finite X gives NaN outputs.
 * Both operands enter the tensor cores packed two codes to a byte, as stored.
 * The activation carries E2M1's rounding (one mantissa bit), a different
 * product from qmm's.  Result within 2^-12 * sum_k |q4(x)||w| + 1e-6 of the
 * exact Q4(X) . W^T (float32 accumulation).  x bf16 [M, K]; out bf16 or
 * float32 per out_dtype; K a multiple of 256 (else QFMT_ESHAPE); another
 * weight format gives QFMT_EUNSUPPORTED; global_scale is read for nvfp4 only.
 * Workspace of at least qmm_a4_workspace_bytes(fmt, M, K) bytes, 128-byte
 * aligned, else QFMT_ENOSPACE (scratch: ordered on one stream between calls);
 * after the call it holds Q4(X): the codes [M, K/2] at offset 0, then (1 KiB
 * aligned) the scales in 512-byte atoms of 128 rows x 4 blocks (16-byte chunk
 * r % 32 holds rows r, r + 32, r + 64, r + 96, byte j of each 4-byte word is
 * block j of the atom's 4), atoms ordered by 128-row tile then along K; for
 * nvfp4 then (1 KiB aligned) 1,024 float32 words of scratch and the
 * activation's global.  codes 16-byte, scales 8-byte (nvfp4: 16-byte)
 * aligned.  Any M >= 1.  Asynchronous on `stream`.
 */
int qmm_a4(int fmt, const void* codes, const void* scales, float global_scale, const void* x, void* out,
           int out_dtype, int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes, void* stream);
/* Workspace bytes of qmm_a4: align(M K / 2) + align(M' K / 32) (mxfp4) or
 * align(M' K / 16) + align(4100) (nvfp4), M' = M rounded up to 128, each part
 * 1 KiB aligned; 0 for another format or K not a positive multiple of 256. */
size_t qmm_a4_workspace_bytes(int fmt, int64_t M, int64_t K);

/*
 * qmm_noalloc -- qmm_ex's block-scaled tensor-core GEMM (mxfp4, mxfp8 E4M3 /
 * E5M2; M > 16; K a multiple of 128; bf16 X and out) for callers that cannot
 * allocate device memory for scratch: an inference engine's plugin interface
 * that hands an op only its inputs and outputs, or a latency-critical path
 * that cannot take cudaMalloc's implicit device-wide synchronisation.  It
 * allocates nothing.  The scratch (X split into two E4M3 code planes and
 * their scale atoms, qmm_workspace_bytes(fmt, M, K) bytes) lives in one
 * static device array of QMM_NOALLOC_SCRATCH_BYTES inside this library,
 * present on every GPU that loads the library until the process exits.
 * The method's pages have no counterpart to this call; the arithmetic and
 * the result are qmm_ex's with a workspace.
 *   - The first call on a device looks up the array's device address there
 *     (cudaGetSymbolAddress with that device current); make that first call
 *     before any stream capture.
 *   - Every call shares the array and leaves its contents behind; each call
 *     writes all the scratch it reads before reading it.  Calls that overlap
 *     on the GPU (on different streams) race on the array.
 *   - QFMT_EUNSUPPORTED for another format, M <= 16 or K not a multiple of
 *     128; QFMT_ENOSPACE when the scratch needed exceeds the array; codes
 *     32-byte aligned for mxfp4 (16 otherwise), else QFMT_EALIGN; the other
 *     arguments and errors as qmm (global_scale is ignored).
 */
#define QMM_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int qmm_noalloc(int fmt, const void* codes, const void* scales, float global_scale, const void* x, void* out,
                int64_t M, int64_t N, int64_t K, int group, void* stream);

/*
 * qmm_gather -- device, expert-routed rows (mixture of experts):
 *   out[m, n] (bf16) = sum_k X[m, k] (bf16) . dequant(W)[expert_idx[m] * N + n, k]
 * where the E experts' [N, K] weights are stacked row-wise into one packed
 * matrix W [E*N, K] (codes and scales laid out as for qmm with E*N rows; one
 * nvfp4 global scale for all experts).  (metaltile PR #250, the MoE
 * gather-qmm commit: the qmm with one indirection, weight row
 * expert_ids[m] * out_dim + n over one stacked packed tensor; rlx-cpu
 * thunk/ops/quant.rs lowp_scaled_grouped_matmul: one row per token against
 * its routed expert.)
 * expert_idx: device int32 [M], 4-byte aligned.  It is read only after every
 * preceding kernel in the stream has completed (it may be the router's
 * output), so this call's weight reads wait for that kernel too.  Each row
 * runs as its own decode GEMV: rows that share an expert are not grouped, so
 * the call suits decode batches.  Bounds: 1 <= E, E*N <= 2^31, M <= 65535, K
 * within the single-row GEMV's shared-memory plan (QFMT_EUNSUPPORTED
 * beyond).  An index outside [0, E) makes that row's output zero and is
 * reported by the next qfmt_device_status (QFMT_EINDEX).  Tolerance as qmm.
 */
int qmm_gather(int fmt, const void* codes, const void* scales, float global_scale,
               const void* x, const int32_t* expert_idx, void* out,
               int64_t M, int64_t N, int64_t K, int64_t E, int group, void* stream);

/*
 * qmm_grouped -- device, expert-routed rows grouped by expert (rlx-cpu
 * thunk/ops/quant.rs lowp_scaled_grouped_matmul; metaltile PR #250's MoE
 * gather-qmm: weight row expert_ids[m] * out_dim + n of one stacked packed
 * tensor): the product of qmm_gather, for prefill batches.  A routing kernel
 * buckets the rows by expert on the device (no host synchronisation), every
 * expert's rows run through the block-scaled tensor-core GEMM together (the
 * activation split into two MXFP8 E4M3 terms as in qmm_ex), so each expert's
 * weights are read once per 128 rows routed to it rather than once per row.
 * Formats mxfp4, mxfp8 E4M3 / E5M2; K a multiple of 128; 1 <= E <= 1024; out
 * bf16 or float32 per out_dtype; workspace of at least
 * qmm_grouped_workspace_bytes(fmt, M, K, E) bytes (128-byte aligned; scratch
 * ordered on one stream), else QFMT_ENOSPACE; mxfp4 codes 32-byte aligned.
 * expert_idx: device int32 [M], read after every preceding kernel in the
 * stream has completed; an index outside [0, E) zeroes its output row and is
 * reported by the next qfmt_device_status (QFMT_EINDEX).  Tolerance as qmm.
 */
int qmm_grouped(int fmt, const void* codes, const void* scales, const void* x, const int32_t* expert_idx, void* out,
                int out_dtype, int64_t M, int64_t N, int64_t K, int64_t E, void* workspace, size_t workspace_bytes,
                void* stream);
/* Workspace bytes of qmm_grouped: the routing tables ((E + 1) + R int32),
 * then qmm_ex's workspace for R rows, R = M + 127 min(E, M) rounded up to 128
 * (every expert's rows padded to whole 128-row tiles); 0 for another format,
 * K not a positive multiple of 128, or E outside 1..1024. */
size_t qmm_grouped_workspace_bytes(int fmt, int64_t M, int64_t K, int64_t E);

/*
 * qmm_batched -- device: `count` (1..4) products sharing one activation:
 *   out[i][M, N[i]] (bf16) = X[M, K] (bf16) . dequant(W_i[N[i], K])^T
 * (metaltile PR #250, the batched Q/K/V and batched-4 dequantizing GEMV
 * commits: one dispatch projects [Wq x | Wk x | Wv x] over a shared
 * activation, each matrix into its own output).  codes, scales,
 * global_scales, N and out are HOST arrays of `count` entries (device
 * pointers inside, each laid out as for qmm; the matrices may differ in N but
 * not in format, K or group).  M <= 2 runs one launch over every matrix's row
 * tiles; larger M runs one qmm per matrix.  Errors as qmm, per matrix;
 * QFMT_EINVAL for count outside 1..4 or a NULL array.  Tolerance as qmm.
 */
int qmm_batched(int fmt, int count, const void* const* codes, const void* const* scales,
                const float* global_scales, const int64_t* N, const void* x, void* const* out,
                int64_t M, int64_t K, int group, void* stream);

/*
 * qmm_rmsnorm -- device, RMSNorm fused in front of the decode GEMV:
 *   out[m, n] (bf16) = sum_k (x[m,k] * gamma[k] / sqrt(mean_k x[m,k]^2 + eps))
 *                      * dequant(W)[n, k]
 * (metaltile PR #250, the fused RMSNorm + dequantizing GEMV commit: phase 1
 * the sum of x^2 and its inverse root, phase 2 the GEMV over the normalised
 * activation x * norm_weight * inv_rms).  x bf16 [M, K], norm_weight (gamma)
 * bf16 [K], both 16-byte aligned; eps finite and >= 0.  M <= 2 (the decode
 * form; QFMT_EUNSUPPORTED beyond); K = 0 is QFMT_ESHAPE.  Result within
 * 2e-3 * sum_k |x~||w| + 1e-6 of the exact value, x~ the exactly normalised
 * activation.
 */
int qmm_rmsnorm(int fmt, const void* codes, const void* scales, float global_scale,
                const void* x, const void* norm_weight, float eps, void* out,
                int64_t M, int64_t N, int64_t K, int group, void* stream);

/*
 * qmm_gated_rmsnorm -- device, gated RMSNorm fused in front of the decode GEMV:
 *   out[m, n] (bf16) = sum_k (x[m,k] * gamma[k] * silu(gate[m,k])
 *                             / sqrt(mean_k x[m,k]^2 + eps)) * dequant(W)[n, k]
 * with silu(z) = z / (1 + e^-z) (metaltile PR #250, the fused gated-RMSNorm +
 * dequantizing GEMV commit: the silu gate times the per-row inverse RMS
 * times the norm weight, staged, then the GEMV).  The root mean square is of
 * x alone.  gate bf16 [M, K], 16-byte aligned (NULL is QFMT_EINVAL); every
 * other argument, limit and the tolerance as qmm_rmsnorm, x~ the exactly
 * gated and normalised activation.
 */
int qmm_gated_rmsnorm(int fmt, const void* codes, const void* scales, float global_scale, const void* x,
                      const void* gate, const void* norm_weight, float eps, void* out, int64_t M, int64_t N,
                      int64_t K, int group, void* stream);

/*
 * qfmt_device_status -- waits for `stream`, then reads and clears the
 * library's device status word for the current device.  Every pipeline wait
 * inside the tensor-core GEMM is bounded in time; when one expires the kernel
 * records it there, drains its in-flight copies and MMAs, frees its tensor
 * memory and exits without writing its output tile.  Returns QFMT_OK, or
 * QFMT_ETIMEOUT if any such kernel since the last call gave up, QFMT_EINDEX
 * if a qmm_gather row met an expert index outside [0, E), or QFMT_ECUDA.
 */
int qfmt_device_status(void* stream);

/*
 * qfmt_debug_set -- testing aid for the bounded waits (process-wide, applies
 * to launches made afterwards): key 1 sets the wait limit in nanoseconds
 * (value <= 0 restores the default of 2 s); key 2 with value 1 makes the GEMM's
 * decoder warps skip signalling their stages, so the MMA warp's waits expire
 * (value 0 restores normal operation); keys 3 and 4 force the block-scaled
 * GEMM's tile width (224 or 256) and K split (1-4), value 0 restoring its own
 * plan; key 5 with value 1 sends the MX formats' decode GEMV (M <= 16) to the
 * mma.sync kernels instead of the block-scaled tensor-core one, key 6 forces
 * that kernel's K split; key 7 with value 1 sends the batch decode GEMV
 * (3 <= M <= 16) to the K-split kernel; key 8 sets the order in which the
 * bf16-decode GEMM walks its tiles (0 its own choice, 1 N tiles first, 2 M
 * tiles first); key 9 sets the quantized-activation GEMM's 256-row tiles
 * (0 its own plan, 1 never, 2 wherever the plan has no K split and M > 128)
 * -- all for measurements and tests.  Returns QFMT_EINVAL for other keys and
 * values.
 */
int qfmt_debug_set(int key, int64_t value);

/* Human-readable description of the last failure on this thread ("" if none). */
const char* qfmt_last_error(void);

/* ABI version (major * 100 + minor). */
int qfmt_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QFMT_H */
