// Launchers of the device kernels (internal to libqfmt).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qfmt_dev {

// out [N, K] float32 or bf16 <- dequant(codes, scales, glob).
cudaError_t launch_dequant(int fmt, const void* codes, const void* scales, float glob, void* out,
                           bool out_bf16, int64_t N, int64_t K, cudaStream_t st, int sms);

// Decode GEMV, 1 <= M <= 16: out [M, N] (bf16 or f32) = X [M, K] bf16 . W^T.
cudaError_t launch_qgemv(int fmt, const void* codes, const void* scales, float glob, const void* x,
                         void* out, bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st,
                         int sms);

// Register-direct decode GEMV for M <= 2 (when its staged activations fit).
bool qgemv_m2_fits(int fmt, int64_t M, int64_t K);
cudaError_t launch_qgemv_m2(int fmt, const void* codes, const void* scales, float glob, const void* x,
                            void* out, bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st,
                            int sms);

// Batch decode GEMV for 3 <= M <= 16, K split over a thread-block cluster.
bool qgemv_mb_fits(int fmt, int64_t M, int64_t K);
cudaError_t launch_qgemv_mb(int fmt, const void* codes, const void* scales, float glob, const void* x,
                            void* out, bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st,
                            int sms);

// Float32-activation path (CUDA cores, exact products), any M.
cudaError_t launch_qmm_f32x(int fmt, const void* codes, const void* scales, float glob,
                            const float* x, void* out, bool out_f32, int64_t M, int64_t N,
                            int64_t K, cudaStream_t st, int sms);

// Tensor-core GEMM (tcgen05), M > 16: out [M, N] = X [M, K] bf16 . W^T.
// Returns cudaErrorNotSupported when the device lacks tcgen05.
cudaError_t launch_qgemm_tc(int fmt, const void* codes, const void* scales, float glob,
                            const void* x, void* out, bool out_f32, int64_t M, int64_t N,
                            int64_t K, cudaStream_t st, int sms);

// The 2/3/5/6-bit integer formats (ids 21-32): dequant and the dequantizing
// matmul on CUDA cores (any M; bf16 or float32 activations).
bool is_sub_byte(int fmt);
cudaError_t launch_dequant_sub(int fmt, const void* codes, const void* scales, void* out, bool out_bf16, int64_t N,
                               int64_t K, cudaStream_t st, int sms);
cudaError_t launch_qmm_sub(int fmt, const void* codes, const void* scales, const void* x, bool x_f32, void* out,
                           bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st);

// Block-scaled tensor-core GEMM (tcgen05 kind::mxf8f6f4) for mxfp4 / mxfp8
// E4M3 / E5M2 weights: X is split into two MXFP8 E4M3 terms in `workspace`
// (qgemm_mx_workspace_bytes), then both go through the block-scaled MMA
// against the weights as stored.  M > 16, K a multiple of 128.
bool qgemm_mx_supported(int fmt, int64_t M, int64_t K);
size_t qgemm_mx_workspace_bytes(int64_t M, int64_t K);
cudaError_t launch_qgemm_mx(int fmt, const void* codes, const void* scales, const void* x, void* out, bool out_f32,
                            int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st, int sms);
// Decode GEMV on the same block-scaled MMA (M <= 16, K a multiple of 128 up to
// 1024, mxfp4 codes 32-byte aligned): weights as stored, activations split in
// the CTA; no workspace.
bool qgemv_mx_supported(int fmt, int64_t M, int64_t N, int64_t K, const void* codes, int sms);
// Expert-grouped rows on the block-scaled GEMM: a stacked [E N, K] MX weight,
// row m against expert idx[m]; rows of one expert share the expert's tiles.
size_t qgemm_grouped_workspace_bytes(int64_t M, int64_t K, int64_t E);
int qgemm_grouped_max_experts();
cudaError_t launch_qgemm_grouped(int fmt, const void* codes, const void* scales, const void* x, const int32_t* idx,
                                 void* out, bool out_f32, int64_t M, int64_t N, int64_t K, int64_t E, void* workspace,
                                 cudaStream_t st, int sms);
// The quantized-activation product: X packed to MXFP8 E4M3 (the packer's
// rule) in `workspace`, then one block-scaled MMA per block (any M >= 1).
size_t qgemm_a8_workspace_bytes(int64_t M, int64_t K);
cudaError_t launch_qgemm_a8(int fmt, const void* codes, const void* scales, const void* x, void* out, bool out_f32,
                            int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st, int sms);
// The all-FP4 product: X packed in W's FP4 family in `workspace` (MXFP4
// against mxfp4, one kind::mxf4 MMA per 64 K; NVFP4 with its global against
// nvfp4, kind::mxf4nvf4), any M >= 1, K a multiple of 256.
size_t qgemm_a4_workspace_bytes(int fmt, int64_t M, int64_t K);
cudaError_t launch_qgemm_a4(int fmt, const void* codes, const void* scales, float global_scale, const void* x,
                            void* out, bool out_f32, int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st,
                            int sms);
// The activation quantizer: X [M, K] (bf16 or float32) -> codes + E8M0 scales
// of mxfp4 / mxfp8 E4M3 / E5M2 in the weight layout, or (E4M3, mxfp4) the
// workspace layout of the quantized-activation products.
cudaError_t launch_quantize(int fmt, const void* x, bool x_f32, void* codes, void* scales, int64_t M, int64_t K,
                            cudaStream_t st);
cudaError_t launch_quantize_e4m3_atoms(const void* x, void* codes, void* atoms, int64_t M, int64_t K,
                                       cudaStream_t st);
cudaError_t launch_quantize_mxfp4_atoms(const void* x, void* codes, void* atoms, int64_t M, int64_t K,
                                        cudaStream_t st);
// NVFP4 activations for the all-FP4 product over nvfp4: per-CTA maxima of |x|
// into `partials` (quantize_nvfp4_partials(M, K) <= 1024 floats), then codes [M, K/2],
// E4M3 scale atoms (4 blocks of 16 a cell) and the global into *g_out.
int quantize_nvfp4_partials(int64_t M, int64_t K);
cudaError_t launch_quantize_nvfp4_atoms(const void* x, void* codes, void* atoms, float* partials, float* g_out,
                                        int64_t M, int64_t K, cudaStream_t st);
cudaError_t launch_qgemv_mx(int fmt, const void* codes, const void* scales, const void* x, void* out, bool out_f32,
                            int64_t M, int64_t N, int64_t K, cudaStream_t st, int sms);
void set_mx_wait_limit_ns(uint64_t ns);
void set_mx_drop_arrivals(int on);
void set_mx_plan(int bn, int s);   // measurement hook: force the tile width (224/256) and K split (1-4); 0 = planner
void set_mx_tall(int v);           // measurement hook: quantized-activation GEMM tall tiles: 0 = planner, 1 = never, 2 = where allowed
void set_tc_order(int v);          // measurement hook: bf16-decode GEMM tile order: 0 = host's choice, 1 = N first, 2 = M first
void set_mx_gemv(int off, int s);  // measurement hook: 1 = the mma.sync GEMVs for the MX formats; forced K split
cudaError_t read_and_clear_mx_status(unsigned int* status);

// Bounded-wait test hooks and the device status word of the tensor-core GEMM.
void set_wait_limit_ns(uint64_t ns);
void set_drop_arrivals(int on);
int drop_arrivals();
cudaError_t read_and_clear_device_status(unsigned int* status);
cudaError_t read_and_clear_gemv_status(unsigned int* status);

// Expert-routed decode GEMV: out[m, :] = x[m, :] . dequant(W[eidx[m] N .. + N))^T
// for a stacked [E N, K] weight (one single-row GEMV per row m).
cudaError_t launch_qgemv_gather(int fmt, const void* codes, const void* scales, float glob, const void* x,
                                const int32_t* eidx, void* out, bool out_f32, int64_t M, int64_t N, int64_t K,
                                int64_t E, cudaStream_t st);
cudaError_t read_and_clear_gather_status(unsigned int* status);

// Decode GEMV (M <= 2) over `count` (1..4) weight matrices sharing the
// activations, one launch; with gamma != nullptr the activations are
// RMS-normalised first (x * gamma / sqrt(mean(x^2) + eps)); with gate !=
// nullptr as well (count 1) they are also multiplied by silu(gate).
cudaError_t launch_qgemv_multi(int fmt, int count, const void* const* codes, const void* const* scales,
                               const float* globs, const int64_t* Ns, const void* x, const void* gamma, float eps,
                               void* const* outs, bool out_f32, int64_t M, int64_t K, cudaStream_t st,
                               const void* gate = nullptr);
uint64_t wait_limit_ns();

// Batch decode GEMV, 3 <= M <= 16: one decode of each weight block serves
// every activation row (qgemv_rb.cuh); where it fits (qgemv_rb_fits).
bool qgemv_rb_fits(int fmt, int64_t M, int64_t N, int64_t K, int sms);
cudaError_t launch_qgemv_rb(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                            bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st, int sms);
void set_gemv_rb(int off);   // measurement hook: 1 = the K-split batch GEMV instead
cudaError_t read_and_clear_rb_status(unsigned int* status);

}  // namespace qfmt_dev
