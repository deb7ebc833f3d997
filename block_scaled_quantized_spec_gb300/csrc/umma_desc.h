// Descriptors of the 5th-generation tensor-core instructions (tcgen05), as
// plain constexpr C++ so that host code, device code and a host-only unit test
// compile the same encoders.  Field positions follow the PTX ISA's tcgen05
// sections ("Instruction descriptor" and "Shared memory descriptor").
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define QFMT_HD __host__ __device__
#else
#define QFMT_HD
#endif

namespace umma {

// Operand types of kind::mxf8f6f4 (the atype / btype field).
enum : uint32_t { F8F6F4_E4M3 = 0, F8F6F4_E5M2 = 1, F8F6F4_E2M3 = 3, F8F6F4_E3M2 = 4, F8F6F4_E2M1 = 5 };

// Instruction descriptor of tcgen05.mma ... kind::mxf8f6f4.block_scale, dense,
// both operands K-major, float32 accumulator, UE8M0 scale factors:
//   bits  4- 5  scale-factor data id of B (the byte of each 32-bit TMEM
//               scale cell read for this instruction's K block)
//   bits  7- 9  A type,  bits 10-12  B type
//   bit  13/14  negate A / B (0),  bit 15/16  A / B transposed (0: K-major)
//   bits 17-22  N >> 3
//   bit  23     scale type (1: UE8M0)
//   bits 24-28  M >> 4
//   bits 29-30  scale-factor data id of A
QFMT_HD constexpr uint32_t idesc_mxf8f6f4(uint32_t atype, uint32_t btype, uint32_t m, uint32_t n, uint32_t sfa_id,
                                          uint32_t sfb_id) {
  return ((sfb_id & 3u) << 4) | ((atype & 7u) << 7) | ((btype & 7u) << 10) | (((n >> 3) & 63u) << 17) | (1u << 23) |
         (((m >> 4) & 31u) << 24) | ((sfa_id & 3u) << 29);
}

// kind::mxf4.block_scale.scale_vec::2X: both operands E2M1 packed two to a
// byte (the type field's E2M1 is 1 in this kind), K = 64 per instruction, so
// each instruction reads two consecutive bytes of every row's 32-bit scale
// cell, starting at data id 0 or 2; bit 31 (0) selects the dense K of 64.
enum : uint32_t { MXF4_E2M1 = 1 };
QFMT_HD constexpr uint32_t idesc_mxf4(uint32_t m, uint32_t n, uint32_t sfa_id, uint32_t sfb_id) {
  return idesc_mxf8f6f4(MXF4_E2M1, MXF4_E2M1, m, n, sfa_id, sfb_id);
}

// kind::mxf4nvf4.block_scale.scale_vec::4X: both operands E2M1 packed, K = 64
// an instruction, one UE4M3 scale per 16 values (bit 23 = 0), so each
// instruction reads all four bytes of every row's 32-bit scale cell (id 0).
QFMT_HD constexpr uint32_t idesc_mxf4nvf4(uint32_t m, uint32_t n) {
  return idesc_mxf8f6f4(MXF4_E2M1, MXF4_E2M1, m, n, 0u, 0u) & ~(1u << 23);
}

// Instruction descriptor of tcgen05.mma ... kind::f16: float32 accumulator
// (bits 4-5 = 1), A and B bf16 (bits 7-9 and 10-12 = 1), both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24.
QFMT_HD constexpr uint32_t idesc_bf16(uint32_t m, uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (((n >> 3) & 63u) << 17) | (((m >> 4) & 31u) << 24);
}

// Shared-memory matrix descriptor:
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-48  fixed 0b001
//   bits 61-63  swizzle mode (0 none, 2 128-byte)
QFMT_HD constexpr uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(swizzle & 7u) << 61);
}

// K-major operand in the 128-byte-swizzle canonical layout: 8-row x 128-byte
// atoms 1024 bytes apart; the leading offset is unused by this layout.
QFMT_HD constexpr uint64_t smem_desc_sw128(uint32_t saddr) { return smem_desc(saddr, 16, 1024, 2); }

// Source of tcgen05.cp .32x128b: 32 rows of 16 bytes stored contiguously (four
// 8-row x 16-byte core matrices 128 bytes apart), no swizzle.
QFMT_HD constexpr uint64_t smem_desc_sf32x16(uint32_t saddr) { return smem_desc(saddr, 128, 128, 0); }

// Byte offset of scale factor (row r of a 128-row group, K block j of 4) inside
// its 512-byte atom: 32 chunks of 16 bytes, chunk r % 32 holding rows r % 32,
// + 32, + 64, + 96 (4 bytes each: K blocks 0..3).  tcgen05.cp .32x128b.warpx4
// copies the atom to 4 TMEM columns of every lane quadrant, where the MMA
// finds the scale of row r at lane r, column r / 32, byte j.
QFMT_HD constexpr uint32_t sf_atom_offset(uint32_t r, uint32_t j) { return 16u * (r & 31u) + 4u * ((r >> 5) & 3u) + (j & 3u); }

}  // namespace umma
