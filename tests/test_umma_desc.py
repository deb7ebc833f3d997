"""The tensor-core descriptor encoders (csrc/umma_desc.h), pinned on the CPU.

The header is plain C++: a small host program built here with g++ prints
each encoder's output for a set of arguments, and every field is checked
against the bit positions the PTX ISA's tcgen05 sections give (instruction
descriptor of kind::f16, kind::mxf8f6f4, kind::mxf4 and kind::mxf4nvf4 with block scaling; shared-memory
matrix descriptor), restated below field by field.  A wrong shift or mask in
the encoder fails here before any kernel built on it runs on a GPU.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
HDR = os.path.join(os.path.dirname(HERE), "block_scaled_quantized_spec_gb300", "csrc", "umma_desc.h")

PROG = r"""
#include <cstdio>
#include <initializer_list>
#include "umma_desc.h"
int main() {
  using namespace umma;
  const unsigned types[] = {F8F6F4_E4M3, F8F6F4_E5M2, F8F6F4_E2M1};
  for (unsigned a : types) for (unsigned b : types)
    for (unsigned m : {64u, 128u, 256u}) for (unsigned n : {8u, 64u, 224u, 256u})
      for (unsigned sa = 0; sa < 4; ++sa) for (unsigned sb = 0; sb < 4; ++sb)
        std::printf("mx %u %u %u %u %u %u %u\n", a, b, m, n, sa, sb, idesc_mxf8f6f4(a, b, m, n, sa, sb));
  for (unsigned m : {64u, 128u}) for (unsigned n : {8u, 224u, 256u}) for (unsigned sa : {0u, 2u})
    for (unsigned sb : {0u, 2u}) std::printf("m4 %u %u %u %u %u\n", m, n, sa, sb, idesc_mxf4(m, n, sa, sb));
  for (unsigned m : {64u, 128u}) for (unsigned n : {8u, 224u, 256u})
    std::printf("n4 %u %u %u\n", m, n, idesc_mxf4nvf4(m, n));
  for (unsigned m : {64u, 128u}) for (unsigned n : {16u, 128u, 224u, 256u})
    std::printf("bf %u %u %u\n", m, n, idesc_bf16(m, n));
  for (unsigned addr : {0u, 1024u, 0x12340u, 0x3FFF0u})
    for (unsigned lbo : {16u, 128u, 4096u}) for (unsigned sbo : {128u, 1024u, 0xFFF0u}) for (unsigned sw : {0u, 2u})
      std::printf("sd %u %u %u %u %llu\n", addr, lbo, sbo, sw, (unsigned long long)smem_desc(addr, lbo, sbo, sw));
  std::printf("sw %llu %llu\n", (unsigned long long)smem_desc_sw128(0x2400u), (unsigned long long)smem_desc_sf32x16(0x2400u));
  for (unsigned r = 0; r < 128; ++r) for (unsigned j = 0; j < 4; ++j) std::printf("sf %u %u %u\n", r, j, sf_atom_offset(r, j));
  return 0;
}
"""


def bits(v, lo, width):
    return (v >> lo) & ((1 << width) - 1)


@pytest.fixture(scope="module")
def encoded(tmp_path_factory):
    cxx = os.environ.get("CXX") or shutil.which("g++") or shutil.which("c++")
    if not cxx:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("umma")
    src, exe = d / "t.cpp", d / "t"
    src.write_text(PROG)
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", os.path.dirname(HDR), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    rows = {}
    for line in out.splitlines():
        tag, *vals = line.split()
        rows.setdefault(tag, []).append([int(v) for v in vals])
    return rows


def test_block_scaled_instruction_descriptor(encoded):
    # kind::mxf8f6f4 / mxf4 / mxf4nvf4 instruction descriptor (32 bits):
    #  0-1 reserved, 2 sparsity (0 dense), 3 reserved, 4-5 B scale-factor id,
    #  6 reserved, 7-9 A type, 10-12 B type, 13 negate A, 14 negate B,
    #  15 transpose A, 16 transpose B (0: K-major), 17-22 N >> 3,
    #  23 scale type (1: UE8M0), 24-28 M >> 4, 29-30 A scale-factor id,
    #  31 reserved
    # Operand type codes of kind::mxf8f6f4: E4M3 0, E5M2 1, E2M3 3, E3M2 4, E2M1 5.
    assert len(encoded["mx"]) == 3 * 3 * 3 * 4 * 16
    for a, b, m, n, sa, sb, d in encoded["mx"]:
        assert bits(d, 0, 4) == 0
        assert bits(d, 4, 2) == sb
        assert bits(d, 6, 1) == 0
        assert bits(d, 7, 3) == a and a in (0, 1, 5)
        assert bits(d, 10, 3) == b
        assert bits(d, 13, 4) == 0
        assert bits(d, 17, 6) == n >> 3
        assert bits(d, 23, 1) == 1
        assert bits(d, 24, 5) == m >> 4
        assert bits(d, 29, 2) == sa
        assert bits(d, 31, 1) == 0


def test_mxf4_instruction_descriptor(encoded):
    # kind::mxf4 (scale_vec::2X): the same fields; both types E2M1, which this
    # kind codes as 1; the scale-factor ids 0 or 2 (each instruction reads two
    # bytes of the 32-bit cell); bit 31 = 0 (dense, K = 64)
    assert len(encoded["m4"]) == 2 * 3 * 4
    for m, n, sa, sb, d in encoded["m4"]:
        assert bits(d, 0, 4) == 0 and bits(d, 4, 2) == sb and bits(d, 6, 1) == 0
        assert bits(d, 7, 3) == 1 and bits(d, 10, 3) == 1 and bits(d, 13, 4) == 0
        assert bits(d, 17, 6) == n >> 3 and bits(d, 23, 1) == 1 and bits(d, 24, 5) == m >> 4
        assert bits(d, 29, 2) == sa and bits(d, 31, 1) == 0


def test_mxf4nvf4_instruction_descriptor(encoded):
    # kind::mxf4nvf4 (scale_vec::4X): both types E2M1 (1), scale type UE4M3
    # (bit 23 = 0), both scale-factor ids 0 (the instruction reads the whole cell)
    assert len(encoded["n4"]) == 2 * 3
    for m, n, d in encoded["n4"]:
        assert bits(d, 0, 7) == 0 and bits(d, 7, 3) == 1 and bits(d, 10, 3) == 1 and bits(d, 13, 4) == 0
        assert bits(d, 17, 6) == n >> 3 and bits(d, 23, 1) == 0 and bits(d, 24, 5) == m >> 4
        assert bits(d, 29, 3) == 0


def test_bf16_instruction_descriptor(encoded):
    # kind::f16: 4-5 D format (1: F32), 7-9 A format (1: BF16), 10-12 B format
    # (1: BF16), 13-16 no negate / transpose, 17-22 N >> 3, 24-28 M >> 4
    for m, n, d in encoded["bf"]:
        assert bits(d, 0, 4) == 0 and bits(d, 4, 2) == 1 and bits(d, 6, 1) == 0
        assert bits(d, 7, 3) == 1 and bits(d, 10, 3) == 1 and bits(d, 13, 4) == 0
        assert bits(d, 17, 6) == n >> 3 and bits(d, 23, 1) == 0 and bits(d, 24, 5) == m >> 4
        assert bits(d, 29, 3) == 0


def test_shared_memory_descriptor(encoded):
    # 0-13 start address >> 4, 16-29 leading byte offset >> 4, 32-45 stride
    # byte offset >> 4, 46-48 fixed 0b001, 49-51 base offset (0), 52 leading
    # offset mode (0), 61-63 swizzle mode
    for addr, lbo, sbo, sw, d in encoded["sd"]:
        assert bits(d, 0, 14) == (addr >> 4) & 0x3FFF
        assert bits(d, 14, 2) == 0
        assert bits(d, 16, 14) == lbo >> 4
        assert bits(d, 30, 2) == 0
        assert bits(d, 32, 14) == sbo >> 4
        assert bits(d, 46, 3) == 1
        assert bits(d, 49, 12) == 0
        assert bits(d, 61, 3) == sw
    sw128, sf = encoded["sw"][0]
    # 128B swizzle: 8-row x 128-byte atoms 1024 bytes apart, swizzle mode 2
    assert bits(sw128, 0, 14) == 0x240 and bits(sw128, 32, 14) == 64 and bits(sw128, 61, 3) == 2
    # scale atom source of tcgen05.cp .32x128b: 8-row x 16-byte core matrices, 128 bytes apart, no swizzle
    assert bits(sf, 0, 14) == 0x240 and bits(sf, 32, 14) == 8 and bits(sf, 61, 3) == 0


def test_scale_atom_layout(encoded):
    # 128 rows x 4 K blocks in 512 bytes: 16-byte chunk r % 32, 4-byte word
    # r / 32 within it, byte j; every (row, block) lands on its own byte
    seen = set()
    for r, j, off in encoded["sf"]:
        assert off == 16 * (r % 32) + 4 * (r // 32) + j
        seen.add(off)
    assert seen == set(range(512))
