"""Oracle packer: float32 W [N, K] -> block-scaled codes + scales (TEST INFRASTRUCTURE ONLY).

An independent restatement of the packing the pages describe; the library's own
C++ packer must produce the same bytes.  All arithmetic is IEEE float32
(numpy float32 ops round once per operation, no contraction).

Steps, per row n and block b along K (metaltile PR #250, commit "Foundation for
the spec-conformant nvfp4/mxfp4/mxfp8/nvfp8 formats"; rlx-cpu
``thunk/ops/quant.rs`` ``lowp_compute_scales`` / ``lowp_snap_scale`` /
``lowp_quantize``):

1. amax = max |w| over the block;
2. raw scale s = amax / max_finite(element), or 1.0 for an all-zero block;
3. snap s to the stored scale grid (E8M0, E4M3 or float32);
4. quantize every element against the *effective* (decoded, snapped) scale:
   code = encode(w / eff), code 0 when eff == 0;
5. pack codes LSB-first (two 4-bit codes per byte, element 2i in the low
   nibble; one byte per 8-bit code).

Readings taken where the pages are silent:

* E8M0 snapping is ceil(log2 s): the smallest power of two >= amax/max_finite,
  so no element needs to clip.
* nvfp4 global scale = amax(W) / (6 * 448) (1.0 for an all-zero W), so the
  largest micro-scale lands at 448; micro-scale u = E4M3_RNE((amax_b / 6) /
  global); an all-zero block stores u = E4M3(1.0) = 0x38.
* Element encoders round to nearest, ties to the even code, saturating.
* nvfp8_f16, the fp16-scale twin of nvfp8 (PR #250, "fp16-scale axis": the
  same element and block, the per-block scale stored as a 2-byte IEEE half,
  rounded to nearest even with subnormals kept): scale = half(amax / 448).
* mxint8 (PR #250's MXINT axis: a symmetric signed integer element -- sign-
  extended from its top bit, clamped to +-(2^(N-1) - 1) -- under an E8M0 scale
  per 32): s = amax / 127 snapped up to a power of two as for mxfp8, q =
  clamp(round_half_away(w / s), -127, 127) stored as a two's-complement byte.
* mxint4 (PR #250's MXINT4: the signed nibble under an E8M0 scale per 32):
  as mxint8 with 7 in place of 127, the nibble stored LSB-first two per byte.
* int8 / int8_f16 (PR #250's symmetric integer formats: "Int8 (symmetric
  affine, scale-only, group 64)" on the FP32 per-group scale path, the int8
  codec symmetric at +-127; the fp16-scale axis gives int8 its half-scale
  twin): s = amax / 127 in float32 (1.0 for an all-zero group), stored raw
  (int8) or rounded to an IEEE half (int8_f16, as nvfp8_f16); q =
  clamp(round_half_away(w / eff), -127, 127), 0 where eff is 0 (a half that
  underflowed).  K that 64 does not divide leaves a ragged last group of 32
  with its own amax (the pages' own example: int8's group of 64 over a
  dimension of 96 tiles as a 64-block and a 32-block).
* int4 / int4_f16 (PR #250's symmetric int2-6 on the FP32 group-64 scale
  path, the intN codec sign-extending from bit N-1 and clamping to
  +-(2^(N-1) - 1); the fp16-scale twin): as int8 with 7 in place of 127, the
  4-bit two's-complement code stored LSB-first two per byte (the 4-bit
  bit-stream is the nibble layout).
* mxfp4x2, the two-level residual E2M1 weight of rlx-cpu
  ``dequant_matmul_mxfp4x2`` (w = s0 LUT[q0] + s1 LUT[q1], two E2M1 code
  planes, a float32 scale per plane and block): the pages print the decode
  only.  Reading of the encode: level 0 packs the block as an E2M1 block with
  the float32 scale s0 = amax / 6; level 1 packs the float32 residual
  r = w - s0 LUT[q0] (a float32 product, then a float32 difference) the same
  way with s1 = amax(r) / 6 (1.0 for an all-zero residual).  Block 32 (the MX
  block).  Layout: codes [N, 2, K/2] (a row's plane-0 nibbles, then its
  plane-1 nibbles), scales [N, 2, K/32] float32 (s0 of every block, then s1).
* fp4 / fp8_e4m3 / fp8_e5m2 (PR #250's legacy float formats: the E2M1 /
  E4M3 / E5M2 element under a float32 scale per group of 32, "the existing F32
  per-group scale path") and their fp16-scale twins *_f16: s = amax /
  max_finite(element) in float32 (1.0 for an all-zero group), stored raw or
  rounded once to an IEEE half (as nvfp8_f16); codes as step 4.
* int2 / int3 / int5 / int6 (PR #250's symmetric intN on the FP32 group-64
  scale path), their fp16-scale twins *_f16, and mxint2 / mxint3 / mxint5 /
  mxint6 (the signed N-bit element under an E8M0 scale per 32): as int4 /
  mxint4 with 2^(N-1) - 1 in place of 7; the N-bit two's-complement codes of
  a row form one LSB-first bit stream (code j in bits [jN, jN + N) of the
  row's little-endian bit sequence; a 4-bit stream is the nibble layout).  K
  a multiple of 32 makes every row a whole number of 32-bit words, so no code
  straddles two rows.
* int4 affine (MLX style, group 64): s = (max - min) / 15 (1.0 when 0), stored
  as bf16 (RNE); bias = bf16(min); q = clamp(round_half_away((w - b) / s), 0, 15);
  scale and bias are interleaved per group as bf16 pairs [N, ceil(K/64), 2].
* K is a multiple of 32.  A K that 64 does not divide leaves int4 affine a
  ragged trailing group of 32 values with its own statistics (metaltile PR
  #250 body: a group size that does not divide the dimension tiles with a
  ragged trailing block, n_blocks = ceil(dim / block_size), packer and kernel
  rounding up alike).
"""
from __future__ import annotations

import numpy as np

from . import codec

FORMATS = ("mxfp4", "nvfp4", "mxfp8_e4m3", "mxfp8_e5m2", "nvfp8", "int4_affine", "nvfp8_f16", "mxint8",
           "int8", "int8_f16", "int4", "int4_f16", "mxfp4x2", "mxint4",
           "fp4", "fp4_f16", "fp8_e4m3", "fp8_e4m3_f16", "fp8_e5m2", "fp8_e5m2_f16",
           "int2", "int3", "int5", "int6", "int2_f16", "int3_f16", "int5_f16", "int6_f16",
           "mxint2", "mxint3", "mxint5", "mxint6")
INTN = {f: int(f.split("_")[0][-1]) for f in FORMATS if f.split("_")[0] in ("int2", "int3", "int5", "int6",
                                                                            "mxint2", "mxint3", "mxint5", "mxint6")}
RAGGED = ("int4_affine", "int8", "int8_f16", "int4", "int4_f16",   # block 64: K may end in a group of 32
          "int2", "int3", "int5", "int6", "int2_f16", "int3_f16", "int5_f16", "int6_f16")
SYM_INT = RAGGED[1:]                                                # symmetric integers, float scale per 64

BLOCK = {"mxfp4": 32, "nvfp4": 16, "mxfp8_e4m3": 32, "mxfp8_e5m2": 32, "nvfp8": 16, "int4_affine": 64,
         "nvfp8_f16": 16, "mxint8": 32, "int8": 64, "int8_f16": 64, "int4": 64, "int4_f16": 64, "mxfp4x2": 32,
         "mxint4": 32, "fp4": 32, "fp4_f16": 32, "fp8_e4m3": 32, "fp8_e4m3_f16": 32, "fp8_e5m2": 32,
         "fp8_e5m2_f16": 32}
ELEM_BITS = {"mxfp4": 4, "nvfp4": 4, "mxfp8_e4m3": 8, "mxfp8_e5m2": 8, "nvfp8": 8, "int4_affine": 4, "nvfp8_f16": 8,
             "mxint8": 8, "int8": 8, "int8_f16": 8, "int4": 4, "int4_f16": 4,
             "mxfp4x2": 8, "mxint4": 4,                      # bits per weight (mxfp4x2: two nibbles)
             "fp4": 4, "fp4_f16": 4, "fp8_e4m3": 8, "fp8_e4m3_f16": 8, "fp8_e5m2": 8, "fp8_e5m2_f16": 8}
SCALE_BYTES = {"mxfp4": 1, "nvfp4": 1, "mxfp8_e4m3": 1, "mxfp8_e5m2": 1, "nvfp8": 4, "int4_affine": 4,
               "nvfp8_f16": 2, "mxint8": 1, "int8": 4, "int8_f16": 2, "int4": 4, "int4_f16": 2,
               "mxfp4x2": 8, "mxint4": 1,                    # bytes per block (mxfp4x2: s0 and s1)
               "fp4": 4, "fp4_f16": 2, "fp8_e4m3": 4, "fp8_e4m3_f16": 2, "fp8_e5m2": 4, "fp8_e5m2_f16": 2}
_ELEM = {"mxfp4": ("e2m1", codec.E2M1_MAX), "nvfp4": ("e2m1", codec.E2M1_MAX),
         "mxfp8_e4m3": ("e4m3", codec.E4M3_MAX), "mxfp8_e5m2": ("e5m2", codec.E5M2_MAX),
         "nvfp8": ("e4m3", codec.E4M3_MAX), "nvfp8_f16": ("e4m3", codec.E4M3_MAX), "mxint8": ("int8", 127.0),
         "int8": ("int8", 127.0), "int8_f16": ("int8", 127.0), "int4": ("int4", 7.0), "int4_f16": ("int4", 7.0),
         "mxint4": ("int4", 7.0),
         "fp4": ("e2m1", codec.E2M1_MAX), "fp4_f16": ("e2m1", codec.E2M1_MAX),
         "fp8_e4m3": ("e4m3", codec.E4M3_MAX), "fp8_e4m3_f16": ("e4m3", codec.E4M3_MAX),
         "fp8_e5m2": ("e5m2", codec.E5M2_MAX), "fp8_e5m2_f16": ("e5m2", codec.E5M2_MAX)}

for _f, _b in INTN.items():
    BLOCK[_f] = 32 if _f.startswith("mx") else 64
    ELEM_BITS[_f] = _b
    SCALE_BYTES[_f] = 1 if _f.startswith("mx") else (2 if _f.endswith("_f16") else 4)
    _ELEM[_f] = (f"int{_b}", float(2 ** (_b - 1) - 1))

F32 = np.float32


def codes_nbytes(fmt: str, n: int, k: int) -> int:
    return n * k * ELEM_BITS[fmt] // 8


def n_blocks(fmt: str, k: int) -> int:
    """Blocks per row: ceil(K / block) (only int4 affine can have a ragged last one)."""
    return -(-k // BLOCK[fmt])


def scales_nbytes(fmt: str, n: int, k: int) -> int:
    return n * n_blocks(fmt, k) * SCALE_BYTES[fmt]


def _pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[N, K] uint8 codes (0..15) -> [N, K/2] bytes, element 2i in the low nibble."""
    c = codes.astype(np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def pack_bits(codes: np.ndarray, bits: int) -> np.ndarray:
    """[N, K] codes of `bits` bits -> [N, K * bits / 8] bytes, one LSB-first bit stream per row."""
    c = np.asarray(codes, dtype=np.uint8)
    stream = ((c[..., None] >> np.arange(bits, dtype=np.uint8)) & 1).reshape(c.shape[0], -1)
    return np.packbits(stream, axis=1, bitorder="little")


def _quantize(w_blocks: np.ndarray, eff: np.ndarray, elem: str) -> np.ndarray:
    """codes = encode(w / eff) with eff broadcast over the block; eff == 0 -> code 0."""
    safe = np.where(eff == 0, F32(1.0), eff).astype(F32)
    v = (w_blocks / safe[..., None]).astype(F32)
    codes = codec.encode_rne_sat(v, elem)
    return np.where((eff == 0)[..., None], np.uint8(0), codes)


def pack(fmt: str, w: np.ndarray):
    """Pack float32 W [N, K].  Returns (codes bytes, scales bytes, global_scale float32).

    Raises ValueError on non-finite weights, K not a multiple of 32 (and of the
    block, except int4 affine's ragged last group), or a scale that overflows
    float32.
    """
    if fmt not in FORMATS:
        raise ValueError(f"unknown format {fmt!r}")
    w = np.ascontiguousarray(w, dtype=F32)
    n, k = w.shape
    blk = BLOCK[fmt]
    if k % 32 or (k % blk and fmt not in RAGGED):
        raise ValueError("K must be a multiple of 32 and of the block size (the group-64 formats: of 32)")
    if not np.all(np.isfinite(w)):
        raise ValueError("non-finite weight")
    if fmt == "int4_affine" and k % blk:
        # the ragged last group, padded with copies of its own first value:
        # its min and max, hence its scale, bias and codes, are unchanged
        kp = n_blocks(fmt, k) * blk
        wp = np.concatenate([w, np.repeat(w[:, (kp - blk):(kp - blk) + 1], kp - k, axis=1)], axis=1)
        c, s, g = _pack_int4_affine(wp.reshape(n, kp // blk, blk), n, kp)
        return np.ascontiguousarray(c[:, : k // 2]), s, g
    if fmt in SYM_INT and k % blk:
        # the ragged last group, padded with zeros: its amax, hence its scale and codes, are unchanged
        kp = n_blocks(fmt, k) * blk
        c, s, g = pack(fmt, np.concatenate([w, np.zeros((n, kp - k), F32)], axis=1))
        return np.ascontiguousarray(c[:, : codes_nbytes(fmt, 1, k)]), s, g
    wb = w.reshape(n, k // blk, blk)
    amax = np.max(np.abs(wb), axis=2).astype(F32)          # step 1
    glob = F32(1.0)

    if fmt == "int4_affine":
        return _pack_int4_affine(wb, n, k)
    if fmt == "mxfp4x2":
        return _pack_mxfp4x2(wb, n, k)

    elem, maxf = _ELEM[fmt]
    if fmt in ("mxfp4", "mxfp8_e4m3", "mxfp8_e5m2", "mxint8", "mxint4") or fmt.startswith("mxint"):
        s = np.where(amax > 0, amax / F32(maxf), F32(1.0)).astype(F32)   # step 2
        scode = codec.e8m0_encode_ceil(s)                                  # step 3
        eff = codec.E8M0_TABLE[scode].astype(F32)                          # exact power of two
        scales = scode
    elif fmt == "nvfp4":
        amax_t = F32(np.max(amax)) if amax.size else F32(0.0)
        glob = F32(amax_t / F32(6.0 * 448.0)) if amax_t > 0 else F32(1.0)
        t = ((amax / F32(6.0)).astype(F32) / glob).astype(F32)
        ucode = codec.encode_rne_sat(t, "e4m3")
        ucode = np.where(amax > 0, ucode, np.uint8(0x38)).astype(np.uint8)
        eff = (codec.E4M3_TABLE[ucode].astype(F32) * glob).astype(F32)
        scales = ucode
    elif fmt.endswith("_f16"):
        # the fp16-scale twin: amax / 448 rounded once to an IEEE half (nearest
        # even, subnormals kept, overflow to inf, rejected below)
        s = np.where(amax > 0, amax / F32(maxf), F32(1.0)).astype(F32)
        with np.errstate(over="ignore"):
            h = s.astype(np.float16)
        eff = h.astype(F32)
        scales = h
    else:  # nvfp8 and the legacy float formats: float32 scale stored raw
        s = np.where(amax > 0, amax / F32(maxf), F32(1.0)).astype(F32)
        eff = s
        scales = s
    if not np.all(np.isfinite(eff)):
        raise ValueError("scale overflows float32")

    if elem.startswith("int"):   # symmetric integer element: round half away from zero, clamp to +-maxf
        safe = np.where(eff == 0, F32(1.0), eff).astype(F32)
        v = (wb / safe[..., None]).astype(F32)
        q = np.clip(_round_half_away(v), -maxf, maxf)
        q = np.where((eff == 0)[..., None], 0, q).astype(np.int8).reshape(n, k)
        scales_b = np.ascontiguousarray(scales).view(np.uint8).reshape(n, -1)
        bits = ELEM_BITS[fmt]
        if bits == 4:           # 4-bit two's complement, two per byte
            return _pack_nibbles(q.view(np.uint8) & np.uint8(0x0F)), scales_b, F32(glob)
        if bits == 8:
            return q.view(np.uint8), scales_b, F32(glob)
        return pack_bits(q.view(np.uint8) & np.uint8((1 << bits) - 1), bits), scales_b, F32(glob)
    codes = _quantize(wb, eff, elem).reshape(n, k)                        # step 4
    codes_b = _pack_nibbles(codes) if ELEM_BITS[fmt] == 4 else codes.astype(np.uint8)
    scales_b = np.ascontiguousarray(scales).view(np.uint8).reshape(n, -1)
    return codes_b, scales_b, F32(glob)


def _pack_mxfp4x2(wb: np.ndarray, n: int, k: int):
    planes, scales = [], []
    r = wb.astype(F32)
    for _level in range(2):
        amax = np.max(np.abs(r), axis=2).astype(F32)
        s = np.where(amax > 0, amax / F32(6.0), F32(1.0)).astype(F32)
        if not np.all(np.isfinite(s)):
            raise ValueError("scale overflows float32")
        c = _quantize(r, s, "e2m1")                                    # 0 where s underflowed to 0
        planes.append(_pack_nibbles(c.reshape(n, k)))
        scales.append(s)
        approx = (s[..., None] * codec.E2M1_TABLE[c].astype(F32)).astype(F32)
        r = (r - approx).astype(F32)                                   # the residual, float32
    codes = np.stack(planes, axis=1).reshape(n, k)                     # [N, 2, K/2]
    sc = np.ascontiguousarray(np.stack(scales, axis=1)).view(np.uint8).reshape(n, -1)   # [N, 2, nb] f32
    return codes, sc, F32(1.0)


def _round_half_away(v: np.ndarray) -> np.ndarray:
    a = np.abs(v.astype(np.float64))
    return np.copysign(np.floor(a + 0.5), v)


def _pack_int4_affine(wb: np.ndarray, n: int, k: int):
    mn = np.min(wb, axis=2).astype(F32)
    mx = np.max(wb, axis=2).astype(F32)
    s = ((mx - mn).astype(F32) / F32(15.0)).astype(F32)
    s = np.where(s == 0, F32(1.0), s).astype(F32)
    if not np.all(np.isfinite(s)):
        raise ValueError("scale overflows float32")
    s_bits = codec.bf16_round(s)
    b_bits = codec.bf16_round(mn)
    s_b = codec.decode_bf16(s_bits).astype(F32)
    b_b = codec.decode_bf16(b_bits).astype(F32)
    safe = np.where(s_b == 0, F32(1.0), s_b).astype(F32)
    v = ((wb - b_b[..., None]).astype(F32) / safe[..., None]).astype(F32)
    q = np.clip(_round_half_away(v), 0, 15).astype(np.uint8)
    q = np.where((s_b == 0)[..., None], np.uint8(0), q)
    codes_b = _pack_nibbles(q.reshape(n, k))
    pair = np.stack([s_bits, b_bits], axis=-1).astype(np.uint16)     # [N, K/64, 2]
    scales_b = np.ascontiguousarray(pair).view(np.uint8).reshape(n, -1)
    return codes_b, scales_b, F32(1.0)
