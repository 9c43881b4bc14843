// Device-side NVFP4 codec: e2m1 element codes and e4m3 (E4M3FN) block scales.
//
// The reading stated with the C ABI: block scale = e4m3(amax / 6), codes =
// e2m1(v / scale), both quotients the correctly rounded fp32 ones, both
// conversions round to nearest with ties to even and saturate (448, 6); a
// block whose scale is 0 keeps all-zero codes; a negative value that rounds
// to zero keeps its sign. The first rocket blog page ("The CUTLASS grouped
// GEMM beats the scalar GEMV loop", section "Proof") checks the device
// quantizer byte for byte against a host codec; this file is the device half
// of that contract.
//
// How the device meets it without dividing: the conversions are the
// hardware's (`cvt.rn.satfinite` to e4m3x2 and e2m1x2: nearest-even,
// saturating, subnormal e4m3 codes, the sign of zero kept), and each quotient
// comes from an approximate reciprocal and one fused multiply-add
// refinement (Markstein's method), whose conversion equals that of the
// correctly rounded quotient (see block_quotient).
#pragma once
#include <cstdint>

namespace moe {

__device__ __forceinline__ float bf16_to_f32(uint32_t bits) { return __uint_as_float(bits << 16); }

// 1 / d, the hardware approximation (at most one ulp from the exact value).
__device__ __forceinline__ float rcp_approx(float d) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
  return r;
}

// v / d for the codec, given r within a few ulps of 1 / d: q0 = v r, the
// residual v - q0 d (exact: one fused multiply-add), then q0 + residual * r.
// For a bf16 v (8 significant bits) and an e4m3 d (4), v / d is either exact
// in fp32 (then it is the result) or far from every fp32 rounding midpoint
// and from every e2m1 / e4m3 rounding threshold compared with the refined
// error, so converting the result to e2m1 or e4m3 gives the code of the
// correctly rounded quotient. Checked for every nonzero e4m3 d, every bf16 v
// with |v| <= 9 d (the codec's range) in both signs and every r within three
// ulps of 1 / d; for d = 6 (the block scale), every finite bf16 v. The
// residual is formed as q0 d - v and subtracted, so that v = -0 gives -0 (a
// negative value that rounds to zero keeps its sign).
__device__ __forceinline__ float block_quotient(float v, float d, float r) {
  const float q0 = v * r;
  return fmaf(-fmaf(q0, d, -v), r, q0);
}

// e2m1 codes of two fp32 values (`lo` in the low nibble): nearest-even on
// {0, .5, 1, 1.5, 2, 3, 4, 6}, saturating at 6, sign of zero kept.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint16_t b;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(b)
      : "f"(hi), "f"(lo));
  return b;
}

// Block scale code of a block maximum amax >= 0: e4m3 of amax / 6,
// nearest-even, saturating at 448 (0x7E); 0 when amax / 6 rounds to zero.
__device__ __forceinline__ uint32_t block_scale_code(float amax) {
  const float q = block_quotient(amax, 6.0f, 1.0f / 6.0f);
  uint16_t b;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(b) : "f"(0.0f), "f"(q));
  return b & 0xFFu;
}

// The value of an e4m3 code (exact; the codes made here are 0x00 .. 0x7E).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)code));
  float f;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}

// NVFP4 codec for one 16-value block held by one lane: its block scale code
// and its eight packed code bytes (value 2i in the low nibble of byte i; bytes
// 0-3 in codes.x). `v` holds fp32 values exact in bf16.
__device__ __forceinline__ void quantize_block16(const float (&v)[16], uint2& codes, uint32_t& scale) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  scale = block_scale_code(amax);
  codes = make_uint2(0u, 0u);
  if (scale != 0u) {  // an underflowed block keeps all-zero codes
    const float d = e4m3_value(scale), r = rcp_approx(d);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      codes.x |= e2m1x2(block_quotient(v[2 * i], d, r), block_quotient(v[2 * i + 1], d, r)) << (8 * i);
      codes.y |= e2m1x2(block_quotient(v[8 + 2 * i], d, r), block_quotient(v[9 + 2 * i], d, r)) << (8 * i);
    }
  }
}

// Byte offset of scale (row m, column c) in a region of 128-row atoms with
// Kc scale columns: atoms run along K, then along rows; inside an atom,
// 16 bytes per row of a 32-row slab and 4 bytes per 32-row quarter.
__device__ __forceinline__ uint32_t sf_atom_offset(uint32_t m, uint32_t c, uint32_t Kc) {
  return ((m >> 7) * (Kc >> 2) + (c >> 2)) * 512u + (m & 31u) * 16u + ((m >> 5) & 3u) * 4u + (c & 3u);
}

}  // namespace moe
