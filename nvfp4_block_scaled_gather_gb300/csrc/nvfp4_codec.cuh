// Device-side NVFP4 codec: e2m1 element codes and e4m3 (E4M3FN) block scales.
//
// Rounding follows the reading stated with the C ABI (round to nearest, ties
// to even, saturating): written here from the value sets, not from any
// vendor conversion routine. The first rocket blog page ("The CUTLASS grouped
// GEMM beats the scalar GEMV loop", section "Proof") checks the device
// quantizer byte for byte against a host codec; this file is the device half
// of that contract.
#pragma once
#include <cstdint>

namespace moe {

// e4m3 code -> fp32 (exact). E4M3FN: bias 7, subnormals m * 2^-9; the codes
// produced here never include 0x7F (NaN).
__device__ __forceinline__ float e4m3_decode(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xF, m = code & 0x7;
  if (e == 0) return (float)m * 0.001953125f;  // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// fp32 >= 0 -> e4m3 code, round to nearest even, saturating at 448 (0x7E).
__device__ __forceinline__ uint32_t e4m3_encode(float v) {
  if (!(v > 0.0f)) return 0u;
  if (v >= 448.0f) return 0x7Eu;
  if (v < 0.015625f) {                    // below 2^-6: subnormal grid, step 2^-9
    return (uint32_t)rintf(v * 512.0f);   // exact scaling; rintf is half-to-even
  }
  const uint32_t b = __float_as_uint(v);
  const uint32_t keep = (b >> 20) & 0x7u;   // top 3 mantissa bits
  const uint32_t rest = b & 0xFFFFFu;       // 20 dropped bits
  uint32_t code = ((((b >> 23) & 0xFFu) - 120u) << 3) | keep;
  if (rest > 0x80000u || (rest == 0x80000u && (keep & 1u))) code += 1u;  // carry may bump the exponent
  return code > 0x7Eu ? 0x7Eu : code;
}

// fp32 -> e2m1 code (bit 3 = sign), nearest with ties to the even code,
// saturating at 6. Grid {0, .5, 1, 1.5, 2, 3, 4, 6}; each midpoint belongs to
// the neighbour whose code is even.
__device__ __forceinline__ uint32_t e2m1_encode(float v) {
  const float a = fabsf(v);
  uint32_t m;
  if (a <= 0.25f) m = 0;
  else if (a < 0.75f) m = 1;
  else if (a <= 1.25f) m = 2;
  else if (a < 1.75f) m = 3;
  else if (a <= 2.5f) m = 4;
  else if (a < 3.5f) m = 5;
  else if (a <= 5.0f) m = 6;
  else m = 7;
  return m | (signbit(v) ? 8u : 0u);
}

__device__ __forceinline__ float bf16_to_f32(uint32_t bits) { return __uint_as_float(bits << 16); }

// e2m1 codes of two fp32 values, round to nearest even, saturating at 6: the
// hardware conversion (the same rounding as e2m1_encode, sign of zero kept);
// `lo` goes to the low nibble.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint16_t b;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(b)
      : "f"(hi), "f"(lo));
  return b;
}

// The e2m1 code of a bf16 value v divided by a nonzero e4m3 scale d, equal to
// e2m1 of the correctly rounded fp32 quotient fl(v / d) without dividing.
// Why it is exact: v has at most 8 significant bits and d at most 4, so
// v / d is either exactly one of the e2m1 rounding thresholds t (0.25, 0.75,
// ..., 5; then v = t d, a number of at most 7 bits) or at least ~2^-12 of t
// away from every one of them, far beyond fp32 rounding. With r ~ 1/d,
// q0 = v r and the residual e = v - q0 d (exact, one fused multiply-add), the
// corrected q1 = q0 + e r (Markstein's FMA-based refinement of a quotient) is
// within a fraction of an ulp of v / d: on the same side of every threshold,
// and exactly t at a tie, where the conversion applies ties-to-even. The sign
// is v's, so that -0 keeps its code (the sum in the refinement would give +0).
__device__ __forceinline__ float quotient_for_e2m1(float v, float d, float r) {
  const float q0 = v * r;
  return copysignf(fmaf(fmaf(-q0, d, v), r, q0), v);
}

// NVFP4 codec for eight values per lane, a lane pair (2j, 2j+1) holding one
// 16-value block: the pair's block scale (e4m3 of amax / 6, a correctly
// rounded division) and this lane's four packed code bytes (value 2i in the
// low nibble of byte i). `v` holds fp32 values exact in bf16. Every lane of
// the warp must take part (one shuffle).
__device__ __forceinline__ void quantize_oct(const float (&v)[8], uint32_t& codes, uint32_t& scale) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, 1));
  scale = e4m3_encode(__fdiv_rn(amax, 6.0f));
  const float d = e4m3_decode(scale);
  codes = 0u;
  if (d != 0.0f) {  // an underflowed block keeps all-zero codes
    const float r = __frcp_rn(d);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      codes |= e2m1x2(quotient_for_e2m1(v[2 * i], d, r), quotient_for_e2m1(v[2 * i + 1], d, r)) << (8 * i);
  }
}

// Eight bf16 values (one 16-byte load) as fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&v)[8]) {
  v[0] = bf16_to_f32(u.x & 0xFFFFu); v[1] = bf16_to_f32(u.x >> 16);
  v[2] = bf16_to_f32(u.y & 0xFFFFu); v[3] = bf16_to_f32(u.y >> 16);
  v[4] = bf16_to_f32(u.z & 0xFFFFu); v[5] = bf16_to_f32(u.z >> 16);
  v[6] = bf16_to_f32(u.w & 0xFFFFu); v[7] = bf16_to_f32(u.w >> 16);
}

// Byte offset of scale (row m, column c) in a region of 128-row atoms with
// Kc scale columns: atoms run along K, then along rows; inside an atom,
// 16 bytes per row of a 32-row slab and 4 bytes per 32-row quarter.
__device__ __forceinline__ uint32_t sf_atom_offset(uint32_t m, uint32_t c, uint32_t Kc) {
  return ((m >> 7) * (Kc >> 2) + (c >> 2)) * 512u + (m & 31u) * 16u + ((m >> 5) & 3u) * 4u + (c & 3u);
}

}  // namespace moe
