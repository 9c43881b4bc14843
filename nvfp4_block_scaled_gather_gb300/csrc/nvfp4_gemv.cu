// W4A16 grouped GEMV: the exact bf16 activations of each group's rows against
// the group's expert's NVFP4 weight, no activation quantization. This is the
// GEMV path of the rocket blog page "The CUTLASS grouped GEMM beats the scalar
// GEMV loop at every M" (section "Proof", its paragraph comparing the two
// paths at M=1): kept there as an explicit override and fallback, and the
// reference for how far the W4A4 path's activation quantization moves the
// result.
//
//   d[r, n] = sum_k a[r, k] * W[e, n, k]      (dequantized weight, no global)
//
// CUDA cores, not the tensor pipe: the block-scaled MMA needs FP4 on both
// operands, and a decode GEMV does two multiply-adds per weight byte. The
// weights are read in the GEMM's tiled format (no second copy): one CTA per
// (group, 128-row weight tile) walks the tile's 18 KB K stages; thread pair
// (2r, 2r+1) owns tile row r, each thread four of the row's eight 16-byte
// pieces per stage. Codes are widened with cvt.rn.f16x2.e2m1x2 (exact), the
// products of 16 values summed in fp32 and scaled once by their e4m3 block
// scale. A row's result depends only on its own activations (fixed K order,
// the two halves added last), so it is the same alone or in any batch.
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ldcg.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kGemvThreads = 256;
constexpr int kRowsPass = 4;          // activation rows staged per pass
constexpr int kStageBytes = 18432;    // one tiled K stage: 16 KB of codes, 2 KB of scale atoms
constexpr int kCodeBytes = 16384;
constexpr int kMaxK = 14336;          // kRowsPass fp32 rows of K in 224 KB of shared memory

// Eight e2m1 codes (element 2j in the low nibble of byte j) -> four f16x2,
// element 2j in the low half.
__device__ __forceinline__ void e2m1x8_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Two e4m3 scale bytes (first in the low byte) -> their values (exact).
__device__ __forceinline__ float2 e4m3x2_f32(uint32_t two_bytes) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)two_bytes));
  return __half22float2(*reinterpret_cast<const __half2*>(&d));
}

// acc[j] += scale * sum_{v < 16} w[v] * x_j[v] for the np rows of the pass.
__device__ __forceinline__ void block16(uint32_t w_lo, uint32_t w_hi, float scale, const float* xs, int K, int np,
                                        float (&acc)[kRowsPass]) {
  uint32_t h[8];
  e2m1x8_f16x2(w_lo, *reinterpret_cast<uint32_t(*)[4]>(h));
  e2m1x8_f16x2(w_hi, *reinterpret_cast<uint32_t(*)[4]>(h + 4));
  float wv[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
    wv[2 * i] = f.x;
    wv[2 * i + 1] = f.y;
  }
#pragma unroll
  for (int j = 0; j < kRowsPass; ++j) {
    if (j < np) {
      const float4* x4 = reinterpret_cast<const float4*>(xs + (size_t)j * K);
      float s = 0.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 x = x4[q];
        s = fmaf(wv[4 * q], x.x, s);
        s = fmaf(wv[4 * q + 1], x.y, s);
        s = fmaf(wv[4 * q + 2], x.z, s);
        s = fmaf(wv[4 * q + 3], x.w, s);
      }
      acc[j] = fmaf(scale, s, acc[j]);
    }
  }
}

__global__ void __launch_bounds__(kGemvThreads) gemv_w4a16_kernel(const uint16_t* __restrict__ a, int src_k,
                                                                  moe_groups_t g, const uint8_t* __restrict__ w_tiled,
                                                                  int interleaved, int N, int K,
                                                                  float* __restrict__ d) {
  pdl_wait();  // the previous kernel in the stream may still be running
  pdl_trigger();
  extern __shared__ float xs[];  // [kRowsPass][K] activations of the pass, fp32
  const int nt = blockIdx.x, gi = blockIdx.y;
  if (gi >= ld_cg(g.counts + 0)) return;
  const int r0 = ld_cg(g.group_offsets + gi), r1 = ld_cg(g.group_offsets + gi + 1);
  const int e = ld_cg(g.group_expert + gi);
  const int nk = (K + 255) / 256, kc4 = K / 64;
  const uint8_t* tile = w_tiled + ((size_t)e * (N / 128) + nt) * nk * kStageBytes;
  const int t = threadIdx.x, tr = t >> 1, hf = t & 1;
  // output column of tile row tr (interleaved w13 tiles: 64 rows of each half)
  const int n = !interleaved ? nt * 128 + tr : (tr < 64 ? nt * 64 + tr : N / 2 + nt * 64 + (tr - 64));
  // this row's scale words: atom a holds scale columns 4a .. 4a+3 at a*512 + (tr%32)*16 + (tr/32)*4
  const uint32_t sf_off = (uint32_t)kCodeBytes + (tr & 31) * 16 + (tr >> 5) * 4;
  for (int p0 = r0; p0 < r1; p0 += kRowsPass) {
    const int np = min(kRowsPass, r1 - p0);
    __syncthreads();  // the previous pass is done with xs
    const int k8 = K / 8;
    for (int i = t; i < np * k8; i += kGemvThreads) {
      const int j = i / k8, c = i - j * k8;
      const int r = p0 + j;
      const int src = src_k > 0 ? ld_cg(g.row_slot + r) / src_k : r;
      const uint4 u = ld_cg(reinterpret_cast<const uint4*>(a + (size_t)src * K) + c);
      float4* dst = reinterpret_cast<float4*>(xs + (size_t)j * K + c * 8);
      dst[0] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
      dst[1] = make_float4(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xFFFF0000u),
                           __uint_as_float(u.w << 16), __uint_as_float(u.w & 0xFFFF0000u));
    }
    __syncthreads();
    float acc[kRowsPass];
#pragma unroll
    for (int j = 0; j < kRowsPass; ++j) acc[j] = 0.0f;
    // this thread's four pieces of a stage and the two scale words they use
    // (atoms 2hf, 2hf+1), the next stage's loaded while this one is summed
    uint4 qn[4];
    uint32_t swn[2];
    auto load_stage = [&](int ks) {
      const uint8_t* st = tile + (size_t)ks * kStageBytes;
      const int pieces = 2 * min(4, kc4 - 4 * ks);  // 16-byte pieces of this stage that hold K values
#pragma unroll
      for (int ci = 0; ci < 4; ++ci) {
        const int c = 4 * hf + ci;  // piece c: K values ks*256 + 32c .. +31, stored at piece c ^ (tr % 8)
        qn[ci] = c < pieces ? __ldg(reinterpret_cast<const uint4*>(st + tr * 128 + ((c ^ (tr & 7)) << 4)))
                            : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int at = 2 * hf + i;
        swn[i] = 2 * at < pieces ? __ldg(reinterpret_cast<const uint32_t*>(st + sf_off + at * 512)) : 0u;
      }
    };
    load_stage(0);
    for (int ks = 0; ks < nk; ++ks) {
      const uint4 q[4] = {qn[0], qn[1], qn[2], qn[3]};
      const uint32_t sw[2] = {swn[0], swn[1]};
      if (ks + 1 < nk) load_stage(ks + 1);
      const int pieces = 2 * min(4, kc4 - 4 * ks);
#pragma unroll
      for (int ci = 0; ci < 4; ++ci) {
        const int c = 4 * hf + ci;
        if (c < pieces) {
          // scale columns 2c and 2c+1: bytes 2(c%2), 2(c%2)+1 of atom c/2's word
          const float2 sc = e4m3x2_f32(sw[ci >> 1] >> (16 * (c & 1)));
          const float* x = xs + ks * 256 + 32 * c;
          block16(q[ci].x, q[ci].y, sc.x, x, K, np, acc);
          block16(q[ci].z, q[ci].w, sc.y, x + 16, K, np, acc);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kRowsPass; ++j) {
      const float other = __shfl_xor_sync(~0u, acc[j], 1);
      const float v = hf == 0 ? acc[j] + other : other + acc[j];  // first half + second half, in both threads
      if (j < np && hf == 0) d[(size_t)(p0 + j) * N + n] = v;
    }
  }
}

}  // namespace

cudaError_t launch_gemv_w4a16(const uint16_t* a, int src_k, int R_max, int E, const moe_groups_t& g,
                              const uint8_t* w_tiled, bool interleaved, int N, int K, float* d, cudaStream_t s) {
  if (N % 128 || K % 64 || K <= 0 || K > kMaxK || (interleaved && N % 256)) return cudaErrorInvalidValue;
  const int smem = kRowsPass * K * (int)sizeof(float);
  // One fixed limit for every launch: lowering it for a smaller K would leave
  // an already captured larger launch (a graph node of the w13 GEMV) above it.
  cudaError_t err = cudaFuncSetAttribute(gemv_w4a16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kRowsPass * kMaxK * (int)sizeof(float));
  if (err != cudaSuccess) return err;
  const int groups = R_max < E ? R_max : E;
  if (groups <= 0) return cudaSuccess;
  return launch_pdl(gemv_w4a16_kernel, dim3(N / 128, groups), dim3(kGemvThreads), smem, s, a, src_k, g, w_tiled,
                    interleaved ? 1 : 0, N, K, d);
}

}  // namespace moe
