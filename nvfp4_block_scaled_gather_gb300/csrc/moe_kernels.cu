// Route-group, gather, NVFP4 quantize, SwiGLU(+requantize), scatter-add and
// the load-time scale swizzle: every step of the MoE layer except the two
// grouped GEMMs (nvfp4_gemm.cu).
//
// Steps as named on the rocket blog page "The CUTLASS grouped GEMM beats the
// scalar GEMV loop at every M" (section "What changed"): moe_gather_rows,
// nvfp4_quantize_rows, swiglu_grouped, moe_scatter_add; grouping by ascending
// expert id; scale layout from section "The seam CUTLASS forced open".
// All of these are HBM- or latency-bound: plain coalesced loads and stores,
// grid-stride loops sized from the SM count, no tensor cores.
#include <climits>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "nvfp4_codec.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int find_group(const int32_t* __restrict__ starts, int G, int key) {
  // largest g in [0, G) with starts[g] <= key; starts strictly ascending from 0
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(starts + mid) <= key) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// a1 route-group: one CTA of 1024 threads. Warp w owns the contiguous slot
// range [s0, s1); per-(warp, expert) counts give every slot its row without
// atomics on the order: row = (rows of lower experts) + (rows of the same
// expert in lower warps) + (rows of the same expert earlier in this warp).
// Rows therefore ascend by (expert, slot), a pure function of the routing.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) route_kernel(const int32_t* __restrict__ ids, int S, int E,
                                                     moe_groups_t g) {
  extern __shared__ int32_t smem[];
  int32_t* wc = smem;                // [32][E]: counts, then running row cursors
  int32_t* rowbase = smem + 32 * E;  // [E]: first row of each expert
  __shared__ int32_t wsum[32][3];
  __shared__ int32_t wmax[32];
  __shared__ int32_t tot[4];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;

  for (int i = tid; i < 32 * E; i += blockDim.x) wc[i] = 0;
  __syncthreads();
  const int per = (S + 31) / 32;
  const int s0 = min(S, w * per), s1 = min(S, s0 + per);
  for (int s = s0 + lane; s < s1; s += 32) {
    const int e = ids[s];
    if (e >= 0 && e < E) atomicAdd(&wc[w * E + e], 1);
  }
  __syncthreads();

  // per expert (one thread each): total and the exclusive prefix over warps
  int cnt = 0;
  if (tid < E) {
    for (int ww = 0; ww < 32; ++ww) {
      const int c = wc[ww * E + tid];
      wc[ww * E + tid] = cnt;
      cnt += c;
    }
  }
  // block-wide exclusive scans of rows, group flags, 128-row scale blocks; max Mg
  const int own0 = cnt, own1 = cnt > 0, own2 = (cnt + 127) >> 7;
  int v0 = own0, v1 = own1, v2 = own2, mx = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a0 = __shfl_up_sync(~0u, v0, o), a1 = __shfl_up_sync(~0u, v1, o),
              a2 = __shfl_up_sync(~0u, v2, o);
    if (lane >= o) { v0 += a0; v1 += a1; v2 += a2; }
    mx = max(mx, __shfl_xor_sync(~0u, mx, o));
  }
  if (lane == 31) { wsum[w][0] = v0; wsum[w][1] = v1; wsum[w][2] = v2; }
  if (lane == 0) wmax[w] = mx;
  __syncthreads();
  if (w == 0) {
    const int t0 = wsum[lane][0], t1 = wsum[lane][1], t2 = wsum[lane][2];
    int i0 = t0, i1 = t1, i2 = t2, m = wmax[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a0 = __shfl_up_sync(~0u, i0, o), a1 = __shfl_up_sync(~0u, i1, o),
                a2 = __shfl_up_sync(~0u, i2, o);
      if (lane >= o) { i0 += a0; i1 += a1; i2 += a2; }
      m = max(m, __shfl_xor_sync(~0u, m, o));
    }
    wsum[lane][0] = i0 - t0; wsum[lane][1] = i1 - t1; wsum[lane][2] = i2 - t2;
    if (lane == 31) { tot[0] = i0; tot[1] = i1; tot[2] = i2; tot[3] = m; }
  }
  __syncthreads();
  if (tid < E) {
    const int row0 = v0 - own0 + wsum[w][0];
    const int gi = v1 - own1 + wsum[w][1];
    const int blk0 = v2 - own2 + wsum[w][2];
    rowbase[tid] = row0;
    if (cnt > 0) {
      g.group_expert[gi] = tid;
      g.group_offsets[gi] = row0;
      g.group_sf_block[gi] = blk0;
    }
  }
  if (tid == 0) {
    g.counts[0] = tot[1];
    g.counts[1] = tot[0];
    g.counts[2] = tot[3];
    g.counts[3] = tot[2];
    g.group_offsets[tot[1]] = tot[0];
    g.group_sf_block[tot[1]] = tot[2];
  }
  __syncthreads();

  // stable placement, each warp walking its own range in order
  for (int c0 = s0; c0 < s1; c0 += 32) {
    const int s = c0 + lane;
    const bool in = s < s1;
    const int e = in ? ids[s] : -1;
    const bool ok = in && e >= 0 && e < E;
    const unsigned peers = __match_any_sync(~0u, ok ? e : -1);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int n = __popc(peers);
    int cur = 0;
    if (ok) {
      cur = wc[w * E + e];
      const int row = rowbase[e] + cur + rank;
      g.row_slot[row] = s;
      g.slot_row[s] = row;
    } else if (in) {
      g.slot_row[s] = -1;
    }
    __syncwarp();
    if (ok && rank == n - 1) wc[w * E + e] = cur + n;
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// a2 gather: xg[r, :] = x[row_slot[r] / k, :], 16 bytes per thread.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) gather_kernel(const uint16_t* __restrict__ x, int H, int k,
                                                          moe_groups_t g, uint16_t* __restrict__ xg) {
  const int R = __ldg(g.counts + 1);
  const int per_row = H / 8;
  const long long total = (long long)R * per_row;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i / per_row), j = (int)(i % per_row);
    const int t = __ldg(g.row_slot + r) / k;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H) + j);
    reinterpret_cast<uint4*>(xg + (size_t)r * H)[j] = v;
  }
}

// Loads 64 bf16 (128 bytes) as fp32.
__device__ __forceinline__ void load64_bf16(const uint16_t* __restrict__ p, float* v) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 u = __ldg(q + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = bf16_to_f32(w[j] & 0xFFFFu);
      v[8 * i + 2 * j + 1] = bf16_to_f32(w[j] >> 16);
    }
  }
}

// Quantizes 64 values (4 blocks): 32 packed bytes and 4 scale bytes.
__device__ __forceinline__ void quantize64_store(const float* v, uint8_t* __restrict__ packed_dst,
                                                 uint32_t* __restrict__ sf_word) {
  uint32_t words[8], scales = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const Nvfp4Block q = quantize16(v + 16 * b);
    words[2 * b] = q.lo;
    words[2 * b + 1] = q.hi;
    scales |= q.scale << (8 * b);
  }
  uint4* dst = reinterpret_cast<uint4*>(packed_dst);
  dst[0] = make_uint4(words[0], words[1], words[2], words[3]);
  dst[1] = make_uint4(words[4], words[5], words[6], words[7]);
  *sf_word = scales;
}

// ---------------------------------------------------------------------------
// a3 / a6 quantize (with optional a2 gather). Work item = (scale row rho of
// the padded per-group region, 64-column chunk j). Real rows are quantized;
// padding rows get zero scale words.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) quantize_kernel(const uint16_t* __restrict__ src, int src_k,
                                                            int K, moe_groups_t g, uint8_t* __restrict__ packed,
                                                            uint8_t* __restrict__ sf) {
  const int G = __ldg(g.counts + 0);
  const int nblk = __ldg(g.counts + 3);
  const int chunks = K / 64, Kc = K / 16;
  const long long total = (long long)nblk * 128 * chunks;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int rho = (int)(i / chunks), j = (int)(i % chunks);
    const int blk = rho >> 7;
    const int gi = find_group(g.group_sf_block, G, blk);
    const int gblk = __ldg(g.group_sf_block + gi);
    const int m = (blk - gblk) * 128 + (rho & 127);
    const int r0 = __ldg(g.group_offsets + gi);
    const int mg = __ldg(g.group_offsets + gi + 1) - r0;
    uint32_t* word = reinterpret_cast<uint32_t*>(sf + (size_t)gblk * 128 * Kc + sf_atom_offset(m, 4 * j, Kc));
    if (m >= mg) { *word = 0u; continue; }
    const int r = r0 + m;
    const int srow = src_k > 0 ? __ldg(g.row_slot + r) / src_k : r;
    float v[64];
    load64_bf16(src + (size_t)srow * K + 64 * j, v);
    quantize64_store(v, packed + (size_t)r * (K / 2) + 32 * j, word);
  }
}

// ---------------------------------------------------------------------------
// a5 (+ a6) SwiGLU with per-group gate/up globals. Same work items as the
// quantizer over an I-wide operand; each item reads 64 gate and 64 up fp32.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) swiglu_kernel(const float* __restrict__ d13, int I, moe_groups_t g,
                                                          const float* __restrict__ g_gate_up,
                                                          uint16_t* __restrict__ h, uint8_t* __restrict__ packed,
                                                          uint8_t* __restrict__ sf) {
  const int G = __ldg(g.counts + 0);
  const int nblk = __ldg(g.counts + 3);
  const int chunks = I / 64, Kc = I / 16;
  const long long total = (long long)nblk * 128 * chunks;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int rho = (int)(i / chunks), j = (int)(i % chunks);
    const int blk = rho >> 7;
    const int gi = find_group(g.group_sf_block, G, blk);
    const int gblk = __ldg(g.group_sf_block + gi);
    const int m = (blk - gblk) * 128 + (rho & 127);
    const int r0 = __ldg(g.group_offsets + gi);
    const int mg = __ldg(g.group_offsets + gi + 1) - r0;
    uint32_t* word = h ? nullptr
                       : reinterpret_cast<uint32_t*>(sf + (size_t)gblk * 128 * Kc + sf_atom_offset(m, 4 * j, Kc));
    if (m >= mg) {
      if (word) *word = 0u;
      continue;
    }
    const int r = r0 + m;
    const int e = __ldg(g.group_expert + gi);
    const float gg = __ldg(g_gate_up + 2 * e), gu = __ldg(g_gate_up + 2 * e + 1);
    const float4* gate = reinterpret_cast<const float4*>(d13 + (size_t)r * 2 * I + 64 * j);
    const float4* up = reinterpret_cast<const float4*>(d13 + (size_t)r * 2 * I + I + 64 * j);
    float v[64];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float4 a = __ldg(gate + q), b = __ldg(up + q);
      const float ga[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int z = 0; z < 4; ++z) {
        const float gt = ga[z] * gg;
        const float u = ub[z] * gu;
        const float hv = gt / (1.0f + expf(-gt)) * u;
        v[4 * q + z] = __uint_as_float(
            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hv))) << 16);  // h rounded once to bf16
      }
    }
    if (h) {
      uint4* dst = reinterpret_cast<uint4*>(h + (size_t)r * I + 64 * j);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t w4[4];
#pragma unroll
        for (int z = 0; z < 4; ++z)
          w4[z] = (__float_as_uint(v[8 * q + 2 * z]) >> 16) | (__float_as_uint(v[8 * q + 2 * z + 1]) & 0xFFFF0000u);
        dst[q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    } else {
      quantize64_store(v, packed + (size_t)r * (I / 2) + 32 * j, word);
    }
  }
}

// ---------------------------------------------------------------------------
// a8 scatter-add: block (token t, 1024-column chunk). Warp 0 orders the
// token's used slots by grouped row (ascending expert), then every thread
// accumulates 4 columns in that order in fp32.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) scatter_kernel(const float* __restrict__ d2, int H,
                                                           const int32_t* __restrict__ ids,
                                                           const float* __restrict__ topk_w, int k, int E,
                                                           moe_groups_t g, const float* __restrict__ g_down,
                                                           uint16_t* __restrict__ y) {
  __shared__ int s_row[kMaxTopK];
  __shared__ float s_coef[kMaxTopK];
  __shared__ int s_n;
  const int t = blockIdx.x;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int row = INT_MAX;
    float coef = 0.0f;
    if (lane < k) {
      const int slot = t * k + lane;
      const int e = __ldg(ids + slot);
      if (e >= 0 && e < E) {
        row = __ldg(g.slot_row + slot);
        coef = __ldg(topk_w + slot) * __ldg(g_down + e);
      }
    }
    int rank = 0;
    for (int i = 0; i < k; ++i) rank += __shfl_sync(~0u, row, i) < row;
    const unsigned valid = __ballot_sync(~0u, row != INT_MAX);
    if (row != INT_MAX) { s_row[rank] = row; s_coef[rank] = coef; }
    if (lane == 0) s_n = __popc(valid);
  }
  __syncthreads();
  const int col = blockIdx.y * (kThreads * 4) + threadIdx.x * 4;
  if (col >= H) return;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  const int n = s_n;
  for (int i = 0; i < n; ++i) {
    const float c = s_coef[i];
    const float4 d = __ldg(reinterpret_cast<const float4*>(d2 + (size_t)s_row[i] * H + col));
    a0 = __fmaf_rn(c, d.x, a0);
    a1 = __fmaf_rn(c, d.y, a1);
    a2 = __fmaf_rn(c, d.z, a2);
    a3 = __fmaf_rn(c, d.w, a3);
  }
  const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a0)) |
                      ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a1)) << 16);
  const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a2)) |
                      ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a3)) << 16);
  *reinterpret_cast<uint2*>(y + (size_t)t * H + col) = make_uint2(lo, hi);
}

// ---------------------------------------------------------------------------
// Load-time swizzle: linear [N, Kc] scale bytes -> 128-row atoms (rows padded
// with zeros). One 4-byte word (4 scale columns of one row) per thread.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) swizzle_kernel(const uint8_t* __restrict__ linear, int N, int Kc,
                                                           uint8_t* __restrict__ out) {
  const int Np = (N + 127) / 128 * 128;
  const int words = Kc / 4;
  const long long total = (long long)Np * words;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i / words), c4 = (int)(i % words);
    const uint32_t v = r < N ? __ldg(reinterpret_cast<const uint32_t*>(linear + (size_t)r * Kc) + c4) : 0u;
    *reinterpret_cast<uint32_t*>(out + sf_atom_offset(r, 4 * c4, Kc)) = v;
  }
}

int grid_for(long long items) {
  const long long need = (items + kThreads - 1) / kThreads;
  const long long cap = (long long)num_sms() * 16;
  return (int)(need < 1 ? 1 : (need < cap ? need : cap));
}

}  // namespace

cudaError_t launch_route(const int32_t* topk_ids, int S, int E, const moe_groups_t& g, cudaStream_t s) {
  const size_t smem = (size_t)33 * E * sizeof(int32_t);
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  route_kernel<<<1, 1024, smem, s>>>(topk_ids, S, E, g);
  return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t* x, int H, int k, int R_max, const moe_groups_t& g, uint16_t* xg,
                          cudaStream_t s) {
  gather_kernel<<<grid_for((long long)R_max * (H / 8)), kThreads, 0, s>>>(x, H, k, g, xg);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const uint16_t* src, int src_k, int R_max, int K, const moe_groups_t& g,
                            uint8_t* packed, uint8_t* sf, cudaStream_t s) {
  const long long items = sf_blocks_bound(R_max, R_max) * 128 * (K / 64);
  quantize_kernel<<<grid_for(items), kThreads, 0, s>>>(src, src_k, K, g, packed, sf);
  return cudaGetLastError();
}

cudaError_t launch_swiglu(const float* d13, int R_max, int I, const moe_groups_t& g, const float* g_gate_up,
                          uint16_t* h, uint8_t* packed, uint8_t* sf, cudaStream_t s) {
  const long long items = sf_blocks_bound(R_max, R_max) * 128 * (I / 64);
  swiglu_kernel<<<grid_for(items), kThreads, 0, s>>>(d13, I, g, g_gate_up, h, packed, sf);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const float* d2, int H, const int32_t* topk_ids, const float* topk_w, int T, int k,
                           int E, const moe_groups_t& g, const float* g_down, uint16_t* y, cudaStream_t s) {
  dim3 grid(T, (H + kThreads * 4 - 1) / (kThreads * 4));
  scatter_kernel<<<grid, kThreads, 0, s>>>(d2, H, topk_ids, topk_w, k, E, g, g_down, y);
  return cudaGetLastError();
}

cudaError_t launch_swizzle(const uint8_t* linear, int N, int K, uint8_t* swizzled, cudaStream_t s) {
  const long long items = (long long)((N + 127) / 128 * 128) * (K / 64);
  swizzle_kernel<<<grid_for(items), kThreads, 0, s>>>(linear, N, K / 16, swizzled);
  return cudaGetLastError();
}

}  // namespace moe
