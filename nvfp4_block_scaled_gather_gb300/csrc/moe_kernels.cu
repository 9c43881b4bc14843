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
#include "ldcg.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------------------
// a1 route-group: one CTA of 1024 threads. Warp w owns the contiguous slot
// range [s0, s1); per-(warp, expert) counts give every slot its row without
// atomics on the order: row = (rows of lower experts) + (rows of the same
// expert in lower warps) + (rows of the same expert earlier in this warp).
// Rows therefore ascend by (expert, slot), a pure function of the routing.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) route_kernel(const int32_t* __restrict__ ids, int S, int E,
                                                     moe_groups_t g, int* __restrict__ zero, int nzero,
                                                     int* __restrict__ slot_sf, int bt) {
  pdl_wait();  // the previous kernel in the stream may still be running
  pdl_trigger();
  for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
  extern __shared__ int32_t smem[];
  int32_t* wc = smem;                // [32][E]: counts, then running row cursors
  int32_t* rowbase = smem + 32 * E;  // [E]: first row of each expert
  int32_t* blkbase = smem + 33 * E;  // [E]: its first token block of bt rows (slot_sf only)
  __shared__ int32_t wsum[32][4];
  __shared__ int32_t wmax[32];
  __shared__ int32_t tot[5];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;

  for (int i = tid; i < 32 * E; i += blockDim.x) wc[i] = 0;
  __syncthreads();
  const int per = (S + 31) / 32;
  const int s0 = min(S, w * per), s1 = min(S, s0 + per);
  for (int s = s0 + lane; s < s1; s += 32) {
    const int e = ld_cg(ids + s);
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
  // block-wide exclusive scans of rows, group flags, 128-row scale blocks and
  // 32-row GEMM chunks; max Mg
  const int own0 = cnt, own1 = cnt > 0, own2 = (cnt + 127) >> 7, own3 = (cnt + 31) >> 5;
  int v0 = own0, v1 = own1, v2 = own2, v3 = own3, mx = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a0 = __shfl_up_sync(~0u, v0, o), a1 = __shfl_up_sync(~0u, v1, o),
              a2 = __shfl_up_sync(~0u, v2, o), a3 = __shfl_up_sync(~0u, v3, o);
    if (lane >= o) { v0 += a0; v1 += a1; v2 += a2; v3 += a3; }
    mx = max(mx, __shfl_xor_sync(~0u, mx, o));
  }
  if (lane == 31) { wsum[w][0] = v0; wsum[w][1] = v1; wsum[w][2] = v2; wsum[w][3] = v3; }
  if (lane == 0) wmax[w] = mx;
  __syncthreads();
  if (w == 0) {
    const int t0 = wsum[lane][0], t1 = wsum[lane][1], t2 = wsum[lane][2], t3 = wsum[lane][3];
    int i0 = t0, i1 = t1, i2 = t2, i3 = t3, m = wmax[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a0 = __shfl_up_sync(~0u, i0, o), a1 = __shfl_up_sync(~0u, i1, o),
                a2 = __shfl_up_sync(~0u, i2, o), a3 = __shfl_up_sync(~0u, i3, o);
      if (lane >= o) { i0 += a0; i1 += a1; i2 += a2; i3 += a3; }
      m = max(m, __shfl_xor_sync(~0u, m, o));
    }
    wsum[lane][0] = i0 - t0; wsum[lane][1] = i1 - t1; wsum[lane][2] = i2 - t2; wsum[lane][3] = i3 - t3;
    if (lane == 31) { tot[0] = i0; tot[1] = i1; tot[2] = i2; tot[3] = m; tot[4] = i3; }
  }
  __syncthreads();
  if (tid < E) {
    const int row0 = v0 - own0 + wsum[w][0];
    const int gi = v1 - own1 + wsum[w][1];
    const int blk0 = v2 - own2 + wsum[w][2];
    const int chk0 = v3 - own3 + wsum[w][3];
    rowbase[tid] = row0;
    if (slot_sf) blkbase[tid] = bt == 128 ? blk0 : chk0;
    if (cnt > 0) {
      g.group_expert[gi] = tid;
      g.group_offsets[gi] = row0;
      g.group_sf_block[gi] = blk0;
      g.group_chunk[gi] = chk0;
      for (int q = 0; q < own3; ++q)  // the group's 32-row chunks
        reinterpret_cast<int4*>(g.chunk_info)[chk0 + q] = make_int4(row0 + 32 * q, min(32, cnt - 32 * q), tid, gi);
      for (int q = 0; q < own2; ++q)  // and its 128-row blocks
        reinterpret_cast<int4*>(g.block_info)[blk0 + q] = make_int4(row0 + 128 * q, min(128, cnt - 128 * q), tid, gi);
    }
  }
  if (tid == 0) {
    g.counts[0] = tot[1];
    g.counts[1] = tot[0];
    g.counts[2] = tot[3];
    g.counts[3] = tot[2];
    g.counts[4] = tot[4];
    g.group_offsets[tot[1]] = tot[0];
    g.group_sf_block[tot[1]] = tot[2];
    g.group_chunk[tot[1]] = tot[4];
  }
  __syncthreads();

  // stable placement, each warp walking its own range in order
  for (int c0 = s0; c0 < s1; c0 += 32) {
    const int s = c0 + lane;
    const bool in = s < s1;
    const int e = in ? ld_cg(ids + s) : -1;
    const bool ok = in && e >= 0 && e < E;
    const unsigned peers = __match_any_sync(~0u, ok ? e : -1);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int n = __popc(peers);
    int cur = 0;
    if (ok) {
      cur = wc[w * E + e];
      const int local = cur + rank;  // the row's place in its expert's group
      const int row = rowbase[e] + local;
      g.row_slot[row] = s;
      g.slot_row[s] = row;
      if (slot_sf) slot_sf[s] = ((blkbase[e] + local / bt) << 7) | (local % bt);
    } else if (in) {
      g.slot_row[s] = -1;
      if (slot_sf) slot_sf[s] = -1;
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
  pdl_wait();  // the previous kernel in the stream may still be running
  pdl_trigger();
  const int R = ld_cg(g.counts + 1);
  const int per_row = H / 8;
  const long long total = (long long)R * per_row;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i / per_row), j = (int)(i % per_row);
    const int t = ld_cg(g.row_slot + r) / k;
    const uint4 v = ld_cg(reinterpret_cast<const uint4*>(x + (size_t)t * H) + j);
    reinterpret_cast<uint4*>(xg + (size_t)r * H)[j] = v;
  }
}

// Four lanes (4j .. 4j+3 of a warp) hold one 16-value block, four values
// each; sixteen lanes hold the four blocks of one 4-byte scale word. Each lane
// writes its two packed bytes; the first lane of each 16 writes the word.
// Lanes that are not `active` compute along (shuffles need the full warp) but
// write nothing; a 16-lane group is either wholly active or wholly not.
__device__ __forceinline__ void quantize_quad_store(const float (&v)[4], bool active, int lane,
                                                    uint8_t* __restrict__ packed_dst, uint32_t* __restrict__ word) {
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, 2));
  const uint32_t s = block_scale_code(amax);
  uint32_t codes = 0u;
  if (s != 0u) {  // an underflowed block keeps all-zero codes
    const float d = e4m3_value(s), r = rcp_approx(d);
    codes = e2m1x2(block_quotient(v[0], d, r), block_quotient(v[1], d, r)) |
            (e2m1x2(block_quotient(v[2], d, r), block_quotient(v[3], d, r)) << 8);
  }
  const uint32_t s1 = __shfl_down_sync(~0u, s, 4), s2 = __shfl_down_sync(~0u, s, 8),
                 s3 = __shfl_down_sync(~0u, s, 12);
  if (!active) return;
  *reinterpret_cast<uint16_t*>(packed_dst) = (uint16_t)codes;
  if ((lane & 15) == 0) *word = s | (s1 << 8) | (s2 << 16) | (s3 << 24);
}

// Token-scale layouts (include/moe_nvfp4.h): per group 128-row atoms, or per
// 32-row GEMM chunk one 512-byte atom per 64 K values whose 16-byte row i
// holds chunk row i's four scales in its first word (other words zero).
constexpr int kRowsAtom = 128;

struct ScaleTarget {
  uint8_t* base;  // the CTA's row block region
  int layout, Kc;
  // scale byte of column c of row m of the block
  __device__ __forceinline__ uint8_t* byte(int m, int c) const {
    return base + (layout == MOE_SF_ATOM128 ? sf_atom_offset(m, c, Kc)
                                            : (uint32_t)(c >> 2) * 512u + m * 16u + (uint32_t)(c & 3));
  }
  // word holding scale columns c..c+3 (c % 4 == 0) of row m of the block
  __device__ __forceinline__ uint32_t* word(int m, int c) const { return reinterpret_cast<uint32_t*>(byte(m, c)); }
  // zero every word of atoms [a0, a0 + na) that no real row (< nvalid) fills
  __device__ __forceinline__ void zero_rest(int a0, int na, int nvalid) const {
    uint32_t* words = reinterpret_cast<uint32_t*>(base + (size_t)a0 * 512);
    for (int w = threadIdx.x; w < na * 128; w += blockDim.x) {
      const int wi = w & 127;
      const bool real = layout == MOE_SF_ATOM128 ? (wi >> 2) + 32 * (wi & 3) < nvalid  // row (wi/4) + 32*(wi%4)
                                                 : ((wi & 3) == 0 && (wi >> 2) < nvalid);
      if (!real) words[w] = 0u;
    }
  }
};

// The CTA's row block `blk` (128 rows per block in the atom layout, 32 in the
// chunk layout): first grouped row, valid rows and expert.
struct RowBlock {
  int row0, nvalid, expert;
};

__device__ __forceinline__ const int4* block_table(const moe_groups_t& g, int layout) {
  return reinterpret_cast<const int4*>(layout == MOE_SF_CHUNK32 ? g.chunk_info : g.block_info);
}

// One table read, the same value in every thread.
__device__ __forceinline__ RowBlock resolve_block(const moe_groups_t& g, int layout, int blk) {
  const int4 c = ld_cg(block_table(g, layout) + blk);
  return RowBlock{c.x, c.y, c.z};
}

__device__ __forceinline__ int routed_blocks(const moe_groups_t& g, int layout) {
  return ld_cg(g.counts + (layout == MOE_SF_ATOM128 ? 3 : 4));
}

constexpr int kColsPerCta = 1024;  // K values per CTA (grid.y covers K) for the SwiGLU and small-batch kernels
static_assert(kColsPerCta == 4 * kThreads, "the small-batch kernel gives each thread 4 values of a chunk");
constexpr int kQuantCols = 512;    // K values per CTA of the quantizer: one row per warp pass

// ---------------------------------------------------------------------------
// a3 / a6 quantize (with optional a2 gather). Grid: (row block, 512-value
// column chunk); CTAs past the routed block count exit. Lane l of a warp
// quantizes 16-value block l of a row from two 16-byte loads and writes its
// 8 code bytes and its scale byte (four lanes fill a scale word); the eight
// warps take rows w, w + 8, ..., two rows in flight. Scale words no real row
// fills are zeroed.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) quantize_kernel(const uint16_t* __restrict__ src, int src_k, int K,
                                                            moe_groups_t g, int layout, uint8_t* __restrict__ packed,
                                                            uint8_t* __restrict__ sf) {
  pdl_wait();  // the previous kernel in the stream may still be running
  pdl_trigger();
  const int blk = blockIdx.x;
  // the block count and this block's table entry in flight together (the
  // entry is in bounds whether or not the block is routed)
  const int4 c = ld_cg(block_table(g, layout) + blk);
  if (blk >= routed_blocks(g, layout)) return;
  const RowBlock rb{c.x, c.y, c.z};
  const int Kc = K / 16;
  const int kc0 = blockIdx.y * kQuantCols;
  const int kcount = min(kQuantCols, K - kc0);  // a multiple of 64
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool lane_on = 16 * lane < kcount;       // every lane but in a short last chunk
  const ScaleTarget st{sf + (size_t)blk * 128 * Kc, layout, Kc};  // either layout: 128*Kc bytes per block
  // source row of each of the block's rows, read once
  __shared__ int s_src[kRowsAtom];
  if ((int)threadIdx.x < rb.nvalid) {
    const int r = rb.row0 + threadIdx.x;
    s_src[threadIdx.x] = src_k > 0 ? ld_cg(g.row_slot + r) / src_k : r;
  }
  __syncthreads();
  constexpr int kWarps = kThreads / 32;
  constexpr int kBatch = 2;  // rows in flight per warp
  for (int m0 = warp; m0 < rb.nvalid; m0 += kBatch * kWarps) {
    uint4 u[kBatch][2];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int m = m0 + j * kWarps;
      u[j][0] = u[j][1] = make_uint4(0u, 0u, 0u, 0u);
      if (m < rb.nvalid && lane_on) {
        const uint4* p = reinterpret_cast<const uint4*>(src + (size_t)s_src[m] * K + kc0 + 16 * lane);
        u[j][0] = ld_cg(p);
        u[j][1] = ld_cg(p + 1);
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int m = m0 + j * kWarps;  // the same for the whole warp
      if (m >= rb.nvalid) break;
      const uint32_t w[8] = {u[j][0].x, u[j][0].y, u[j][0].z, u[j][0].w, u[j][1].x, u[j][1].y, u[j][1].z, u[j][1].w};
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
      uint2 codes;
      uint32_t scale;
      quantize_block16(v, codes, scale);
      if (lane_on) {
        *reinterpret_cast<uint2*>(packed + (size_t)(rb.row0 + m) * (K / 2) + kc0 / 2 + 8 * lane) = codes;
        *st.byte(m, kc0 / 16 + lane) = (uint8_t)scale;
      }
    }
  }
  st.zero_rest(kc0 / 64, kcount / 64, rb.nvalid);
}

// ---------------------------------------------------------------------------
// a2 + a3 token by token (the layer's path for more than 32 slots): each
// token row of x is read and quantized once, and its codes and block scales
// are written to every routed row of the token (slot_row) and the row's
// place in the token-scale layout (slot_sf); the same bytes as
// quantize_kernel for every routed row. Scale words of rows past a block's
// valid rows are not written: they feed only accumulator columns no result
// reads. Grid: (8 tokens, 512-value column chunk); warp w takes token
// 8 blockIdx.x + w, lane l its 16-value block l.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) quantize_tokens_kernel(const uint16_t* __restrict__ x, int T, int K,
                                                                   int k, moe_groups_t g,
                                                                   const int* __restrict__ slot_sf, int layout,
                                                                   uint8_t* __restrict__ packed,
                                                                   uint8_t* __restrict__ sf) {
  pdl_wait();  // the tables come from the previous kernel
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (t >= T) return;
  const int Kc = K / 16;
  const int kc0 = blockIdx.y * kQuantCols;
  const int kcount = min(kQuantCols, K - kc0);  // a multiple of 64
  const bool lane_on = 16 * lane < kcount;
  // the token's routed rows and scale places, lane j holding slot j's, in flight with the row
  const int row = lane < k ? ld_cg(g.slot_row + (size_t)t * k + lane) : -1;
  const int pos = lane < k ? ld_cg(slot_sf + (size_t)t * k + lane) : -1;
  uint4 u0 = make_uint4(0u, 0u, 0u, 0u), u1 = u0;
  if (lane_on) {
    const uint4* p = reinterpret_cast<const uint4*>(x + (size_t)t * K + kc0 + 16 * lane);
    u0 = ld_cg(p);
    u1 = ld_cg(p + 1);
  }
  const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
  float v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  uint2 codes;
  uint32_t scale;
  quantize_block16(v, codes, scale);
  for (int j = 0; j < k; ++j) {
    const int r = __shfl_sync(~0u, row, j), q = __shfl_sync(~0u, pos, j);
    if (r < 0 || !lane_on) continue;  // an unused slot (the same in every lane)
    *reinterpret_cast<uint2*>(packed + (size_t)r * (K / 2) + kc0 / 2 + 8 * lane) = codes;
    const ScaleTarget st{sf + (size_t)(q >> 7) * 128 * Kc, layout, Kc};
    *st.byte(q & 127, kc0 / 16 + lane) = (uint8_t)scale;
  }
}

// ---------------------------------------------------------------------------
// a1 + a2 + a3 for small batches (T*k <= 32 slots), one launch. Grid: (slot,
// 1024-value column chunk). Warp 0 of every CTA routes the <= 32 slots (one
// per lane): the same rows, groups and tables as route_kernel (rows ascend by
// (expert, slot); with at most 32 rows no group has more than one 32-row chunk
// or 128-row scale block); CTA (0, 0) writes the tables. CTA (s, c) loads
// column chunk c of slot s's token row while warp 0 routes, then quantizes it
// into slot s's routed row in the 32-row-chunk token layout, exactly as
// quantize_kernel does; the CTAs of unused slots exit.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) route_quantize_small_kernel(const int32_t* __restrict__ ids, int S, int E,
                                                                        moe_groups_t g, int* __restrict__ zero,
                                                                        int nzero, const uint16_t* __restrict__ x,
                                                                        int k, int K, uint8_t* __restrict__ packed,
                                                                        uint8_t* __restrict__ sf) {
  pdl_wait();  // the previous kernel in the stream may still be running
  const bool lead = blockIdx.x == 0 && blockIdx.y == 0;
  if (lead) {
    // The next kernel (the GEMM launch) claims work from these counters as
    // soon as it starts, before it waits for this kernel: they are cleared,
    // and the stores performed GPU-wide, before this CTA lets it launch.
    for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
    __threadfence();
    __syncthreads();
  }
  pdl_trigger();
  // This CTA quantizes slot blockIdx.x's row (token blockIdx.x / k): its
  // values are loaded here, in flight while warp 0 routes.
  const int kc0 = blockIdx.y * kColsPerCta;
  const int kcount = min(kColsPerCta, K - kc0);
  const int q = threadIdx.x;  // this thread's 4 values (kColsPerCta = 4 * kThreads)
  const bool q_on = q < kcount / 4 && (int)blockIdx.x < S;
  uint2 xv = make_uint2(0u, 0u);
  if (q_on) xv = ld_cg(reinterpret_cast<const uint2*>(x + (size_t)(blockIdx.x / k) * K + kc0 + 4 * q));
  __shared__ int s_chunk[32], s_m[32], s_cnt[32], s_row[32];
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const bool in = lane < S;
    const int e = in ? ld_cg(ids + lane) : -1;
    const bool ok = in && e >= 0 && e < E;
    const int key = ok ? e : 0x7fffffff;
    const unsigned peers = __match_any_sync(~0u, key);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int n = __popc(peers);
    const unsigned leaders = __ballot_sync(~0u, ok && rank == 0);
    const int R = __popc(__ballot_sync(~0u, ok)), G = __popc(leaders);
    int less = 0, gless = 0;  // rows and groups of lower experts
    for (int j = 0; j < 32; ++j) {
      const int kj = __shfl_sync(~0u, key, j);
      if (kj < key) {
        ++less;
        gless += (leaders >> j) & 1u;
      }
    }
    int mx = ok ? n : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) mx = max(mx, __shfl_xor_sync(~0u, mx, o));
    s_row[lane] = ok ? less + rank : -1;
    if (ok) {
      const int row = less + rank;
      s_chunk[row] = gless;
      s_m[row] = rank;
      if (rank == 0) s_cnt[gless] = n;
      if (lead) {
        g.row_slot[row] = lane;
        g.slot_row[lane] = row;
        if (rank == 0) {
          g.group_expert[gless] = e;
          g.group_offsets[gless] = less;
          g.group_sf_block[gless] = gless;
          g.group_chunk[gless] = gless;
          reinterpret_cast<int4*>(g.chunk_info)[gless] = make_int4(less, n, e, gless);
          reinterpret_cast<int4*>(g.block_info)[gless] = make_int4(less, n, e, gless);
        }
      }
    } else if (in && lead) {
      g.slot_row[lane] = -1;
    }
    if (lane == 0) {
      if (lead) {
        g.counts[0] = G;
        g.counts[1] = R;
        g.counts[2] = mx;
        g.counts[3] = G;
        g.counts[4] = G;
        g.group_offsets[G] = R;
        g.group_sf_block[G] = G;
        g.group_chunk[G] = G;
      }
    }
  }
  __syncthreads();
  if ((int)blockIdx.x >= S) return;
  const int r = s_row[blockIdx.x];  // the slot's routed row
  if (r < 0) return;                // an unused slot has none
  const int Kc = K / 16;
  const int c = s_chunk[r], m = s_m[r];
  const ScaleTarget st{sf + (size_t)c * 128 * Kc, MOE_SF_CHUNK32, Kc};
  const int lane = threadIdx.x & 31;
  if ((threadIdx.x & ~31) < kcount / 4) {  // warps with values (whole warps: kcount % 64 == 0)
    const float v[4] = {bf16_to_f32(xv.x & 0xFFFFu), bf16_to_f32(xv.x >> 16), bf16_to_f32(xv.y & 0xFFFFu),
                        bf16_to_f32(xv.y >> 16)};
    quantize_quad_store(v, q_on, lane, packed + (size_t)r * (K / 2) + (kc0 + 4 * q) / 2,
                        st.word(m, (kc0 + 4 * q) / 16));
  }
  // the chunk's first row also zeroes the words no row fills in these atoms
  if (m == 0) st.zero_rest(kc0 / 64, kcount / 64, s_cnt[c]);
}

// ---------------------------------------------------------------------------
// a5 (+ a6) SwiGLU with per-group gate/up globals; same grid as the quantizer
// over the I-wide output. Each lane reads 4 gate and 4 up fp32 values.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) swiglu_kernel(const float* __restrict__ d13, int I, moe_groups_t g,
                                                          int layout, const float* __restrict__ g_gate_up,
                                                          uint16_t* __restrict__ h, uint8_t* __restrict__ packed,
                                                          uint8_t* __restrict__ sf) {
  pdl_wait();  // the previous kernel in the stream may still be running
  pdl_trigger();
  const int blk = blockIdx.x;
  if (blk >= routed_blocks(g, layout)) return;
  const RowBlock rb = resolve_block(g, layout, blk);
  const int e = rb.expert;
  const float gg = ld_cg(g_gate_up + 2 * e), gu = ld_cg(g_gate_up + 2 * e + 1);
  const int Kc = I / 16;
  const int kc0 = blockIdx.y * kColsPerCta;
  const int kcount = min(kColsPerCta, I - kc0);
  const int quads = kcount / 4;
  const int total = rb.nvalid * quads;
  const int lane = threadIdx.x & 31;
  const ScaleTarget st{h ? nullptr : sf + (size_t)blk * 128 * Kc, layout, Kc};
  for (int base = (threadIdx.x & ~31); base < total; base += blockDim.x) {
    const int item = base + lane;
    const bool active = item < total;
    const int m = active ? item / quads : 0;
    const int q = active ? item - m * quads : 0;
    const int r = rb.row0 + m;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (active) {
      const float* src = d13 + (size_t)r * 2 * I + kc0 + 4 * q;
      const float4 a = ld_cg(reinterpret_cast<const float4*>(src));
      const float4 b = ld_cg(reinterpret_cast<const float4*>(src + I));
      const float ga[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int z = 0; z < 4; ++z) {
        const float gt = ga[z] * gg;
        const float u = ub[z] * gu;
        const float hv = gt / (1.0f + expf(-gt)) * u;
        v[z] = bf16_to_f32(__bfloat16_as_ushort(__float2bfloat16_rn(hv)));  // h rounded once to bf16
      }
    }
    if (h) {
      if (active) {
        const uint32_t lo = (__float_as_uint(v[0]) >> 16) | (__float_as_uint(v[1]) & 0xFFFF0000u);
        const uint32_t hi = (__float_as_uint(v[2]) >> 16) | (__float_as_uint(v[3]) & 0xFFFF0000u);
        *reinterpret_cast<uint2*>(h + (size_t)r * I + kc0 + 4 * q) = make_uint2(lo, hi);
      }
    } else {
      quantize_quad_store(v, active, lane, packed + (size_t)r * (I / 2) + (kc0 + 4 * q) / 2,
                          st.word(m, (kc0 + 4 * q) / 16));
    }
  }
  if (!h) st.zero_rest(kc0 / 64, kcount / 64, rb.nvalid);
}

// ---------------------------------------------------------------------------
// a8 scatter-add: block (token t, 1024-column chunk). Warp 0 orders the
// token's used slots by grouped row (ascending expert), then every thread
// accumulates 4 columns in that order in fp32, the loads of up to 8 slots
// in flight together.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) scatter_kernel(const float* __restrict__ d2, int H,
                                                           const int32_t* __restrict__ ids,
                                                           const float* __restrict__ topk_w, int k, int E,
                                                           moe_groups_t g, const float* __restrict__ g_down,
                                                           uint16_t* __restrict__ y, int tables_early) {
  // The previous kernel in the stream may still be running. With
  // tables_early the routing tables are two or more launches old (complete):
  // only the reads of d2 wait for it.
  if (!tables_early) {
    pdl_wait();
    pdl_trigger();
  }
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
      const int e = ld_cg(ids + slot);
      if (e >= 0 && e < E) {
        row = ld_cg(g.slot_row + slot);
        coef = ld_cg(topk_w + slot) * ld_cg(g_down + e);
      }
    }
    int rank = 0;
    for (int i = 0; i < k; ++i) rank += __shfl_sync(~0u, row, i) < row;
    const unsigned valid = __ballot_sync(~0u, row != INT_MAX);
    if (row != INT_MAX) { s_row[rank] = row; s_coef[rank] = coef; }
    if (lane == 0) s_n = __popc(valid);
  }
  __syncthreads();
  if (tables_early) {
    pdl_wait();
    pdl_trigger();
  }
  const int col = blockIdx.y * (kThreads * 4) + threadIdx.x * 4;
  if (col >= H) return;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  const int n = s_n;
  for (int i0 = 0; i0 < n; i0 += 8) {
    // up to 8 slots' loads in flight, then the sums in slot order
    float4 d[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      d[j] = i0 + j < n ? ld_cg(reinterpret_cast<const float4*>(d2 + (size_t)s_row[i0 + j] * H + col))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (i0 + j >= n) break;
      const float c = s_coef[i0 + j];
      a0 = __fmaf_rn(c, d[j].x, a0);
      a1 = __fmaf_rn(c, d[j].y, a1);
      a2 = __fmaf_rn(c, d[j].z, a2);
      a3 = __fmaf_rn(c, d[j].w, a3);
    }
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
  pdl_wait();  // the previous kernel in the stream may still be running
  pdl_trigger();
  const int Np = (N + 127) / 128 * 128;
  const int words = Kc / 4;
  const long long total = (long long)Np * words;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i / words), c4 = (int)(i % words);
    const uint32_t v = r < N ? ld_cg(reinterpret_cast<const uint32_t*>(linear + (size_t)r * Kc) + c4) : 0u;
    *reinterpret_cast<uint32_t*>(out + sf_atom_offset(r, 4 * c4, Kc)) = v;
  }
}

// ---------------------------------------------------------------------------
// Load-time tiling of weights for the grouped GEMM: for every 128-row tile t
// and 256-value K stage ks, an 18 KB block = 16 KB of e2m1 bytes in the
// 128-byte-swizzled shared-memory image (16-byte chunk c of row r stored at
// chunk c ^ (r % 8)) followed by the stage's four 512-byte scale atoms.
// Values past K are zero. With il > 0 (rows per expert), tile row j of an
// expert's tile tt comes from row 64*tt + j (j < 64) or il/2 + 64*tt + j - 64.
// ---------------------------------------------------------------------------
__device__ __forceinline__ long long tile_src_row(int t, int j, int il) {
  if (il <= 0) return (long long)t * 128 + j;
  const int per = il / 128;  // tiles per expert
  const long long e = t / per, tt = t - e * per;
  return e * il + (j < 64 ? 64 * tt + j : il / 2 + 64 * tt + (j - 64));
}

__global__ void __launch_bounds__(kThreads) tile_kernel(const uint8_t* __restrict__ packed,
                                                        const uint8_t* __restrict__ sf_linear, int tiles, int K,
                                                        int il, uint8_t* __restrict__ out) {
  pdl_wait();  // the previous kernel in the stream may still be running
  pdl_trigger();
  const int nk = (K + 255) / 256, rowb = K / 2, Kc = K / 16;
  const long long chunks = (long long)tiles * nk * 128 * 8;
  const long long words = (long long)tiles * nk * 4 * 128;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < chunks + words;
       i += (long long)gridDim.x * blockDim.x) {
    if (i < chunks) {
      const int c = (int)(i & 7), r = (int)((i >> 3) & 127);
      const long long ts = i >> 10;  // t * nk + ks
      const int ks = (int)(ts % nk), t = (int)(ts / nk);
      const int col = ks * 128 + c * 16;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (col < rowb) v = ld_cg(reinterpret_cast<const uint4*>(packed + (size_t)tile_src_row(t, r, il) * rowb + col));
      *reinterpret_cast<uint4*>(out + (size_t)ts * 18432 + r * 128 + ((c ^ (r & 7)) << 4)) = v;
    } else {
      const long long j = i - chunks;
      const int wi = (int)(j & 127), a = (int)((j >> 7) & 3);
      const long long ts = j >> 9;
      const int ks = (int)(ts % nk), t = (int)(ts / nk);
      const int m = (wi >> 2) + 32 * (wi & 3);
      const int col = (4 * ks + a) * 4;  // first scale column of this atom
      uint32_t v = 0u;
      if (col < Kc) v = ld_cg(reinterpret_cast<const uint32_t*>(sf_linear + (size_t)tile_src_row(t, m, il) * Kc + col));
      *reinterpret_cast<uint32_t*>(out + (size_t)ts * 18432 + 16384 + a * 512 + wi * 4) = v;
    }
  }
}

int grid_for(long long items) {
  const long long need = (items + kThreads - 1) / kThreads;
  const long long cap = (long long)num_sms() * 16;
  return (int)(need < 1 ? 1 : (need < cap ? need : cap));
}

}  // namespace

cudaError_t launch_route(const int32_t* topk_ids, int S, int E, const moe_groups_t& g, cudaStream_t s, int* zero,
                         int nzero, int* slot_sf, int bt) {
  if (slot_sf && bt != 32 && bt != 128) return cudaErrorInvalidValue;
  const size_t smem = (size_t)34 * E * sizeof(int32_t);
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  return launch_pdl(route_kernel, dim3(1), dim3(1024), smem, s, topk_ids, S, E, g, zero, zero ? nzero : 0, slot_sf,
                    bt > 0 ? bt : 32);
}

cudaError_t launch_gather(const uint16_t* x, int H, int k, int R_max, const moe_groups_t& g, uint16_t* xg,
                          cudaStream_t s) {
  return launch_pdl(gather_kernel, dim3(grid_for((long long)R_max * (H / 8))), dim3(kThreads), 0, s, x, H, k, g, xg);
}

cudaError_t launch_quantize(const uint16_t* src, int src_k, int R_max, int E, int K, const moe_groups_t& g,
                            int layout, uint8_t* packed, uint8_t* sf, cudaStream_t s) {
  const dim3 grid((unsigned)row_blocks_bound(R_max, E, layout), (K + kQuantCols - 1) / kQuantCols);
  return launch_pdl(quantize_kernel, grid, dim3(kThreads), 0, s, src, src_k, K, g, layout, packed, sf);
}

cudaError_t launch_quantize_tokens(const uint16_t* x, int T, int K, int k, const moe_groups_t& g,
                                   const int* slot_sf, int layout, uint8_t* packed, uint8_t* sf, cudaStream_t s) {
  if (K % 64 || k < 1 || k > kMaxTopK || (layout != MOE_SF_ATOM128 && layout != MOE_SF_CHUNK32))
    return cudaErrorInvalidValue;
  const dim3 grid((unsigned)((T + kThreads / 32 - 1) / (kThreads / 32)), (K + kQuantCols - 1) / kQuantCols);
  return launch_pdl(quantize_tokens_kernel, grid, dim3(kThreads), 0, s, x, T, K, k, g, slot_sf, layout, packed, sf);
}

cudaError_t launch_route_quantize_small(const int32_t* topk_ids, int S, int E, const moe_groups_t& g, int* zero,
                                        int nzero, const uint16_t* x, int k, int K, uint8_t* packed, uint8_t* sf,
                                        cudaStream_t s) {
  if (S > 32 || k <= 0 || K % 64) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)S, (K + kColsPerCta - 1) / kColsPerCta);
  return launch_pdl(route_quantize_small_kernel, grid, dim3(kThreads), 0, s, topk_ids, S, E, g, zero,
                    zero ? nzero : 0, x, k, K, packed, sf);
}

cudaError_t launch_swiglu(const float* d13, int R_max, int E, int I, const moe_groups_t& g, int layout,
                          const float* g_gate_up, uint16_t* h, uint8_t* packed, uint8_t* sf, cudaStream_t s) {
  const dim3 grid((unsigned)row_blocks_bound(R_max, E, layout), (I + kColsPerCta - 1) / kColsPerCta);
  return launch_pdl(swiglu_kernel, grid, dim3(kThreads), 0, s, d13, I, g, layout, g_gate_up, h, packed, sf);
}

cudaError_t launch_tile(const uint8_t* packed, const uint8_t* sf_linear, int rows, int K, int interleave_rows,
                        uint8_t* tiled, cudaStream_t s) {
  const long long tiles = rows / 128, nk = (K + 255) / 256;
  const long long items = tiles * nk * (128 * 8 + 4 * 128);
  return launch_pdl(tile_kernel, dim3(grid_for(items)), dim3(kThreads), 0, s, packed, sf_linear, (int)tiles, K,
                    interleave_rows, tiled);
}

cudaError_t launch_scatter(const float* d2, int H, const int32_t* topk_ids, const float* topk_w, int T, int k,
                           int E, const moe_groups_t& g, const float* g_down, uint16_t* y, cudaStream_t s,
                           bool tables_early) {
  dim3 grid(T, (H + kThreads * 4 - 1) / (kThreads * 4));
  return launch_pdl(scatter_kernel, grid, dim3(kThreads), 0, s, d2, H, topk_ids, topk_w, k, E, g, g_down, y,
                    tables_early ? 1 : 0);
}

cudaError_t launch_swizzle(const uint8_t* linear, int N, int K, uint8_t* swizzled, cudaStream_t s) {
  const long long items = (long long)((N + 127) / 128 * 128) * (K / 64);
  return launch_pdl(swizzle_kernel, dim3(grid_for(items)), dim3(kThreads), 0, s, linear, N, K / 16, swizzled);
}

}  // namespace moe
