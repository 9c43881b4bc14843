// NVFP4 x NVFP4 grouped GEMM on tcgen05 block-scaled MMA (sm_103a).
//
// Computes, for every group g (expert e) of the routed rows,
//   d[r, n] = sum_k A[r, k] * W[e, n, k]       (dequantized values, alpha = 1)
// which is the "grouped GEMM (w13, fused)" and "grouped GEMM (w2)" step of the
// rocket blog page "The CUTLASS grouped GEMM beats the scalar GEMV loop at
// every M" (section "What changed"). The pages ran CUTLASS's SM120 grouped
// kernel with 128-row token tiles; this kernel is written for GB300 instead:
//
//  * Swap-AB. The weight tile is the MMA's A operand (M = 128 output features)
//    and the group's tokens are the B operand (N = the token block's rows
//    rounded up to 16), so a decode group of one row costs a 16-wide MMA, not
//    a 128-row tile. The second page ("Tiles below M=8") notes that the wasted
//    token extent costs no HBM traffic; here it costs no tensor work either.
//  * Persistent CTAs, two per SM, walk the ragged work list of (token block
//    of a group, 128-row weight tile) units in a fixed order; every unit
//    streams its weight tile over the full K once. Two CTAs per SM because a
//    CTA's tcgen05 operations execute one after another: with one CTA per SM
//    the tensor pipe, not HBM, set the pace (at decode, and at prefill-sized
//    batches even with a ring twice as deep). Token blocks are 32 rows
//    (decode and mid-sized batches: more, smaller units) or 128 rows
//    (prefill-sized batches: each weight tile streams once per 128 rows of a
//    group, N up to 128 MMAs).
//  * Weights arrive pre-tiled (nvfp4_tile_weights, a load-time step): for
//    every 128-row tile and 256-value K stage, 16 KB of e2m1 bytes already in
//    the 128-byte-swizzled shared-memory image followed by the 2 KB of e4m3
//    scale atoms, so a stage is one contiguous 18 KB bulk copy.
//  * Warp roles: warp 0 issues the weight bulk copies (L2 evict-first) into an
//    mbarrier ring; warp 8 copies the token rows (into the 128-byte swizzle)
//    and their scale atoms with 16-byte cp.async copies from all its lanes;
//    warps 6 and 7 copy each stage's scales into tensor memory (tcgen05.cp);
//    warp 1 issues tcgen05.mma.kind::mxf4nvf4 (scale vector 16) into a
//    double-buffered TMEM accumulator; warps 2-5 drain TMEM (tcgen05.ld).
//  * Epilogue either writes fp32 rows, or (w13 in the layer) applies SwiGLU
//    with the per-half globals and requantizes h to NVFP4 right there, so the
//    fp32 gate|up product never reaches HBM. For that the w13 tiles hold 64
//    gate rows and the matching 64 up rows (the first page's gate|up pair,
//    "The seam CUTLASS forced open", reordered at load time); the pages could
//    not express this epilogue in CUTLASS ("SwiGLU as an epilogue").
//  * Every wait is bounded; on expiry the kernel records MOE_ERR_TIMEOUT,
//    drains its own copies, frees tensor memory and returns.
// A row's result never depends on other rows: the K loop order is fixed and
// each output column of the MMA depends only on its own token.
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "nvfp4_codec.cuh"
#include "ldcg.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;            // weight rows per tile = MMA M
constexpr int kStageKBytes = 128;   // K bytes per stage and row = 256 e2m1 values
constexpr int kAtomBytes = 512;     // one scale atom: 128 rows x 4 scales (64 K values)
constexpr int kATileBytes = kBM * kStageKBytes;  // 16 KB
constexpr int kSfStageBytes = 4 * kAtomBytes;    // 2 KB per operand and stage
constexpr int kWStageBytes = kATileBytes + kSfStageBytes;  // one tiled weight stage: 18 KB
constexpr int kTokChunk = 32;       // epilogue columns per pass (and the small batches' token block)
constexpr int kMaxStages = 16;
constexpr int kThreads = 288;       // warp 0: weights, 1: MMA, 2-5: epilogue, 6-7: scale copies, 8: tokens
// Per CTA, with two CTAs per SM: shared memory (half the SM's 228 KB less
// 1 KB reserved per CTA) and tensor memory columns (half of the SM's 512).
constexpr int kCtasPerSm = 2;
constexpr int kSmemBytes = 114688;
constexpr int kTmemCols = 256;
constexpr int kXchStride = kTokChunk + 1;          // fused epilogue: gate and up values [2][64][33] floats
constexpr int kXchHalf = 64 * kXchStride;          // floats of one half (gate or up)
constexpr int kXchBytes = 17408;                   // 2 * 64 * 33 * 4 rounded up to 1 KB
constexpr int kUq = 8;                             // unit queue: producer -> MMA, scale copies, epilogue
constexpr int kHeader = 2048;                      // barriers, TMEM address, queue, small-batch routing tables
constexpr int kSmallSlots = 32;                    // inline routing: at most 32 slots
constexpr int kUqReaders = 1 + 2 + 1 + 128;  // MMA thread, scale-copy threads, token loader, epilogue threads

// One grouped GEMM over the routed rows: weights (tiled), token operand,
// token scales, output.
struct Job {
  const uint8_t* w_tiled;
  const uint8_t* a_packed;  // token rows [R_max, K/2], NVFP4
  const uint8_t* a_sf;      // token scales, MOE_SF_CHUNK32, K wide
  float* d;                 // plain epilogue: fp32 rows [R_max, N]
  int N, K;
  int interleaved;          // tiles hold 64 rows of each half of N
};

struct GemmArgs {
  Job j0, j1;               // j1 is used when njobs == 2
  int njobs;
  int fused0;               // job 0: SwiGLU + requantize epilogue (needs interleaved)
  uint8_t* h_packed;        // ... NVFP4 h [R_max, N0/4] ...
  uint8_t* h_sf;            // ... and its token scales (MOE_SF_CHUNK32, K = N0/2) ...
  const float* g_gate_up;   // ... with the per-expert (gate, up) globals
  int* chunk_done;          // njobs == 2: per (chunk, job-1 K stage), job-0 tiles of that stage's h
                            // features finished (zero at launch)
  int* work_ctr;            // njobs == 2: next unit to claim (zero at launch)
  int* exit_ctr;            // njobs == 2: CTAs done; the last one zeroes the counters again
  // small != 0: T*k <= 32 slots; every CTA routes them itself (one warp)
  // from topk_ids, written two or more launches back, and before waiting for
  // the previous kernel (the gather-quantize of these rows) claims its first
  // unit and issues that unit's first weight stages (early must be 0)
  int small;
  const int32_t* topk_ids;  // [S] slots
  int S, E;
  const int32_t* counts;
  const int4* blk_tab;      // per token block: first row, rows, expert, group
  int bt;                   // token block rows: 32 (chunk_info) or 128 (block_info)
  int* status;
  int early;                // 1: group metadata and weights were written two or more launches back
  long long wait_budget;    // clock64 cycles a single wait may take
};

// ------------------------------- PTX helpers --------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// 16-byte copy global -> shared through L2 only (the source may have been
// written by another CTA or the previous kernel).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// One arrival on the barrier once all of this thread's earlier cp.async
// copies have landed (counts against the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Orders shared memory written through the generic proxy (cp.async, plain
// stores), as seen by this thread, before its later async-proxy reads
// (tcgen05.mma and tcgen05.cp operands).
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bulk copy with an L2 policy (weights are read once per step: evict first).
__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}\n" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void tc_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tc_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_cp_scales(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Orders this thread's view of global memory (after an acquire) before its
// later reads through another proxy.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle
// (16-byte piece c of row r at piece c ^ (r % 8)): rows of 128 bytes, 8-row
// groups 1024 bytes apart (stride byte offset), descriptor version 1,
// swizzle mode 2 (128B).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Descriptor of one 512-byte scale atom for tcgen05.cp.32x128b: 32 rows of
// 16 bytes, no swizzle, 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t desc_scales(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor, kind::mxf4nvf4: A and B e2m1 (format 1), both
// K-major, e4m3 scales, M = 128, N = n (multiple of 16), dense K = 64.
__device__ __forceinline__ uint32_t idesc_nvf4(int n) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

// h = silu(gate) * up for the globals-scaled halves, in fp32 with CUDA's
// expf, rounded once to bf16 (returned as the fp32 value of that bf16).
__device__ __forceinline__ float swiglu_bf16(float gt, float uv) {
  const float hv = gt / (1.0f + expf(-gt)) * uv;
  return bf16_to_f32(__bfloat16_as_ushort(__float2bfloat16_rn(hv)));
}

// NVFP4 codec across a warp holding one value per lane: lanes 16 b .. 16 b +
// 15 are one 16-value block (b = 0, 1). Returns, in every lane, the 32-bit
// word of packed codes of its 8-lane group (lane 8 i + j's code in nibble j)
// and, in `scales`, the two blocks' e4m3 scale bytes (block 0 low byte).
__device__ __forceinline__ void quantize_feature(float v, int lane, uint32_t& word, uint32_t& scales) {
  float amax = fabsf(v);
  amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, 4));
  amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, 8));
  const uint32_t sc = block_scale_code(amax);
  uint32_t code = 0u;  // an underflowed block keeps all-zero codes
  if (sc != 0u) {
    const float dsc = e4m3_value(sc);
    code = e2m1x2(block_quotient(v, dsc, rcp_approx(dsc)), 0.0f) & 0xFu;
  }
  uint32_t w = code << (4 * (lane & 7));
  w |= __shfl_xor_sync(~0u, w, 1);
  w |= __shfl_xor_sync(~0u, w, 2);
  w |= __shfl_xor_sync(~0u, w, 4);
  word = w;
  scales = sc | (__shfl_sync(~0u, sc, 16) << 8);
}

struct Ctl {
  volatile int* abort_flag;
  int* status;
  long long budget;
};

__device__ __forceinline__ void give_up(const Ctl& c) {
  *c.abort_flag = 1;
  atomicExch(c.status, (int)MOE_ERR_TIMEOUT);
}

__device__ __noinline__ bool wait_phase(uint32_t bar, uint32_t parity, const struct Ctl& c);
// Bounded wait with the first poll inline (the common case: already complete).
__device__ __forceinline__ bool wait_fast(uint32_t bar, uint32_t parity, const struct Ctl& c) {
  return mbar_try_wait(bar, parity) || wait_phase(bar, parity, c);
}

// Bounded wait: false if this or another role gave up.
__device__ __noinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Ctl& c) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*c.abort_flag) return false;
    if (clock64() - t0 > c.budget) {
      give_up(c);
      return false;
    }
  }
}

// Warp-wide: how many stages from `ks` on are ready, i.e. their counters
// (stage i: ctr[i] >= min(4, kc4 - 4 i)) have reached their targets. Lane l
// polls stage ks + l with an acquire load, so one L2 round trip covers every
// remaining stage; waits (bounded) until stage ks is ready, then a warp
// barrier makes what the counters published visible to every lane's copies.
// Returns the first stage not known ready (> ks), or -1 if the wait gave up.
__device__ __noinline__ int ready_stages(const int* ctr, int ks, int nk, int kc4, int lane, const Ctl& c) {
  const long long t0 = clock64();
  while (true) {
    const int i = ks + lane;
    bool sat = true;
    if (i < nk) sat = ld_acquire(ctr + i) >= min(4, kc4 - 4 * i);
    const unsigned m = __ballot_sync(~0u, sat);
    if (m & 1u) {
      __syncwarp();                // each lane's acquire is ordered before every lane's copies
      fence_proxy_async_global();
      const int run = (~m) ? __ffs(~m) - 1 : 32;  // leading ready stages
      return min(nk, ks + run);
    }
    int stop = 0;
    if (lane == 0) {
      if (*c.abort_flag) stop = 1;
      else if (clock64() - t0 > c.budget) { give_up(c); stop = 1; }
    }
    if (__shfl_sync(~0u, stop, 0)) return -1;
    __nanosleep(128);
  }
}



// One unit of work: token block `chunk` of a group (32 or 128 rows) against
// 128-row weight tile `nt` of the group's expert, for job 0 (units [0, U0))
// or job 1. The block's token scales are one 512-byte atom per 64 K values.
struct Unit {
  int job, chunk, row0, nvalid, nmma, nt, expert, nk, kc4;
  const uint8_t* w;    // the tile's first 18 KB stage
  const uint8_t* sfb;  // the chunk's first token-scale block
};

__device__ __forceinline__ Unit decode_unit(int u, const GemmArgs& p, int U0, int nt0, int nt1, const int4* tab) {
  Unit un;
  un.job = u >= U0 ? 1 : 0;
  const int v = un.job ? u - U0 : u;
  const int ntl = un.job ? nt1 : nt0;
  un.chunk = v / ntl;
  un.nt = v - un.chunk * ntl;
  // row0, rows, expert, group: the small mode's table in shared memory, else the group metadata
  const int4 c = tab ? tab[un.chunk] : ld_cg(p.blk_tab + un.chunk);
  un.row0 = c.x;
  un.nvalid = c.y;
  un.expert = c.z;
  un.nmma = (un.nvalid + 15) & ~15;
  const int K = un.job ? p.j1.K : p.j0.K;
  un.nk = (K + 255) / 256;
  un.kc4 = K / 64;
  un.w = (un.job ? p.j1.w_tiled : p.j0.w_tiled) + ((size_t)un.expert * ntl + un.nt) * un.nk * kWStageBytes;
  un.sfb = (un.job ? p.j1.a_sf : p.j0.a_sf) + (size_t)un.chunk * un.kc4 * kAtomBytes;
  return un;
}

// Small mode: warp 0 routes the <= 32 slots, one per lane, into this CTA's
// tables: rows ascend by (expert, slot), one group and one 32-row chunk per
// expert, the same rows and chunks moe_route_groups produces.
__device__ __noinline__ void small_route(const GemmArgs& p, int lane, int4* s_tab, int* s_meta) {
  const bool in = lane < p.S;
  const int e = in ? ld_cg(p.topk_ids + lane) : -1;
  const bool ok = in && e >= 0 && e < p.E;
  const int key = ok ? e : 0x7fffffff;
  const unsigned peers = __match_any_sync(~0u, key);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  const int n = __popc(peers);
  const unsigned leaders = __ballot_sync(~0u, ok && rank == 0);
  int less = 0, gless = 0;  // rows and groups of lower experts
  for (int j = 0; j < kSmallSlots; ++j) {
    const int kj = __shfl_sync(~0u, key, j);
    if (kj < key) {
      ++less;
      gless += (leaders >> j) & 1u;
    }
  }
  int mx = ok ? n : 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) mx = max(mx, __shfl_xor_sync(~0u, mx, o));
  if (ok && rank == 0) s_tab[gless] = make_int4(less, n, e, gless);
  if (lane == 0) {
    s_meta[0] = __popc(leaders);
    s_meta[2] = mx;
  }
}

// Two CTAs per SM must fit: the register budget ptxas derives from that is
// 96 a thread (at 108 only one CTA per SM was resident, measured).
__global__ void __launch_bounds__(kThreads, kCtasPerSm) gemm_kernel(GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  // barrier slots: full[16], empty[16], acc_full[2], acc_empty[2], drain, scales_ready[16], unit_done,
  // xch_full, xch_free, drain2, unit queue full/empty[8], drain3, token full[16]
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * kMaxStages + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * kMaxStages + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kMaxStages + 4);
  auto sfr_bar = [&](int s) { return bar0 + 8u * (2 * kMaxStages + 5 + s); };
  const uint32_t udone_bar = bar0 + 8u * (3 * kMaxStages + 5);
  const uint32_t xfull_bar = bar0 + 8u * (3 * kMaxStages + 6);
  const uint32_t xfree_bar = bar0 + 8u * (3 * kMaxStages + 7);
  const uint32_t drain2_bar = bar0 + 8u * (3 * kMaxStages + 8);
  auto uqf_bar = [&](int i) { return bar0 + 8u * (3 * kMaxStages + 9 + i); };
  auto uqe_bar = [&](int i) { return bar0 + 8u * (3 * kMaxStages + 9 + kUq + i); };
  const uint32_t drain3_bar = bar0 + 8u * (3 * kMaxStages + 9 + 2 * kUq);
  auto tfull_bar = [&](int s) { return bar0 + 8u * (3 * kMaxStages + 10 + 2 * kUq + s); };  // token operand landed
  // after the barriers (< 768 bytes): TMEM address, abort flag, unit queue
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 768);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 772);
  volatile int* uq = reinterpret_cast<volatile int*>(smem + 832);
  int4* s_tab = reinterpret_cast<int4*>(smem + 1024);     // small mode: chunk table [32]
  int* s_meta = reinterpret_cast<int*>(smem + 1536);      // small mode: G, -, max rows per group

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(sfr_bar(s), 2);  // weight-scale and token-scale copies
      mbar_init(tfull_bar(s), 32);  // one cp.async arrival per token-loader lane
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 4 * 32);
    }
    mbar_init(drain_bar, 1);
    mbar_init(drain2_bar, 1);
    mbar_init(drain3_bar, 1);
    mbar_init(udone_bar, 4 * 32);
    mbar_init(xfull_bar, 128);  // every epilogue thread stored its row's values
    mbar_init(xfree_bar, 128);  // every epilogue thread finished reading them
    for (int i = 0; i < kUq; ++i) {
      mbar_init(uqf_bar(i), 1);
      mbar_init(uqe_bar(i), kUqReaders);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const Ctl ctl{abort_flag, p.status, p.wait_budget};
  // Programmatic dependent launch: this grid may start while the previous
  // kernel in the stream still runs. Everything it reads must be complete
  // first. With p.early the group metadata, the work counters and the
  // weights are two or more launches old (complete); in small mode the
  // routing is done here from topk_ids (two or more launches old) and the
  // previous kernel cleared the counters before it let this grid launch. In
  // both, only the token operand (and whatever follows from it) waits below,
  // and the first unit's weights stream in meanwhile.
  const bool early_issue = p.early || p.small;
  if (p.small) {
    // Route the <= 32 slots in warp 0 of every CTA (one slot per lane).
    if (warp == 0) small_route(p, lane, s_tab, s_meta);
    __syncthreads();
  } else if (!p.early) {
    pdl_wait();
    pdl_trigger();
  }
  const int4* tab = p.small ? s_tab : nullptr;
  // ---- schedule shape, identical on every thread ----
  const int G = p.small ? s_meta[0] : ld_cg(p.counts + 0);
  const int maxmg = p.small ? s_meta[2] : ld_cg(p.counts + 2);
  const int nchunks = p.small ? G : ld_cg(p.counts + (p.bt == 128 ? 3 : 4));  // token blocks
  const int nt0 = p.j0.N / kBM;
  const int nt1 = p.njobs > 1 ? p.j1.N / kBM : 1;
  const int U0 = nchunks * nt0;
  const int total_units = U0 + (p.njobs > 1 ? nchunks * nt1 : 0);
  const int nk1 = p.njobs > 1 ? (p.j1.K + 255) / 256 : 1;  // job-1 K stages (dependency counters per chunk)
  const bool has_xch = p.fused0 != 0;
  const int tn = min(p.bt, max(16, (maxmg + 15) & ~15));   // token rows per B stage (MMA N at most)
  const int acc_cols = (tn + 31) & ~31;                     // accumulator buffers start 32-column aligned
  const int nacc = 2 * acc_cols + 64 <= kTmemCols ? 2 : 1;  // double-buffered unless TMEM is short
  const int stage_bytes = kWStageBytes + tn * kStageKBytes + kSfStageBytes;
  const int avail = kSmemBytes - 1024 - kHeader - (has_xch ? kXchBytes : 0);
  int stages = min(kMaxStages, avail / stage_bytes);
  stages = min(stages, (kTmemCols - nacc * acc_cols) / 32);
  // per stage: [weights 16 KB | weight scales 2 KB] ... then token rows, token scales, exchange
  const uint32_t sW = smem_u32(smem + kHeader);
  const uint32_t sB = sW + (uint32_t)stages * kWStageBytes;
  const uint32_t sSFB = sB + (uint32_t)stages * tn * kStageKBytes;
  float* xch = reinterpret_cast<float*>(smem + kHeader + (size_t)stages * stage_bytes);


  // The producer hands every role the same unit sequence through the queue:
  // unit ids, then -1. Returns the next unit, -1 at the end, -2 on a timeout.
  int q_idx = 0;
  uint32_t q_phase = 0;
  auto next_unit = [&]() -> int {
    if (!wait_phase(uqf_bar(q_idx), q_phase, ctl)) return -2;
    const int u = uq[q_idx];
    mbar_arrive(uqe_bar(q_idx));
    if (++q_idx == kUq) { q_idx = 0; q_phase ^= 1u; }
    return u;
  };

  if (warp == 0) {
    // ========================= weight stream producer =========================
    // Units are taken in increasing order: with two jobs from a global
    // counter (every job-0 unit is claimed, by a running CTA, before any
    // job-1 unit, so a job-1 wait always ends however many CTAs are
    // resident), otherwise blockIdx.x, blockIdx.x + gridDim.x, ...
    // This thread issues only the weight copies (one 18 KB bulk copy per
    // stage); warp 8 issues the token copies: a thread issues a bulk copy
    // every few hundred cycles whatever its size, so the two streams go out
    // from two warps.
    if (lane == 0) {
      const bool dynamic = p.work_ctr != nullptr;
      int static_next = blockIdx.x;
      auto claim = [&]() -> int {
        int u;
        if (dynamic) {
          u = atomicAdd(p.work_ctr, 1);
        } else {
          u = static_next;
          static_next += gridDim.x;
        }
        return u < total_units ? u : -1;
      };
      int wq = 0;
      uint32_t wq_phase = 0;
      bool ok = true;
      auto push = [&](int u) {
        if (!wait_phase(uqe_bar(wq), wq_phase ^ 1u, ctl)) return false;
        uq[wq] = u;
        mbar_arrive(uqf_bar(wq));
        if (++wq == kUq) { wq = 0; wq_phase ^= 1u; }
        return true;
      };
      int stage = 0;
      uint32_t phase = 0, filled = 0, fill_parity = 0;
      const uint64_t stream_policy = policy_evict_first();
      // With early_issue, the first unit's first weight stages go out before
      // waiting for the previous kernel (they do not depend on it).
      int cur = (total_units > 0) ? claim() : -1;
      int prefetched = 0;
      if (early_issue) {
        if (cur >= 0) {
          const Unit un = decode_unit(cur, p, U0, nt0, nt1, tab);
          for (int ks = 0; ks < un.nk && ks < stages; ++ks) {
            const int natoms = min(4, un.kc4 - 4 * ks);
            const uint32_t wbytes = kATileBytes + natoms * kAtomBytes;
            mbar_expect_tx(full_bar(ks), wbytes);
            bulk_load_hint(sW + ks * kWStageBytes, un.w + (size_t)ks * kWStageBytes, wbytes, full_bar(ks),
                           stream_policy);
            filled |= 1u << ks;
            ++prefetched;
          }
        }
        pdl_wait();
        pdl_trigger();
      }
      int issued = 0;
      while (ok) {
        if (!push(cur)) { ok = false; break; }
        if (cur < 0) break;
        const Unit un = decode_unit(cur, p, U0, nt0, nt1, tab);
        for (int ks = 0; ks < un.nk; ++ks, ++issued) {
          if (issued >= prefetched) {
            if (!wait_fast(empty_bar(stage), phase ^ 1u, ctl)) { ok = false; break; }
            const int natoms = min(4, un.kc4 - 4 * ks);
            const uint32_t wbytes = kATileBytes + natoms * kAtomBytes;
            mbar_expect_tx(full_bar(stage), wbytes);
            bulk_load_hint(sW + stage * kWStageBytes, un.w + (size_t)ks * kWStageBytes, wbytes, full_bar(stage),
                           stream_policy);
            filled |= 1u << stage;
            fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
        // the next unit is claimed once this one's copies are all issued (a
        // ring's worth of stages still in flight hides the atomic's latency);
        // claiming earlier would let a CTA hoard units behind a job-1 wait
        cur = claim();
      }
      if (!ok || *abort_flag) {  // this role, or another, gave up: nothing of ours may be in flight at exit
        // let every copy this thread issued land before the CTA exits
        for (int s = 0; s < stages; ++s)
          if (filled & (1u << s)) {
            const long long t0 = clock64();
            while (!mbar_try_wait(full_bar(s), (fill_parity >> s) & 1u) && clock64() - t0 < ctl.budget) {
            }
          }
      }
    }
  } else if (warp == 8) {
    // ========================= token operand loader =========================
    // Per stage, once the slot is free: the stage's 128 bytes of each valid
    // token row, stored in the 128-byte swizzle the MMA reads, and the rows'
    // scale atoms, as 16-byte cp.async copies spread over the warp's lanes;
    // each lane's copies make one of tfull[s]'s 32 arrivals. (A bulk or TMA
    // copy costs its issuing thread a few hundred cycles; these cost a load
    // instruction.) Rows past the chunk's valid rows are not copied: they only
    // feed accumulator columns the epilogue never reads. Job 1 reads h,
    // written by job 0: the copies of its K stage ks wait until the job-0
    // tiles that write those h features are done (the weights stream on
    // meanwhile).
    if (early_issue) pdl_wait();  // the token rows come from the previous kernel
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    while (ok) {
      int u = 0;
      if (lane == 0) u = next_unit();
      u = __shfl_sync(~0u, u, 0);
      if (u < 0) { ok = u == -1; break; }
      const Unit un = decode_unit(u, p, U0, nt0, nt1, tab);
      const int K = un.job ? p.j1.K : p.j0.K;
      const uint8_t* rows = (un.job ? p.j1.a_packed : p.j0.a_packed) + (size_t)un.row0 * (K / 2);
      int ready = un.job == 1 ? 0 : un.nk;  // stages whose token operand is known to be written
      for (int ks = 0; ks < un.nk; ++ks) {
        int got = 0;
        if (lane == 0) got = wait_fast(empty_bar(stage), phase ^ 1u, ctl) ? 1 : 0;
        if (!__shfl_sync(~0u, got, 0)) { ok = false; break; }
        const int natoms = min(4, un.kc4 - 4 * ks);
        // job 1's K stage ks is h features [256 ks, 256 ks + 256): the job-0
        // tiles 4 ks .. 4 ks + natoms - 1 of the chunk write them
        if (ks >= ready) {
          ready = ready_stages(p.chunk_done + (size_t)un.chunk * un.nk, ks, un.nk, un.kc4, lane, ctl);
          if (ready < 0) { ok = false; break; }
        }
        // row r's 16-byte piece c (2 per 64-value K atom) goes to piece c ^ (r % 8) of the row
        const uint32_t dst = sB + (uint32_t)(stage * tn * kStageKBytes);
        const int per_row = 2 * natoms;
        const uint8_t* src = rows + (size_t)ks * kStageKBytes;
        if (per_row == 8) {  // a full stage: 8 pieces per row (shifts, not a division)
          for (int i = lane; i < un.nvalid * 8; i += 32) {
            const int r = i >> 3, c = i & 7;
            cp_async16(dst + (uint32_t)(r * kStageKBytes + ((c ^ (r & 7)) << 4)), src + (size_t)r * (K / 2) + c * 16);
          }
        } else {
          for (int i = lane; i < un.nvalid * per_row; i += 32) {
            const int r = i / per_row, c = i - r * per_row;
            cp_async16(dst + (uint32_t)(r * kStageKBytes + ((c ^ (r & 7)) << 4)), src + (size_t)r * (K / 2) + c * 16);
          }
        }
        const uint32_t sdst = sSFB + (uint32_t)(stage * kSfStageBytes);
        const uint8_t* ssrc = un.sfb + (size_t)ks * kSfStageBytes;
        for (int i = lane; i < natoms * (kAtomBytes / 16); i += 32) cp_async16(sdst + (uint32_t)(i * 16), ssrc + i * 16);
        cp_async_arrive(tfull_bar(stage));
        if (++stage == stages) { stage = 0; phase ^= 1u; }
      }
    }
    // this role, or another, gave up: let every copy of this warp land before the CTA exits
    if (!ok || *abort_flag) cp_async_wait_all();
  } else if (warp == 6 || warp == 7) {
    // ======================== scale copies into TMEM =======================
    // Warp 6 copies the weight scales, warp 7 the token scales of every stage
    // (two issuing threads: a single one's tcgen05 issue rate would pace the
    // stage). Slot s's scale columns are rewritten only after the slot was
    // refilled, i.e. after the MMAs that read them completed (empty[s]).
    if (lane == 0) {
      const bool tok = warp == 7;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      while (ok) {
        const int u = next_unit();
        if (u < 0) { ok = u == -1; break; }
        const int K = u >= U0 ? p.j1.K : p.j0.K;
        const int nk = (K + 255) / 256, kc4 = K / 64;
        for (int ks = 0; ks < nk; ++ks) {
          if (!wait_fast(tok ? tfull_bar(stage) : full_bar(stage), phase, ctl)) { ok = false; break; }
          tc_fence_after();
          if (tok) fence_proxy_async_shared();  // token scales were written by cp.async
          const int natoms = min(4, kc4 - 4 * ks);
          const uint32_t col = tmem_base + (uint32_t)(nacc * acc_cols + 32 * stage + (tok ? 16 : 0));
          const uint64_t src = desc_scales(tok ? sSFB + stage * kSfStageBytes : sW + stage * kWStageBytes + kATileBytes);
          // atom a at +512 bytes: +32 in the descriptor's address field
          for (int a = 0; a < natoms; ++a) tc_cp_scales(col + 4 * a, src + 32 * a);
          tc_commit(sfr_bar(stage));
          if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok || *abort_flag) {  // this role, or another, gave up: nothing of ours may be in flight at exit
        // wait for this thread's copies before TMEM is freed
        const uint32_t db = tok ? drain3_bar : drain2_bar;
        tc_commit(db);
        const long long t0 = clock64();
        while (!mbar_try_wait(db, 0) && clock64() - t0 < ctl.budget) {
        }
      }
    }
  } else if (warp == 1) {
    // ============================= MMA issuer =============================
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      while (ok) {
        const int u = next_unit();
        if (u < 0) { ok = u == -1; break; }
        const Unit un = decode_unit(u, p, U0, nt0, nt1, tab);
        if (!wait_phase(acce_bar(acc), acc_phase ^ 1u, ctl)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * acc_cols);
        const uint32_t idesc = idesc_nvf4(un.nmma);
        for (int ks = 0; ks < un.nk; ++ks) {
          // operands landed (full) and their scales are in tensor memory (scales ready)
          if (!wait_fast(full_bar(stage), phase, ctl) || !wait_fast(tfull_bar(stage), phase, ctl) ||
              !wait_fast(sfr_bar(stage), phase, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          fence_proxy_async_shared();  // the token rows were written by cp.async
          const int natoms = min(4, un.kc4 - 4 * ks);
          const uint32_t sf_col = tmem_base + (uint32_t)(nacc * acc_cols + 32 * stage);
          // K step a (32 bytes along the 128-byte swizzled rows): +2 in the address field
          const uint64_t adesc = desc_sw128(sW + stage * kWStageBytes);
          const uint64_t bdesc = desc_sw128(sB + stage * tn * kStageKBytes);
          if (natoms == 4) {
            tc_mma_nvf4(d_tmem, adesc, bdesc, idesc, sf_col, sf_col + 16, ks != 0);
            tc_mma_nvf4(d_tmem, adesc + 2, bdesc + 2, idesc, sf_col + 4, sf_col + 20, 1u);
            tc_mma_nvf4(d_tmem, adesc + 4, bdesc + 4, idesc, sf_col + 8, sf_col + 24, 1u);
            tc_mma_nvf4(d_tmem, adesc + 6, bdesc + 6, idesc, sf_col + 12, sf_col + 28, 1u);
          } else {
            for (int a = 0; a < natoms; ++a)
              tc_mma_nvf4(d_tmem, adesc + 2 * a, bdesc + 2 * a, idesc, sf_col + 4 * a, sf_col + 16 + 4 * a,
                          (ks | a) != 0);
          }
          tc_commit(empty_bar(stage));
          if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(accf_bar(acc));
        if (++acc == nacc) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok || *abort_flag) {  // this role, or another, gave up: nothing of ours may be in flight at exit
        // wait for every MMA issued so far before TMEM is freed
        tc_commit(drain_bar);
        const long long t0 = clock64();
        while (!mbar_try_wait(drain_bar, 0) && clock64() - t0 < ctl.budget) {
        }
      }
    }
  } else {
    // ============================== epilogue ==============================
    // The unit's accumulator (tile rows = TMEM lanes, token rows = columns)
    // is read 32 columns at a time; the buffer is released after the last
    // read. Plain: fp32 rows of d. Fused (job 0 of the layer): SwiGLU with
    // the per-half globals, bf16 rounding and the NVFP4 codec, written as h.
    const int quad = warp & 3;     // TMEM lanes 32*quad .. 32*quad+31 = tile rows
    const int et = threadIdx.x - 64;  // 0..127 over the four epilogue warps
    const int tr = quad * 32 + lane;  // tile row
    const int half = p.j0.N / 2;
    int acc = 0;
    uint32_t acc_phase = 0, xph = 0, uph = 0;
    bool ok = true;
    while (ok) {
      const int u = next_unit();
      if (u < 0) break;
      const Unit un = decode_unit(u, p, U0, nt0, nt1, tab);
      if (!wait_phase(accf_bar(acc), acc_phase, ctl)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * acc_cols);
      const bool fused = un.job == 0 && p.fused0;
      // plain: this thread's output column n of d, rows row0 ..
      const int N = un.job ? p.j1.N : p.j0.N;
      const int il = un.job ? p.j1.interleaved : p.j0.interleaved;
      const int n = !il ? un.nt * kBM + tr : (tr < 64 ? un.nt * 64 + tr : N / 2 + un.nt * 64 + (tr - 64));
      float* dst = fused ? nullptr : (un.job ? p.j1.d : p.j0.d) + (size_t)un.row0 * N + n;
      // fused: atom nt of the block's h scales (h features 64 nt .. 64 nt + 63) and this thread's h bytes
      uint8_t* sfblk = fused ? p.h_sf + ((size_t)un.chunk * (half / 64) + un.nt) * kAtomBytes : nullptr;
      const float gg = fused ? ld_cg(p.g_gate_up + 2 * un.expert) : 0.0f;
      const float gu = fused ? ld_cg(p.g_gate_up + 2 * un.expert + 1) : 0.0f;
      uint8_t* hp_base = fused ? p.h_packed + (size_t)un.row0 * (half / 2) + un.nt * 32 : nullptr;
      for (int c0 = 0; c0 < un.nvalid; c0 += kTokChunk) {
        const int nc = min(kTokChunk, un.nvalid - c0);  // uniform across the warp
        uint32_t r[kTokChunk];
        // 16 or 32 columns from a 32-column-aligned address
        if (nc <= 16) {
          tc_ld_32x32b_x16(taddr + (uint32_t)c0, *reinterpret_cast<uint32_t(*)[16]>(r));
        } else {
          tc_ld_32x32b_x32(taddr + (uint32_t)c0, r);
        }
        tc_wait_ld();
        if (c0 + kTokChunk >= un.nvalid) {
          tc_fence_before();
          mbar_arrive(acce_bar(acc));  // the accumulator buffer is free again
        }
        if (!fused) {
#pragma unroll
          for (int j = 0; j < kTokChunk; ++j)
            if (j < nc) dst[(size_t)(c0 + j) * N] = __uint_as_float(r[j]);
          continue;
        }
        // ---- fused SwiGLU + requantize ----
        // Every epilogue thread stores its row's values (gate rows: tile rows
        // 0..63, up rows: 64..127, feature = row % 64) to shared memory; then
        // warp q computes features 32 (q % 2) .. + 31 for every other column
        // (columns q / 2, q / 2 + 2, ...): all four warps share the per-column
        // chain (SwiGLU, block amax, codec), which with only the two gate-row
        // warps working made the epilogue, not the MMAs, pace 48-row blocks.
        if (!wait_phase(xfree_bar, xph ^ 1u, ctl)) { ok = false; break; }
        {
          float* row = xch + (quad >= 2 ? kXchHalf : 0) + (tr & 63) * kXchStride;
#pragma unroll
          for (int j = 0; j < kTokChunk; ++j)
            if (j < nc) row[j] = __uint_as_float(r[j]);
        }
        mbar_arrive(xfull_bar);
        if (!wait_phase(xfull_bar, xph, ctl)) { ok = false; break; }
        {
          const int f = (quad & 1) * 32 + lane;  // feature 64 nt + f of h
          const float* grow = xch + f * kXchStride;
          const float* urow = xch + kXchHalf + f * kXchStride;
          uint8_t* hpf = hp_base + (quad & 1) * 16 + (lane >> 1);
          uint8_t* sfq = sfblk + 2 * (quad & 1);
          for (int j0 = quad >> 1; j0 < nc; j0 += 2) {
            const float h0 = swiglu_bf16(grow[j0] * gg, urow[j0] * gu);
            uint32_t w0, s0;
            quantize_feature(h0, lane, w0, s0);
            if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(hpf + (size_t)(c0 + j0) * (half / 2)) = w0;
            if (lane == 0) {
              const int m0 = c0 + j0;
              *reinterpret_cast<uint16_t*>(sfq + (m0 & 31) * 16 + (m0 >> 5) * 4) = (uint16_t)s0;
            }
          }
        }
        mbar_arrive(xfree_bar);
        xph ^= 1u;
      }
      if (!ok) break;
      if (++acc == nacc) { acc = 0; acc_phase ^= 1u; }
      if (fused) {
        // the rest of the block's 512-byte scale atom (token rows past the block's rows) is zero:
        // word et holds row (et / 4) + 32 (et % 4)
        if ((et >> 2) + 32 * (et & 3) >= un.nvalid) reinterpret_cast<uint32_t*>(sfblk)[et] = 0u;
      }
      if (un.job == 0 && p.njobs > 1) {
        // publish this tile of the block to job 1: the writers' arrivals
        // (release, CTA scope) reach one thread, whose release-add at GPU
        // scope makes all of them visible to the acquiring reader
        mbar_arrive(udone_bar);
        if (et == 0) {
          if (!wait_phase(udone_bar, uph, ctl)) break;
          red_release_add(p.chunk_done + (size_t)un.chunk * nk1 + un.nt / 4, 1);  // tile nt: h features 64 nt ..
        }
        uph ^= 1u;
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && p.exit_ctr) {
    // The last CTA out leaves the counters zero for the next launch: every
    // other CTA has made its last claim and read its last chunk count.
    __threadfence();
    if (atomicAdd(p.exit_ctr, 1) == (int)gridDim.x - 1) {
      for (int c = 0; c < nchunks * nk1; ++c) p.chunk_done[c] = 0;
      *p.work_ctr = 0;
      *p.exit_ctr = 0;
    }
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols) : "memory");
  }
}

}  // namespace

cudaError_t launch_grouped_gemm(const moe_groups_t& g, int R_max, int E, int layout, const GemmJob& j0,
                                const SwigluOut* swiglu, const GemmJob* j1, int* gate, const SmallFront* front,
                                bool early, int* status, cudaStream_t s) {
  if (front && (early || front->S > kSmallSlots || front->S < 1 || layout != MOE_SF_CHUNK32))
    return cudaErrorInvalidValue;
  if (j1 && !gate) return cudaErrorInvalidValue;
  GemmArgs p = {};
  auto fill = [](Job& J, const GemmJob& src) {
    J.w_tiled = src.w_tiled;
    J.a_packed = src.a_packed;
    J.a_sf = src.a_sf;
    J.d = src.d;
    J.N = src.N;
    J.K = src.K;
    J.interleaved = src.w_interleaved ? 1 : 0;
  };
  fill(p.j0, j0);
  if (j1) fill(p.j1, *j1);
  p.njobs = j1 ? 2 : 1;
  p.fused0 = swiglu ? 1 : 0;
  if (swiglu) {
    p.h_packed = swiglu->packed;
    p.h_sf = swiglu->sf;
    p.g_gate_up = swiglu->g_gate_up;
  }
  p.work_ctr = j1 ? gate : nullptr;
  p.exit_ctr = j1 ? gate + 1 : nullptr;
  p.chunk_done = j1 ? gate + 2 : nullptr;
  p.counts = g.counts;
  const bool big = layout == MOE_SF_ATOM128;
  p.bt = big ? 128 : kTokChunk;
  p.blk_tab = reinterpret_cast<const int4*>(big ? g.block_info : g.chunk_info);
  p.status = status;
  p.early = early ? 1 : 0;
  if (front) {
    p.small = 1;
    p.topk_ids = front->topk_ids;
    p.S = front->S;
    p.E = E;
  }
  p.wait_budget = 2000000000LL;
  const long long units_bound = row_blocks_bound(R_max, E, layout) * (j0.N / kBM + (j1 ? j1->N / kBM : 0));
  cudaError_t err = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  const long long slots = (long long)num_sms() * kCtasPerSm;
  const int grid = (int)(units_bound < slots ? units_bound : slots);
  return launch_pdl(gemm_kernel, dim3(grid > 0 ? grid : 1), dim3(kThreads), kSmemBytes, s, p);
}

}  // namespace moe
