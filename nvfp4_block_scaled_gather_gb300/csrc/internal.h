// Host-side launchers shared by the translation units of libmoe_nvfp4.so.
// Each returns cudaSuccess or the launch error; arguments are validated by
// the C-ABI layer (moe_api.cu) before these are called.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime_api.h>

#include "moe_nvfp4.h"

namespace moe {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;

// Upper bound on 128-row scale blocks for R_max rows in at most G_max groups.
inline long long sf_blocks_bound(long long R_max, long long G_max) {
  long long g = G_max < R_max ? G_max : R_max;
  return g + (R_max + 127) / 128;
}
// Upper bound on 32-row GEMM chunks for R_max rows in at most G_max groups.
inline long long chunks_bound(long long R_max, long long G_max) {
  long long g = G_max < R_max ? G_max : R_max;
  return g + (R_max + 31) / 32;
}
// Row blocks of a token-scale layout (128-row atoms or 32-row chunks).
inline long long row_blocks_bound(long long R_max, long long G_max, int layout) {
  return layout == MOE_SF_ATOM128 ? sf_blocks_bound(R_max, G_max) : chunks_bound(R_max, G_max);
}
// Bytes of a token-scale region for K-wide rows (both layouts: rows x K/16).
inline size_t token_sf_bytes(long long R_max, long long G_max, long long K, int layout) {
  return layout == MOE_SF_ATOM128 ? (size_t)sf_blocks_bound(R_max, G_max) * 128 * (K / 16)
                                  : (size_t)chunks_bound(R_max, G_max) * 32 * (K / 64) * 16;
}

int num_sms();  // SM count of the current device (cached per device)

// Host-side argument checks of moe_nvfp4_layer (everything but the
// workspace): MOE_OK, MOE_ERR_INVALID or MOE_ERR_SHAPE. T == 0 is valid.
int layer_arg_status(const uint16_t* x, int T, int H, int I, const int32_t* topk_ids, const float* topk_w, int k,
                     const moe_nvfp4_weights_t* w, const uint16_t* y);

// zero/nzero: an int array the route kernel also clears (may be null).
// slot_sf (may be null): per slot s, the token block of bt rows (32 or 128)
// and the row in it where slot s's row sits, as (block << 7) | row; -1 for
// an unused slot.
cudaError_t launch_route(const int32_t* topk_ids, int S, int E, const moe_groups_t& g, cudaStream_t s,
                         int* zero = nullptr, int nzero = 0, int* slot_sf = nullptr, int bt = 0);
cudaError_t launch_gather(const uint16_t* x, int H, int k, int R_max, const moe_groups_t& g,
                          uint16_t* xg, cudaStream_t s);
// src_k > 0: rows are x[row_slot[r] / src_k]; src_k == 0: rows are src[r].
// E bounds the group count (grid size); CTAs past the routed blocks exit.
cudaError_t launch_quantize(const uint16_t* src, int src_k, int R_max, int E, int K,
                            const moe_groups_t& g, int layout, uint8_t* packed, uint8_t* sf, cudaStream_t s);
// a2 + a3 token by token: each token row of x [T, K] quantized once and
// written to each of its routed rows (packed [R_max, K/2], token scales in
// `layout` at the places slot_sf gives, from launch_route with the matching
// bt). The same bytes as launch_quantize(x, k, ...) for every routed row;
// scale words of rows past a block's valid rows stay as they were.
cudaError_t launch_quantize_tokens(const uint16_t* x, int T, int K, int k, const moe_groups_t& g,
                                   const int* slot_sf, int layout, uint8_t* packed, uint8_t* sf, cudaStream_t s);
// a1 + a2 + a3 in one launch for S = T*k <= 32 slots (rows x[slot / k]),
// token scales in MOE_SF_CHUNK32; same outputs as launch_route followed by
// launch_quantize(x, k, ...).
cudaError_t launch_route_quantize_small(const int32_t* topk_ids, int S, int E, const moe_groups_t& g, int* zero,
                                        int nzero, const uint16_t* x, int k, int K, uint8_t* packed, uint8_t* sf,
                                        cudaStream_t s);
constexpr int kSmallRouteSlots = 32;
// h != nullptr: write bf16 h; otherwise packed/sf get the quantized h.
cudaError_t launch_swiglu(const float* d13, int R_max, int E, int I, const moe_groups_t& g, int layout,
                          const float* g_gate_up, uint16_t* h, uint8_t* packed, uint8_t* sf, cudaStream_t s);
// Load-time weight tiling for the grouped GEMM (rows % 128 == 0). With
// interleave_rows > 0 (rows per expert, a multiple of 256) each tile takes 64
// rows of an expert's first half and the matching 64 of its second half.
cudaError_t launch_tile(const uint8_t* packed, const uint8_t* sf_linear, int rows, int K, int interleave_rows,
                        uint8_t* tiled, cudaStream_t s);
inline size_t tiled_bytes(long long rows, long long K) { return (size_t)(rows / 128) * ((K + 255) / 256) * 18432; }
// tables_early: the routing tables (and topk_ids, topk_w, g_down) were written
// two or more launches back, so they are read before waiting for the previous
// kernel (which must have waited for its own predecessor before it triggered).
cudaError_t launch_scatter(const float* d2, int H, const int32_t* topk_ids, const float* topk_w, int T, int k,
                           int E, const moe_groups_t& g, const float* g_down, uint16_t* y, cudaStream_t s,
                           bool tables_early = false);
cudaError_t launch_swizzle(const uint8_t* linear, int N, int K, uint8_t* swizzled, cudaStream_t s);

// tcgen05 grouped GEMM (nvfp4_gemm.cu), one persistent launch over one or
// two jobs. A job: token rows a_packed [R_max, K/2] with token scales a_sf
// (in `layout`: MOE_SF_CHUNK32 = 32-row token blocks, MOE_SF_ATOM128 =
// 128-row token blocks), tiled weights [E, N, K], fp32 output d [R_max, N].
// w_interleaved: each 128-row weight tile holds 64 rows of the first half of
// N and the matching 64 rows of the second half (nvfp4_tile_weights with
// interleave); d still gets natural column order.
// swiglu != nullptr (job 0 needs w_interleaved, N = 2I): job 0's epilogue
// applies SwiGLU with the per-expert (gate, up) globals and writes NVFP4 h
// (packed [R_max, I/2], token scales MOE_SF_CHUNK32), bit-identical to
// swiglu_grouped followed by nvfp4_quantize_rows; job 0's d is not written.
// j1 != nullptr: job 1 runs in the same launch and may read what job 0
// wrote: a job-1 unit of a token block starts its token loads once all of
// job 0's tiles writing that stage's features are done. gate holds
// gate_ints(R_max, E, K1) ints, zero at launch: the unit claim counter, the
// count of finished CTAs, then per (token block, job-1 K stage of 256) the
// count of finished job-0 tiles. The last CTA to finish zeroes them again, so a launch
// that completes leaves gate ready for the next.
// early: the group metadata, gate and the weights were written two or more
// launches back (true inside moe_nvfp4_layer), so the GEMM may read them and
// start streaming weights before the previous kernel has finished.
// status: device word that records a wait timeout (MOE_ERR_TIMEOUT).
inline long long gate_ints(long long R_max, long long E, long long K1) {
  return 2 + chunks_bound(R_max, E) * ((K1 + 255) / 256);
}
struct SwigluOut {
  uint8_t* packed;
  uint8_t* sf;
  const float* g_gate_up;
};
struct GemmJob {
  const uint8_t* a_packed;
  const uint8_t* a_sf;
  const uint8_t* w_tiled;
  bool w_interleaved;
  int N, K;
  float* d;
};
// front != nullptr (small batches, S = T*k <= 32; early must be false):
// every CTA routes the slots itself from topk_ids (which must be two or more
// launches old) and, before waiting for the previous kernel (the
// gather-quantize of these rows), claims its first unit and issues that
// unit's first weight stages.
struct SmallFront {
  const int32_t* topk_ids;
  int S;
};
// front requires layout == MOE_SF_CHUNK32.
cudaError_t launch_grouped_gemm(const moe_groups_t& g, int R_max, int E, int layout, const GemmJob& j0,
                                const SwigluOut* swiglu, const GemmJob* j1, int* gate, const SmallFront* front,
                                bool early, int* status, cudaStream_t s);

// The layer's token block size for S = T*k slots over E experts: 128-row
// blocks (MOE_SF_ATOM128) when S >= 16*E (and the batch is not decode-sized),
// else 32-row chunks.
inline int layer_sf_layout(long long S, long long E) {
  return (S > kSmallRouteSlots && S >= 16 * E) ? MOE_SF_ATOM128 : MOE_SF_CHUNK32;
}

// W4A16 grouped GEMV (nvfp4_gemv.cu): d [R_max, N] fp32 = bf16 rows times the
// group's expert's tiled NVFP4 weight [E, N, K] (no global); rows are
// a[row_slot[r] / src_k] (src_k > 0) or a[r]. N % 128 == 0, K % 64 == 0,
// K <= 14336 (four rows of fp32 activations staged in shared memory).
cudaError_t launch_gemv_w4a16(const uint16_t* a, int src_k, int R_max, int E, const moe_groups_t& g,
                              const uint8_t* w_tiled, bool interleaved, int N, int K, float* d, cudaStream_t s);

}  // namespace moe
