/*
 * moe_nvfp4.h -- C ABI of libmoe_nvfp4.so, a GB300 (sm_103a) NVFP4
 * routed-expert MoE layer step.
 *
 * The step, as stated on the rocket blog page "The CUTLASS grouped GEMM beats
 * the scalar GEMV loop at every M, M=1 included" (section "What changed"):
 *   gather -> quantize (NVFP4) -> grouped GEMM w13 (fused gate|up, alpha = 1)
 *   -> SwiGLU with per-group gate/up weight_scale_2 -> quantize -> grouped
 *   GEMM w2 -> scatter-add weighted by router weight * down weight_scale_2.
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers owned by the caller unless a comment says
 *     "host". The library allocates no device memory. Device buffers must be
 *     16-byte aligned (MOE_ERR_INVALID otherwise).
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - Work is enqueued on `stream` and runs asynchronously; nothing here
 *     synchronizes except moe_nvfp4_check_status.
 *   - Return value: MOE_OK, or an error code. Arguments are validated on the
 *     host before anything is enqueued; an error return enqueues nothing,
 *     except MOE_ERR_CUDA (a launch failed part way).
 *   - Results are deterministic: the same inputs give bit-identical outputs,
 *     and a token's output does not depend on which other tokens share the
 *     batch (fixed expert order; every sum runs in a fixed order, atomics
 *     only hand out and count work).
 *
 * NVFP4 formats (page "Fusing the MoE layer's two grouped GEMMs is worth 4%",
 * table "Bytes decide it before the kernel runs": 0.5 + 1/16 byte/element)
 *   - packed e2m1: two 4-bit codes per byte, element 2j in bits 0-3 of byte
 *     j, element 2j+1 in bits 4-7; code bit 3 is the sign, magnitudes
 *     {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *   - block scales: one e4m3 (E4M3FN) byte per 16 consecutive elements of a
 *     row, stored in 128-row atoms (the tcgen05 / CUTLASS SFA-SFB layout the
 *     first page's section "The seam CUTLASS forced open" names). With
 *     Kc = K/16 scale columns, scale (row m, column c) of a region sits at
 *       ((m/128)*(Kc/4) + c/4)*512 + (m%32)*16 + ((m/32)%4)*4 + (c%4).
 *   - activations carry no global scale (alpha = 1): block scale =
 *     e4m3_rne_satfinite(amax/6); codes = e2m1_rne_satfinite(x/scale); both
 *     quotients those of correctly rounded fp32 division (the kernels reach
 *     the same codes by reciprocal and refinement); a block whose scale is 0
 *     has all-zero codes.
 *   - weights carry one fp32 global per projection (weight_scale_2); gate and
 *     up have their own (second page, "Different globals on the two halves").
 *
 * Routing: topk_ids[T, k] int32, topk_w[T, k] fp32. Slot s = t*k + j. An id
 * outside [0, E) marks an unused slot (it adds nothing to its token). Rows are
 * grouped by ascending expert id and, inside a group, by ascending slot
 * (first page, "What changed": ordered map, batch-invariant group order).
 * Activation scale regions are laid out per group, each padded with zero bytes
 * to a multiple of 128 rows; packed rows are contiguous with no padding.
 *
 * Where these signatures depart from the plain per-step seams the first page
 * names (packed weights plus a separate scale array per GEMM, group arrays as
 * loose pointers):
 *   - Weights reach the GEMMs pre-tiled (nvfp4_tile_weights, once at load
 *     time: e2m1 bytes already in the MMA's shared-memory swizzle with each
 *     256-value K stage's scales next to them, w13's gate and up rows
 *     interleaved per 64), so one contiguous copy feeds one pipeline stage and
 *     one accumulator holds both halves of a feature block for the fused
 *     SwiGLU. It is the same idea as the pages' load-time scale swizzle, taken
 *     one step further; the bytes are the same.
 *   - The group metadata (offsets, expert ids, token-block tables, row/slot
 *     maps) travels as one moe_groups_t filled on the device by the route
 *     step, because every later step needs the same tables and the host never
 *     sees them (no device-to-host sync in the step).
 *   - The GEMM entry points take the token-scale layout, which fixes the token
 *     block size a launch works in (32 or 128 rows).
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = 1,   /* null pointer, negative size, k > 32, E > 1024, ... */
  MOE_ERR_SHAPE = 2,     /* unsupported shape: a K not multiple of 64, an N not multiple of 128 */
  MOE_ERR_CUDA = 3,      /* a CUDA call or kernel launch failed */
  MOE_ERR_TIMEOUT = 4,   /* a device-side wait gave up (reported by moe_nvfp4_check_status) */
  MOE_ERR_WORKSPACE = 5  /* workspace smaller than moe_nvfp4_layer_workspace_size() */
};

/* Token-scale layouts (the e4m3 scales of quantized activation rows). Both
 * cut each group's rows into blocks and give block b the region of 128*(K/16)
 * bytes at b*128*(K/16), holding its rows in the atom layout above (row m of
 * the block, scale column c at ((c/4)*512 + (m%32)*16 + ((m/32)%4)*4 + c%4);
 * bytes no row fills are zero). They differ in the block size:
 *   MOE_SF_ATOM128: 128-row blocks (block numbering group_sf_block /
 *     block_info): the CUTLASS SFA layout, per group zero-padded to a multiple
 *     of 128 rows, that the first page's kernels wrote.
 *   MOE_SF_CHUNK32: 32-row blocks ("chunks", numbering group_chunk /
 *     chunk_info): only rows 0..31 of each atom are used.
 * The grouped GEMM takes the token operand in blocks of this size: one MMA of
 * N = the block's rows (rounded up to 16) per 128-row weight tile, so every
 * weight tile streams once per block. Its results are the same bits with
 * either layout (a row's sums do not depend on the MMA width). */
enum { MOE_SF_ATOM128 = 0, MOE_SF_CHUNK32 = 1 };

/* Group metadata produced by moe_route_groups (device int32 arrays, caller
 * owned; moe_groups_carve lays them out in one buffer).
 *   counts[5]            G (groups), R (rows), max Mg, total 128-row scale
 *                        blocks, total 32-row GEMM chunks
 *   group_offsets[E+1]   first row of group g; entry G holds R
 *   group_expert[E]      expert id of group g (ascending)
 *   group_sf_block[E+1]  first 128-row scale block of group g; entry G = total
 *   group_chunk[E+1]     first 32-row GEMM chunk of group g; entry G = total
 *   chunk_info[4*C]      per 32-row chunk c: first grouped row, rows (1..32),
 *                        expert id, group; C = min(E, T*k) + ceil(T*k/32)
 *   block_info[4*B]      per 128-row block b: first grouped row, rows
 *                        (1..128), expert id, group; B = min(E, T*k) +
 *                        ceil(T*k/128)
 *   row_slot[T*k]        slot t*k+j of grouped row r (r < R)
 *   slot_row[T*k]        grouped row of slot s, or -1 for an unused slot     */
typedef struct {
  int32_t* counts;
  int32_t* group_offsets;
  int32_t* group_expert;
  int32_t* group_sf_block;
  int32_t* group_chunk;
  int32_t* chunk_info;
  int32_t* block_info;
  int32_t* row_slot;
  int32_t* slot_row;
} moe_groups_t;

/* Expert weights (device), in the GEMM tiling made once at load time by
 * nvfp4_tile_weights from packed e2m1 [E, N, K/2] and linear e4m3 scales
 * [E, N, K/16]. w13 rows 0..I-1 are gate, I..2I-1 are up, back to back (first
 * page, "The seam CUTLASS forced open": the pair is the fused w13 operand);
 * w13 is tiled with interleave_rows = 2I, so every 128-row tile holds 64 gate
 * rows and the matching 64 up rows and the SwiGLU of a tile is formed in the
 * GEMM's epilogue. w2 is tiled plainly (interleave_rows = 0). */
typedef struct {
  int E;
  const uint8_t* w13_tiled;   /* nvfp4_tiled_bytes(E*2I, H) bytes: w13 [E, 2I, H], interleaved */
  const float* g_gate_up;     /* [E, 2]: gate global, up global */
  const uint8_t* w2_tiled;    /* nvfp4_tiled_bytes(E*H, I) bytes: w2 [E, H, I] */
  const float* g_down;        /* [E] */
} moe_nvfp4_weights_t;

/* Message for a status code (static string; never NULL). */
const char* moe_nvfp4_error_string(int status);

/* Reads and clears the device-side status word of the current device after
 * synchronizing `stream`: MOE_OK, or MOE_ERR_TIMEOUT if a kernel's bounded
 * wait gave up since the last check (its outputs are then invalid). Returns
 * MOE_ERR_CUDA if the synchronization itself fails. The word's device address
 * is looked up on a device's first call and kept for the life of the process:
 * it is not valid after the device's context is reset (cudaDeviceReset). */
int moe_nvfp4_check_status(cudaStream_t stream);

/* Bytes of the group metadata for T tokens, top-k, E experts; and a carve of
 * one caller buffer `mem` (256-byte aligned, that many bytes) into
 * moe_groups_t (host struct filled in; no device work). */
size_t moe_groups_bytes(int T, int k, int E);
int moe_groups_carve(void* mem, int T, int k, int E, moe_groups_t* groups /* host */);

/* Bytes of a token-scale region (layout MOE_SF_ATOM128 or MOE_SF_CHUNK32)
 * able to hold any grouping of up to R_max rows over E experts for a K-wide
 * operand: (min(E, R_max) + ceil(R_max/128)) * 128 * K/16 for ATOM128,
 * (min(E, R_max) + ceil(R_max/32)) * 128 * K/16 for CHUNK32. */
size_t nvfp4_sf_bytes(int R_max, int E, int K, int layout);

/* a1 -- route-group. Counts the T*k slots per expert, scans, and places rows
 * stably by (expert ascending, slot ascending); fills *groups on the device.
 * First page, "What changed" (std::map grouping, one fetch per expert) and
 * "Next" (host grouping cost). One CTA; E <= 1024. */
int moe_route_groups(const int32_t* topk_ids, int T, int k, int E,
                     const moe_groups_t* groups /* host struct of device pointers */,
                     cudaStream_t stream);

/* a1 + a2 -- moe_gather_rows: groups the slots (as moe_route_groups) and
 * copies x[slot/k, :] into grouped row order. xg [T*k, H] bf16; rows >= R
 * are left untouched. First page, "What changed": normed_[stream] -> one row
 * per (stream, expert). */
int moe_gather_rows(const uint16_t* x, int T, int H, const int32_t* topk_ids, int k, int E,
                    const moe_groups_t* groups, uint16_t* xg, cudaStream_t stream);

/* a3 / a6 -- nvfp4_quantize_rows: grouped bf16 rows [R_max, K] -> packed
 * [R_max, K/2] (rows >= R untouched) and the token scales `sf` in `layout`
 * (nvfp4_sf_bytes(R_max, E, K, layout) bytes; bytes no row fills are written
 * as 0). E is the expert count the groups were built for. First page, "What
 * changed" and "Proof" (byte-for-byte vs the host codec, group_m = {1, 130}).
 * K % 64 == 0. */
int nvfp4_quantize_rows(const uint16_t* rows, int R_max, int K, int E, const moe_groups_t* groups, int layout,
                        uint8_t* packed, uint8_t* sf, cudaStream_t stream);

/* a2 + a3 fused: quantizes x[row_slot[r]/k, :] straight into grouped NVFP4
 * rows; output identical to moe_gather_rows followed by nvfp4_quantize_rows. */
int moe_gather_quantize_rows(const uint16_t* x, int T, int H, int k, int E, const moe_groups_t* groups,
                             int layout, uint8_t* packed, uint8_t* sf, cudaStream_t stream);

/* a1 + a2 + a3 -- moe_route_gather_quantize: groups the T*k slots (as
 * moe_route_groups) and writes the routed rows x[row_slot[r]/k, :] as NVFP4
 * (packed [T*k, H/2], token scales in MOE_SF_CHUNK32). For T*k <= 32 (decode
 * batches) it is one launch: one warp routes, the CTA quantizes; otherwise
 * moe_route_groups then moe_gather_quantize_rows. Outputs are identical
 * either way. H % 64 == 0. */
int moe_route_gather_quantize(const int32_t* topk_ids, int T, int k, int E, const uint16_t* x, int H,
                              const moe_groups_t* groups, uint8_t* packed, uint8_t* sf, cudaStream_t stream);

/* a4 / a7 -- nvfp4_grouped_gemm: for every group g (expert e) and row r of
 * it, d[r, n] = sum_k A[r, k] * W[e, n, k] over dequantized values, no global
 * (alpha = 1), fp32 out, d [R_max, N] row-major (rows >= R untouched).
 * a_sf is in a_sf_layout; a group is processed in blocks of that layout's
 * size (32 rows for MOE_SF_CHUNK32, 128 for MOE_SF_ATOM128), each block
 * streaming the expert's weight tiles once: 128-row blocks for groups of
 * many rows (prefill-sized batches), 32-row ones for decode batches, where
 * more, smaller work units keep every SM busy. W [E, N, K] comes tiled by
 * nvfp4_tile_weights; w_interleaved says it was tiled with interleave_rows =
 * N (columns of d are in natural order either way). One launch for all
 * groups on tcgen05 block-scaled MMA (kind::mxf4nvf4, scale vector 16),
 * accumulators in tensor memory. First page, "What changed": grouped GEMM
 * w13 N=4096 K=4096 and w2 N=4096 K=2048, alpha = 1. N % 128 == 0,
 * K % 64 == 0; every pointer 16-byte aligned. */
int nvfp4_grouped_gemm(const uint8_t* a_packed, const uint8_t* a_sf, int a_sf_layout, const moe_groups_t* groups,
                       int R_max, const uint8_t* w_tiled, int w_interleaved, int E, int N, int K, float* d,
                       cudaStream_t stream);

/* a4 + a5 + a6 fused -- the w13 grouped GEMM with SwiGLU and requantization
 * in its epilogue: from the NVFP4 rows (a_sf in a_sf_layout) and w13 tiled
 * with interleave_rows = 2I, writes NVFP4 h: packed [R_max, I/2] and token
 * scales h_sf (the same layout, nvfp4_sf_bytes(R_max, E, I, a_sf_layout)
 * bytes). The fp32 gate|up product never leaves the chip. Bit-identical to
 * nvfp4_grouped_gemm + swiglu_grouped + nvfp4_quantize_rows. The second
 * page's "SwiGLU as an epilogue" found this inexpressible in CUTLASS grouped
 * GEMM; per-half globals are still applied in registers (option (a)).
 * I % 128 == 0, K % 64 == 0. */
int nvfp4_grouped_gemm_swiglu(const uint8_t* a_packed, const uint8_t* a_sf, int a_sf_layout,
                              const moe_groups_t* groups, int R_max, const uint8_t* w13_tiled, int E, int I, int K,
                              const float* g_gate_up, uint8_t* h_packed, uint8_t* h_sf, cudaStream_t stream);

/* a4 .. a7 in one persistent launch -- both grouped GEMMs of the layer: the
 * w13 GEMM with SwiGLU and requantization in its epilogue (as
 * nvfp4_grouped_gemm_swiglu, writing h_packed/h_sf) and the w2 GEMM reading
 * that h (as nvfp4_grouped_gemm into d2 [R_max, H] fp32). Each 256-wide K
 * stage of a token block's w2 work starts once the four w13 tiles writing
 * those h features are done, so w2's weights stream, and its first stages
 * run, while w13 finishes. This is the launch
 * moe_nvfp4_layer makes between quantization and the scatter-add; the pages
 * ran the two GEMMs as separate launches (second page, "Fusing the MoE
 * layer's two grouped GEMMs is worth 4%").
 * x_packed/x_sf: NVFP4 token rows [R_max, H/2] and their scales in
 * sf_layout; h_sf is written in the same layout.
 * gate: moe_expert_gemms_gate_bytes(R_max, E, I) bytes of device scratch for
 * the launch's work counters. Zero it once before the first call; a call
 * that completes leaves it zero. After an error (e.g. MOE_ERR_TIMEOUT from
 * moe_nvfp4_check_status) zero it again. Calls sharing a gate must not run
 * concurrently.
 * H % 128 == 0, I % 128 == 0. */
size_t moe_expert_gemms_gate_bytes(int R_max, int E, int I);
int nvfp4_moe_expert_gemms(const uint8_t* x_packed, const uint8_t* x_sf, int sf_layout, const moe_groups_t* groups,
                           int R_max, const moe_nvfp4_weights_t* w, int H, int I, uint8_t* h_packed,
                           uint8_t* h_sf, float* d2, void* gate, cudaStream_t stream);

/* a5 -- swiglu_grouped: h[r, n] = silu(d13[r, n]*g_gate[e]) * (d13[r, I+n]*g_up[e]),
 * computed in fp32 (CUDA expf) and rounded once to bf16. d13 [R_max, 2I]
 * fp32, h [R_max, I] bf16. Second page, "Different globals on the two halves",
 * option (a): the per-half globals are applied here. */
int swiglu_grouped(const float* d13, int R_max, int I, int E, const moe_groups_t* groups,
                   const float* g_gate_up, uint16_t* h, cudaStream_t stream);

/* a5 + a6 fused: SwiGLU as swiglu_grouped, then the a3 codec on the bf16 h,
 * written as packed [R_max, I/2] + token scales in `layout`
 * (nvfp4_sf_bytes(R_max, E, I, layout) bytes). Identical to swiglu_grouped
 * followed by nvfp4_quantize_rows. */
int swiglu_quantize_grouped(const float* d13, int R_max, int I, int E, const moe_groups_t* groups, int layout,
                            const float* g_gate_up, uint8_t* packed, uint8_t* sf, cudaStream_t stream);

/* a8 -- moe_scatter_add: y[t, :] = sum over t's used slots, in ascending
 * grouped-row order (= ascending expert id), of topk_w[t, j] * g_down[e] *
 * d2[row, :]; fp32 accumulation, rounded once to bf16. y [T, H] is
 * overwritten; a token with no used slot gets zeros. First page, "What
 * changed" (weighted by router weight * down weight_scale_2) and "Proof"
 * (shared accumulator row, ordered accumulation). k <= 32. */
int moe_scatter_add(const float* d2, int H, const int32_t* topk_ids, const float* topk_w,
                    int T, int k, int E, const moe_groups_t* groups, const float* g_down,
                    uint16_t* y, cudaStream_t stream);

/* Workspace bytes of moe_nvfp4_layer for these sizes (the GEMM launch's work
 * counters, group metadata, NVFP4 activations and scales, fp32 GEMM
 * outputs). */
size_t moe_nvfp4_layer_workspace_size(int T, int k, int E, int H, int I);

/* The token-scale layout (token block size) moe_nvfp4_layer uses for T
 * tokens, top-k, E experts: MOE_SF_ATOM128 (128-row blocks) when the batch
 * routes at least 16 rows per expert on average (T*k >= 16*E, prefill-sized:
 * weight tiles then stream once per 128 rows instead of once per 32), else
 * MOE_SF_CHUNK32. A shape rule, not a fallback: the output bits are the same
 * either way. A caller composing the step from the separate entry points can
 * use it to match the layer's choice. */
int moe_nvfp4_layer_sf_layout(int T, int k, int E);

/* The whole step a1..a8 on `stream`: route-group, gather+quantize, grouped
 * GEMM w13 with SwiGLU+requantize in its epilogue, grouped GEMM w2,
 * scatter-add. Four launches for T*k > 32 (route, gather+quantize, both
 * GEMMs in one persistent launch, scatter), three for decode-sized batches
 * (T*k <= 32: route + gather + quantize in one). Each launch may start while
 * the previous one finishes (programmatic dependent launch). Token rows go
 * through the GEMMs in blocks of moe_nvfp4_layer_sf_layout(T, k, E).
 * x [T, H] bf16, y [T, H] bf16 (overwritten). With k > 0, x, topk_ids,
 * topk_w and y may also be pinned host memory (unified addressing): the
 * kernels then read and write them in place over the CPU-GPU link.
 * `workspace` is caller device memory of ws_bytes >=
 * moe_nvfp4_layer_workspace_size(T, k, w->E, H, I), 256-byte aligned (any
 * contents). Calls sharing a workspace run in stream
 * order. H % 128 == 0, I % 128 == 0, k <= 32, E <= 1024. */
int moe_nvfp4_layer(const uint16_t* x, int T, int H, int I, const int32_t* topk_ids,
                    const float* topk_w, int k, const moe_nvfp4_weights_t* w /* host struct */,
                    void* workspace, size_t ws_bytes, uint16_t* y, cudaStream_t stream);

/* moe_nvfp4_layer_static -- moe_nvfp4_layer without a workspace argument,
 * for callers that cannot allocate device memory: a plugin or kernel library
 * whose host owns every allocation, code that must not synchronize the device
 * (cudaMalloc/cudaFree can), or a caller that builds the step into work it
 * does not own. The pages have no counterpart; it exists for such callers.
 * The workspace is one device array inside the library of
 * MOE_NVFP4_STATIC_SCRATCH_BYTES (8 MiB), held by every GPU that loads the
 * library until the process exits. Sizes whose
 * moe_nvfp4_layer_workspace_size() exceeds it return MOE_ERR_WORKSPACE (at
 * H = 4096, I = 2048, E = 288 that allows T*k <= 119, i.e. decode up to 14
 * streams of top-8); arguments are checked as by moe_nvfp4_layer first, with
 * the same status codes. Nothing is allocated: the first call on a device
 * looks up the array's device address once and keeps it for the life of the
 * process (make that first call before any stream capture; the address is
 * not valid after the device's context is reset with cudaDeviceReset, and
 * calls after such a reset are not supported); no part of the array needs to
 * start at zero, every byte the step reads is written earlier in the same
 * call. All calls share the one array:
 * calls that can overlap on the GPU (different streams, or the same stream
 * from several host threads without ordering) race and must be serialized by
 * the caller. Arguments and results otherwise as moe_nvfp4_layer. */
#define MOE_NVFP4_STATIC_SCRATCH_BYTES (8u << 20)
int moe_nvfp4_layer_static(const uint16_t* x, int T, int H, int I, const int32_t* topk_ids,
                           const float* topk_w, int k, const moe_nvfp4_weights_t* w /* host struct */,
                           uint16_t* y, cudaStream_t stream);

/* The GEMV path (W4A16). First page, section "Proof", the paragraph comparing
 * the grouped and GEMV paths at M=1: the GEMV path multiplies the exact bf16 activations
 * against the NVFP4 weights (no activation quantization), so its output
 * differs materially from the W4A4 grouped path's; the page keeps it as an
 * explicit override and fallback. Here it is the reference against which the
 * grouped path's activation quantization is measured.
 *
 * nvfp4_grouped_gemv_w4a16 -- d[r, n] = sum_k a(r)[k] * W[e, n, k] for the
 * rows r of each group (expert e), dequantized weight without its global,
 * fp32 accumulation in a fixed K order (a row's result does not depend on the
 * batch). Rows: a(r) = a[row_slot[r] / src_k] when src_k > 0 (gathered from
 * the token rows [T, K], src_k = top-k), else a[r] ([R_max, K]); bf16,
 * 16-byte aligned. w_tiled: nvfp4_tile_weights output for [E, N, K]
 * (w_interleaved as there). d [R_max, N] fp32 (rows of routed slots written).
 * N % 128 == 0, K % 64 == 0, K <= 14336; MOE_ERR_SHAPE otherwise. */
int nvfp4_grouped_gemv_w4a16(const uint16_t* a, int src_k, const moe_groups_t* groups, int R_max,
                             const uint8_t* w_tiled, int w_interleaved, int E, int N, int K, float* d,
                             cudaStream_t stream);

/* moe_nvfp4_layer_w4a16 -- the whole step a1..a8 on the GEMV path: route,
 * w13 GEMV on the gathered bf16 rows, SwiGLU to bf16 h (no requantization),
 * w2 GEMV on h, scatter-add; five launches. Arguments, weights and results as
 * moe_nvfp4_layer; workspace of moe_nvfp4_layer_w4a16_workspace_size() bytes
 * (256-byte aligned, any contents). H, I <= 14336. */
size_t moe_nvfp4_layer_w4a16_workspace_size(int T, int k, int E, int H, int I);
int moe_nvfp4_layer_w4a16(const uint16_t* x, int T, int H, int I, const int32_t* topk_ids,
                          const float* topk_w, int k, const moe_nvfp4_weights_t* w /* host struct */,
                          void* workspace, size_t ws_bytes, uint16_t* y, cudaStream_t stream);

/* Load-time helper (not part of the timed step): weight tiling for the
 * grouped GEMM. packed [rows, K/2] e2m1 and linear scales [rows, K/16] ->
 * `tiled` (nvfp4_tiled_bytes(rows, K) bytes): for each 128-row tile and each
 * 256-value K stage, 16 KB of packed bytes in the 128-byte-swizzled order the
 * MMA reads from shared memory (16-byte chunk c of row r at chunk c ^ (r%8))
 * followed by the stage's 2 KB of scales in the atom layout; values past K
 * are zero. Same bytes as the inputs (up to the K padding), reordered so that
 * each stage is one contiguous read. Like the first page's load-time scale
 * swizzle ("The seam CUTLASS forced open"), it is paid once per weight, not
 * per step. For stacked experts pass rows = E*N. interleave_rows = 0 keeps
 * row order; interleave_rows = N (rows per expert, a multiple of 256) makes
 * tile t of an expert hold its rows 64t..64t+63 and N/2+64t..N/2+64t+63.
 * rows % 128 == 0, K % 64 == 0. */
size_t nvfp4_tiled_bytes(int rows, int K);
int nvfp4_tile_weights(const uint8_t* packed, const uint8_t* sf_linear, int rows, int K, int interleave_rows,
                       uint8_t* tiled, cudaStream_t stream);

/* Load-time helper (not part of the timed step): linear row-major scales
 * [N, K/16] -> the atom layout, N padded up to a multiple of 128 with zero
 * bytes (output ceil(N/128)*128*K/16 bytes). First page, "The seam CUTLASS
 * forced open": fuel::swizzle_block_scales, once per projection.
 * K % 64 == 0. */
int nvfp4_swizzle_block_scales(const uint8_t* linear, int N, int K, uint8_t* swizzled,
                               cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_H */
