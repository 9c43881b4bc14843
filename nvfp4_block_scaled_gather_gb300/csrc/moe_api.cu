// C ABI of libmoe_nvfp4.so: argument checks, workspace carving and the fused
// layer entry. The kernels live in moe_kernels.cu and nvfp4_gemm.cu.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"

namespace moe {

// Device-side status word: kernels whose bounded waits expire write
// MOE_ERR_TIMEOUT here; moe_nvfp4_check_status reads and clears it.
__device__ int g_status_word = 0;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices] = {0};
int* g_status_ptr[kMaxDevices] = {nullptr};

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

// Device address of g_status_word on the current device (set up once per device).
int* status_ptr() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(ptr);
  }
  return g_status_ptr[dev];
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Every device buffer the kernels read or write with vector accesses must be
// 16-byte aligned; a null pointer passes here and is checked separately.
bool misaligned(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 != 0; }

bool groups_ok(const moe_groups_t* g) {
  return g && g->counts && g->group_offsets && g->group_expert && g->group_sf_block && g->group_chunk &&
         g->chunk_info && g->block_info && g->row_slot && g->slot_row;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool layout_ok(int layout) { return layout == MOE_SF_ATOM128 || layout == MOE_SF_CHUNK32; }

struct LayerWs {
  moe_groups_t groups;
  uint8_t *xq, *xsf, *hq, *hsf;
  int* slot_sf;  // per slot, its place in the token-scale layout (batches of more than 32 slots)
  float* d2;
  int* gate;  // the GEMM's unit claim counter, finished CTAs, then w13 tiles finished per token block
  int ngate;
  size_t bytes;
};

// Carves the layer workspace; base may be null to only compute the size.
LayerWs carve_layer(void* base, int T, int k, int E, int H, int I) {
  LayerWs w;
  const size_t S = (size_t)T * k;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? static_cast<uint8_t*>(base) + off : nullptr;
    off += align256(bytes);
    return p;
  };
  w.ngate = (int)gate_ints((long long)S, E, I);
  w.gate = reinterpret_cast<int*>(take((size_t)w.ngate * sizeof(int)));
  uint8_t* gmem = take(moe_groups_bytes(T, k, E));
  if (base) moe_groups_carve(gmem, T, k, E, &w.groups);
  w.xq = take(S * H / 2);
  w.slot_sf = S > (size_t)kSmallRouteSlots ? reinterpret_cast<int*>(take(S * sizeof(int))) : nullptr;
  const int layout = layer_sf_layout((long long)S, E);
  w.xsf = take(token_sf_bytes((long long)S, E, H, layout));
  w.hq = take(S * I / 2);
  w.hsf = take(token_sf_bytes((long long)S, E, I, layout));
  w.d2 = reinterpret_cast<float*>(take(S * H * sizeof(float)));
  w.bytes = off;
  return w;
}

// The GEMV path's workspace: group metadata, fp32 w13 output, bf16 h, fp32 w2 output.
struct GemvWs {
  moe_groups_t groups;
  float* d13;
  uint16_t* h;
  float* d2;
  size_t bytes;
};

GemvWs carve_layer_w4a16(void* base, int T, int k, int E, int H, int I) {
  GemvWs w;
  const size_t S = (size_t)T * k;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? static_cast<uint8_t*>(base) + off : nullptr;
    off += align256(bytes);
    return p;
  };
  uint8_t* gmem = take(moe_groups_bytes(T, k, E));
  if (base) moe_groups_carve(gmem, T, k, E, &w.groups);
  w.d13 = reinterpret_cast<float*>(take(S * 2 * I * sizeof(float)));
  w.h = reinterpret_cast<uint16_t*>(take(S * I * sizeof(uint16_t)));
  w.d2 = reinterpret_cast<float*>(take(S * H * sizeof(float)));
  w.bytes = off;
  return w;
}

constexpr int kGemvMaxK = 14336;  // four fp32 activation rows of K in 227 KB of shared memory

}  // namespace

int layer_arg_status(const uint16_t* x, int T, int H, int I, const int32_t* topk_ids, const float* topk_w, int k,
                     const moe_nvfp4_weights_t* w, const uint16_t* y) {
  if (!w || T < 0 || k < 0 || k > kMaxTopK || H <= 0 || I <= 0 || w->E <= 0 || w->E > kMaxExperts)
    return MOE_ERR_INVALID;
  if (H % 128 || I % 128) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!x || !y || (k > 0 && (!topk_ids || !topk_w))) return MOE_ERR_INVALID;
  if (misaligned(x) || misaligned(y)) return MOE_ERR_INVALID;
  if (!w->w13_tiled || !w->g_gate_up || !w->w2_tiled || !w->g_down) return MOE_ERR_INVALID;
  if (misaligned(w->w13_tiled) || misaligned(w->w2_tiled)) return MOE_ERR_INVALID;
  if ((long long)T * k > (1LL << 30) || (long long)w->E * 2 * I > (1LL << 31)) return MOE_ERR_SHAPE;
  return MOE_OK;
}

int num_sms() {
  const int dev = current_device();
  if (dev < 0) return 148;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_nvfp4_error_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID: return "invalid argument";
    case MOE_ERR_SHAPE: return "unsupported shape";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

int moe_nvfp4_check_status(cudaStream_t stream) {
  int* p = status_ptr();
  if (!p) return MOE_ERR_CUDA;
  int host = 0;
  if (cudaMemcpyAsync(&host, p, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(p, 0, sizeof(int), stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  return host;
}

size_t moe_groups_bytes(int T, int k, int E) {
  if (T < 0 || k < 0 || E < 0) return 0;
  const size_t S = (size_t)T * k;
  return align256(16 * 4) + align256(4 * (size_t)(E + 1)) + align256(4 * (size_t)E) +
         2 * align256(4 * (size_t)(E + 1)) + align256(16 * (size_t)chunks_bound((long long)S, E)) +
         align256(16 * (size_t)sf_blocks_bound((long long)S, E)) + 2 * align256(4 * S);
}

int moe_groups_carve(void* mem, int T, int k, int E, moe_groups_t* g) {
  if (!mem || !g || T < 0 || k < 0 || E <= 0) return MOE_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(mem) % 256) return MOE_ERR_INVALID;
  const size_t S = (size_t)T * k;
  uint8_t* p = static_cast<uint8_t*>(mem);
  g->counts = reinterpret_cast<int32_t*>(p); p += align256(16 * 4);
  g->group_offsets = reinterpret_cast<int32_t*>(p); p += align256(4 * (size_t)(E + 1));
  g->group_expert = reinterpret_cast<int32_t*>(p); p += align256(4 * (size_t)E);
  g->group_sf_block = reinterpret_cast<int32_t*>(p); p += align256(4 * (size_t)(E + 1));
  g->group_chunk = reinterpret_cast<int32_t*>(p); p += align256(4 * (size_t)(E + 1));
  g->chunk_info = reinterpret_cast<int32_t*>(p); p += align256(16 * (size_t)chunks_bound((long long)S, E));
  g->block_info = reinterpret_cast<int32_t*>(p); p += align256(16 * (size_t)sf_blocks_bound((long long)S, E));
  g->row_slot = reinterpret_cast<int32_t*>(p); p += align256(4 * S);
  g->slot_row = reinterpret_cast<int32_t*>(p);
  return MOE_OK;
}

size_t nvfp4_sf_bytes(int R_max, int E, int K, int layout) {
  if (R_max < 0 || E < 0 || K < 0 || (layout != MOE_SF_ATOM128 && layout != MOE_SF_CHUNK32)) return 0;
  return token_sf_bytes(R_max, E, K, layout);
}

int moe_route_groups(const int32_t* topk_ids, int T, int k, int E, const moe_groups_t* groups, cudaStream_t stream) {
  if (!groups_ok(groups) || T < 0 || k < 0 || E <= 0) return MOE_ERR_INVALID;
  if (E > kMaxExperts || k > kMaxTopK) return MOE_ERR_INVALID;
  if ((long long)T * k > (1LL << 30)) return MOE_ERR_INVALID;
  if ((long long)T * k > 0 && !topk_ids) return MOE_ERR_INVALID;
  return status_of(launch_route(topk_ids, T * k, E, *groups, stream));
}

int moe_gather_rows(const uint16_t* x, int T, int H, const int32_t* topk_ids, int k, int E,
                    const moe_groups_t* groups, uint16_t* xg, cudaStream_t stream) {
  if (H <= 0 || H % 8 || (T > 0 && k > 0 && (!x || !xg))) return MOE_ERR_INVALID;
  if (misaligned(x) || misaligned(xg)) return MOE_ERR_INVALID;
  const int st = moe_route_groups(topk_ids, T, k, E, groups, stream);
  if (st != MOE_OK || T * k == 0) return st;
  return status_of(launch_gather(x, H, k, T * k, *groups, xg, stream));
}

int nvfp4_quantize_rows(const uint16_t* rows, int R_max, int K, int E, const moe_groups_t* groups, int layout,
                        uint8_t* packed, uint8_t* sf, cudaStream_t stream) {
  if (!groups_ok(groups) || R_max < 0 || K <= 0 || E <= 0 || E > kMaxExperts || !layout_ok(layout))
    return MOE_ERR_INVALID;
  if (K % 64) return MOE_ERR_SHAPE;
  if (R_max == 0) return MOE_OK;
  if (!rows || !packed || !sf) return MOE_ERR_INVALID;
  if (misaligned(rows) || misaligned(packed) || misaligned(sf)) return MOE_ERR_INVALID;
  return status_of(launch_quantize(rows, 0, R_max, E, K, *groups, layout, packed, sf, stream));
}

int moe_gather_quantize_rows(const uint16_t* x, int T, int H, int k, int E, const moe_groups_t* groups, int layout,
                             uint8_t* packed, uint8_t* sf, cudaStream_t stream) {
  if (!groups_ok(groups) || T < 0 || k < 0 || k > kMaxTopK || H <= 0 || E <= 0 || E > kMaxExperts ||
      !layout_ok(layout))
    return MOE_ERR_INVALID;
  if (H % 64) return MOE_ERR_SHAPE;
  if (T * k == 0) return MOE_OK;
  if (!x || !packed || !sf) return MOE_ERR_INVALID;
  if (misaligned(x) || misaligned(packed) || misaligned(sf)) return MOE_ERR_INVALID;
  return status_of(launch_quantize(x, k, T * k, E, H, *groups, layout, packed, sf, stream));
}

int moe_route_gather_quantize(const int32_t* topk_ids, int T, int k, int E, const uint16_t* x, int H,
                              const moe_groups_t* groups, uint8_t* packed, uint8_t* sf, cudaStream_t stream) {
  if (!groups_ok(groups) || T < 0 || k < 0 || k > kMaxTopK || H <= 0 || E <= 0 || E > kMaxExperts)
    return MOE_ERR_INVALID;
  if (H % 64) return MOE_ERR_SHAPE;
  if ((long long)T * k > (1LL << 30)) return MOE_ERR_INVALID;
  const int S = T * k;
  if (S == 0) return status_of(launch_route(topk_ids, 0, E, *groups, stream));
  if (!topk_ids || !x || !packed || !sf) return MOE_ERR_INVALID;
  if (misaligned(x) || misaligned(packed) || misaligned(sf)) return MOE_ERR_INVALID;
  if (S <= kSmallRouteSlots)
    return status_of(launch_route_quantize_small(topk_ids, S, E, *groups, nullptr, 0, x, k, H, packed, sf, stream));
  cudaError_t err = launch_route(topk_ids, S, E, *groups, stream);
  if (err == cudaSuccess) err = launch_quantize(x, k, S, E, H, *groups, MOE_SF_CHUNK32, packed, sf, stream);
  return status_of(err);
}

int nvfp4_grouped_gemm(const uint8_t* a_packed, const uint8_t* a_sf, int a_sf_layout, const moe_groups_t* groups,
                       int R_max, const uint8_t* w_tiled, int w_interleaved, int E, int N, int K, float* d,
                       cudaStream_t stream) {
  if (!groups_ok(groups) || R_max < 0 || E <= 0 || N <= 0 || K <= 0 || !layout_ok(a_sf_layout))
    return MOE_ERR_INVALID;
  if (N % 128 || K % 64 || (w_interleaved && N % 256)) return MOE_ERR_SHAPE;
  if ((long long)E * N > (1LL << 31)) return MOE_ERR_SHAPE;
  if (R_max == 0) return MOE_OK;
  if (!a_packed || !a_sf || !w_tiled || !d) return MOE_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(a_packed) % 16 || reinterpret_cast<uintptr_t>(w_tiled) % 16 ||
      reinterpret_cast<uintptr_t>(a_sf) % 16)
    return MOE_ERR_INVALID;
  int* st = status_ptr();
  if (!st) return MOE_ERR_CUDA;
  const GemmJob job{a_packed, a_sf, w_tiled, w_interleaved != 0, N, K, d};
  return status_of(
      launch_grouped_gemm(*groups, R_max, E, a_sf_layout, job, nullptr, nullptr, nullptr, nullptr, false, st, stream));
}

int nvfp4_grouped_gemm_swiglu(const uint8_t* a_packed, const uint8_t* a_sf, int a_sf_layout,
                              const moe_groups_t* groups, int R_max, const uint8_t* w13_tiled, int E, int I, int K,
                              const float* g_gate_up, uint8_t* h_packed, uint8_t* h_sf, cudaStream_t stream) {
  if (!groups_ok(groups) || R_max < 0 || E <= 0 || I <= 0 || K <= 0 || !layout_ok(a_sf_layout))
    return MOE_ERR_INVALID;
  if (I % 128 || K % 64) return MOE_ERR_SHAPE;
  if ((long long)E * 2 * I > (1LL << 31)) return MOE_ERR_SHAPE;
  if (R_max == 0) return MOE_OK;
  if (!a_packed || !a_sf || !w13_tiled || !g_gate_up || !h_packed || !h_sf) return MOE_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(a_packed) % 16 || reinterpret_cast<uintptr_t>(w13_tiled) % 16 ||
      reinterpret_cast<uintptr_t>(a_sf) % 16 || reinterpret_cast<uintptr_t>(h_packed) % 16 ||
      reinterpret_cast<uintptr_t>(h_sf) % 16)
    return MOE_ERR_INVALID;
  int* st = status_ptr();
  if (!st) return MOE_ERR_CUDA;
  const SwigluOut out{h_packed, h_sf, g_gate_up};
  const GemmJob job{a_packed, a_sf, w13_tiled, true, 2 * I, K, nullptr};
  return status_of(
      launch_grouped_gemm(*groups, R_max, E, a_sf_layout, job, &out, nullptr, nullptr, nullptr, false, st, stream));
}

size_t moe_expert_gemms_gate_bytes(int R_max, int E, int I) {
  if (R_max < 0 || E <= 0 || I <= 0) return 0;
  return (size_t)gate_ints(R_max, E, I) * sizeof(int);
}

int nvfp4_moe_expert_gemms(const uint8_t* x_packed, const uint8_t* x_sf, int sf_layout, const moe_groups_t* groups,
                           int R_max, const moe_nvfp4_weights_t* w, int H, int I, uint8_t* h_packed, uint8_t* h_sf,
                           float* d2, void* gate, cudaStream_t stream) {
  if (!w || !groups_ok(groups) || R_max < 0 || H <= 0 || I <= 0 || w->E <= 0 || w->E > kMaxExperts ||
      !layout_ok(sf_layout))
    return MOE_ERR_INVALID;
  if (H % 128 || I % 128) return MOE_ERR_SHAPE;
  if ((long long)w->E * 2 * I > (1LL << 31)) return MOE_ERR_SHAPE;
  if (R_max == 0) return MOE_OK;
  if (!x_packed || !x_sf || !w->w13_tiled || !w->g_gate_up || !w->w2_tiled || !h_packed || !h_sf || !d2 || !gate)
    return MOE_ERR_INVALID;
  if (misaligned(x_packed) || misaligned(x_sf) || misaligned(w->w13_tiled) || misaligned(w->w2_tiled) ||
      misaligned(h_packed) || misaligned(h_sf) || misaligned(d2) || misaligned(gate))
    return MOE_ERR_INVALID;
  int* st = status_ptr();
  if (!st) return MOE_ERR_CUDA;
  const int E = w->E;
  const SwigluOut swiglu{h_packed, h_sf, w->g_gate_up};
  const GemmJob w13{x_packed, x_sf, w->w13_tiled, true, 2 * I, H, nullptr};
  const GemmJob w2{h_packed, h_sf, w->w2_tiled, false, H, I, d2};
  return status_of(
      launch_grouped_gemm(*groups, R_max, E, sf_layout, w13, &swiglu, &w2, static_cast<int*>(gate), nullptr, false,
                          st, stream));
}

int swiglu_grouped(const float* d13, int R_max, int I, int E, const moe_groups_t* groups, const float* g_gate_up,
                   uint16_t* h, cudaStream_t stream) {
  if (!groups_ok(groups) || R_max < 0 || I <= 0 || E <= 0 || E > kMaxExperts) return MOE_ERR_INVALID;
  if (I % 64) return MOE_ERR_SHAPE;
  if (R_max == 0) return MOE_OK;
  if (!d13 || !g_gate_up || !h) return MOE_ERR_INVALID;
  if (misaligned(d13) || misaligned(h)) return MOE_ERR_INVALID;
  return status_of(launch_swiglu(d13, R_max, E, I, *groups, MOE_SF_CHUNK32, g_gate_up, h, nullptr, nullptr, stream));
}

int swiglu_quantize_grouped(const float* d13, int R_max, int I, int E, const moe_groups_t* groups, int layout,
                            const float* g_gate_up, uint8_t* packed, uint8_t* sf, cudaStream_t stream) {
  if (!groups_ok(groups) || R_max < 0 || I <= 0 || E <= 0 || E > kMaxExperts || !layout_ok(layout))
    return MOE_ERR_INVALID;
  if (I % 64) return MOE_ERR_SHAPE;
  if (R_max == 0) return MOE_OK;
  if (!d13 || !g_gate_up || !packed || !sf) return MOE_ERR_INVALID;
  if (misaligned(d13) || misaligned(packed) || misaligned(sf)) return MOE_ERR_INVALID;
  return status_of(launch_swiglu(d13, R_max, E, I, *groups, layout, g_gate_up, nullptr, packed, sf, stream));
}

int moe_scatter_add(const float* d2, int H, const int32_t* topk_ids, const float* topk_w, int T, int k, int E,
                    const moe_groups_t* groups, const float* g_down, uint16_t* y, cudaStream_t stream) {
  if (!groups_ok(groups) || T < 0 || k < 0 || k > kMaxTopK || E <= 0 || H <= 0) return MOE_ERR_INVALID;
  if (H % 4) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!y || (k > 0 && (!d2 || !topk_ids || !topk_w || !g_down))) return MOE_ERR_INVALID;
  if (misaligned(d2) || misaligned(y)) return MOE_ERR_INVALID;
  if (k == 0) return status_of(cudaMemsetAsync(y, 0, (size_t)T * H * sizeof(uint16_t), stream));
  return status_of(launch_scatter(d2, H, topk_ids, topk_w, T, k, E, *groups, g_down, y, stream));
}

size_t moe_nvfp4_layer_workspace_size(int T, int k, int E, int H, int I) {
  if (T < 0 || k < 0 || E <= 0 || H <= 0 || I <= 0) return 0;
  return carve_layer(nullptr, T, k, E, H, I).bytes;
}

int moe_nvfp4_layer_sf_layout(int T, int k, int E) {
  if (T < 0 || k < 0 || E <= 0) return MOE_SF_CHUNK32;
  return layer_sf_layout((long long)T * k, E);
}

int moe_nvfp4_layer(const uint16_t* x, int T, int H, int I, const int32_t* topk_ids, const float* topk_w, int k,
                    const moe_nvfp4_weights_t* w, void* workspace, size_t ws_bytes, uint16_t* y,
                    cudaStream_t stream) {
  const int arg_status = layer_arg_status(x, T, H, I, topk_ids, topk_w, k, w, y);
  if (arg_status != MOE_OK) return arg_status;
  if (T == 0) return MOE_OK;
  if (k == 0) return status_of(cudaMemsetAsync(y, 0, (size_t)T * H * sizeof(uint16_t), stream));
  const int E = w->E;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256) return MOE_ERR_INVALID;
  const LayerWs ws = carve_layer(workspace, T, k, E, H, I);
  if (ws_bytes < ws.bytes) return MOE_ERR_WORKSPACE;
  int* st = status_ptr();
  if (!st) return MOE_ERR_CUDA;
  const int S = T * k;
  // a1-a3: decode-sized batches (T*k <= 32) in one launch (route + gather + quantize), else
  // route, then gather+quantize; either clears the GEMM launch's work counters. The GEMM
  // launch starts on weights before the previous kernel ends: with a group table two launches
  // old it claims units and streams them (early); for decode-sized batches it routes the
  // slots itself from topk_ids and issues its first unit's first weight stages while it waits.
  // Token blocks (and scale layout): 128 rows for prefill-sized batches, else 32.
  const bool small = S <= kSmallRouteSlots;
  const int layout = layer_sf_layout(S, E);
  cudaError_t err;
  if (small) {
    err = launch_route_quantize_small(topk_ids, S, E, ws.groups, ws.gate, ws.ngate, x, k, H, ws.xq, ws.xsf, stream);
  } else {
    // each token row read and quantized once, written to all of its routed rows
    err = launch_route(topk_ids, S, E, ws.groups, stream, ws.gate, ws.ngate, ws.slot_sf,
                       layout == MOE_SF_ATOM128 ? 128 : 32);
    if (err == cudaSuccess)
      err = launch_quantize_tokens(x, T, H, k, ws.groups, ws.slot_sf, layout, ws.xq, ws.xsf, stream);
  }
  const SmallFront front{topk_ids, S};
  // a4 + a5 + a6 (w13 with SwiGLU and requantization in its epilogue) and a7
  // (w2) in one persistent launch; a w2 unit starts once its chunk's h is in
  const SwigluOut swiglu{ws.hq, ws.hsf, w->g_gate_up};
  const GemmJob w13{ws.xq, ws.xsf, w->w13_tiled, true, 2 * I, H, nullptr};
  const GemmJob w2{ws.hq, ws.hsf, w->w2_tiled, false, H, I, ws.d2};
  if (err == cudaSuccess)
    err = launch_grouped_gemm(ws.groups, S, E, layout, w13, &swiglu, &w2, ws.gate, small ? &front : nullptr, !small,
                              st, stream);
  if (err == cudaSuccess)  // its routing tables are two or more launches old
    err = launch_scatter(ws.d2, H, topk_ids, topk_w, T, k, E, ws.groups, w->g_down, y, stream, true);
  return status_of(err);
}

int nvfp4_grouped_gemv_w4a16(const uint16_t* a, int src_k, const moe_groups_t* groups, int R_max,
                             const uint8_t* w_tiled, int w_interleaved, int E, int N, int K, float* d,
                             cudaStream_t stream) {
  if (!groups_ok(groups) || R_max < 0 || E <= 0 || N <= 0 || K <= 0 || src_k < 0 || src_k > kMaxTopK)
    return MOE_ERR_INVALID;
  if (N % 128 || K % 64 || K > kGemvMaxK || (w_interleaved && N % 256)) return MOE_ERR_SHAPE;
  if ((long long)E * N > (1LL << 31)) return MOE_ERR_SHAPE;
  if (R_max == 0) return MOE_OK;
  if (!a || !w_tiled || !d) return MOE_ERR_INVALID;
  if (misaligned(a) || misaligned(w_tiled) || misaligned(d)) return MOE_ERR_INVALID;
  return status_of(launch_gemv_w4a16(a, src_k, R_max, E, *groups, w_tiled, w_interleaved != 0, N, K, d, stream));
}

size_t moe_nvfp4_layer_w4a16_workspace_size(int T, int k, int E, int H, int I) {
  if (T < 0 || k < 0 || E <= 0 || H <= 0 || I <= 0) return 0;
  return carve_layer_w4a16(nullptr, T, k, E, H, I).bytes;
}

int moe_nvfp4_layer_w4a16(const uint16_t* x, int T, int H, int I, const int32_t* topk_ids, const float* topk_w,
                          int k, const moe_nvfp4_weights_t* w, void* workspace, size_t ws_bytes, uint16_t* y,
                          cudaStream_t stream) {
  if (!w || T < 0 || k < 0 || k > kMaxTopK || H <= 0 || I <= 0 || w->E <= 0 || w->E > kMaxExperts)
    return MOE_ERR_INVALID;
  if (H % 128 || I % 128 || H > kGemvMaxK || I > kGemvMaxK) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!x || !y || (k > 0 && (!topk_ids || !topk_w))) return MOE_ERR_INVALID;
  if (misaligned(x) || misaligned(y)) return MOE_ERR_INVALID;
  if (!w->w13_tiled || !w->g_gate_up || !w->w2_tiled || !w->g_down) return MOE_ERR_INVALID;
  if (misaligned(w->w13_tiled) || misaligned(w->w2_tiled)) return MOE_ERR_INVALID;
  if ((long long)T * k > (1LL << 30) || (long long)w->E * 2 * I > (1LL << 31)) return MOE_ERR_SHAPE;
  if (k == 0) return status_of(cudaMemsetAsync(y, 0, (size_t)T * H * sizeof(uint16_t), stream));
  const int E = w->E, S = T * k;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256) return MOE_ERR_INVALID;
  const GemvWs ws = carve_layer_w4a16(workspace, T, k, E, H, I);
  if (ws_bytes < ws.bytes) return MOE_ERR_WORKSPACE;
  // a1 route; a2+a4 gather and w13 GEMV on the exact bf16 rows; a5 SwiGLU to
  // bf16 h (no requantization); a7 w2 GEMV on h; a8 scatter-add
  cudaError_t err = launch_route(topk_ids, S, E, ws.groups, stream);
  if (err == cudaSuccess)
    err = launch_gemv_w4a16(x, k, S, E, ws.groups, w->w13_tiled, true, 2 * I, H, ws.d13, stream);
  if (err == cudaSuccess)
    err = launch_swiglu(ws.d13, S, E, I, ws.groups, MOE_SF_CHUNK32, w->g_gate_up, ws.h, nullptr, nullptr, stream);
  if (err == cudaSuccess) err = launch_gemv_w4a16(ws.h, 0, S, E, ws.groups, w->w2_tiled, false, H, I, ws.d2, stream);
  if (err == cudaSuccess)  // its routing tables are two or more launches old
    err = launch_scatter(ws.d2, H, topk_ids, topk_w, T, k, E, ws.groups, w->g_down, y, stream, true);
  return status_of(err);
}

size_t nvfp4_tiled_bytes(int rows, int K) {
  if (rows < 0 || K <= 0) return 0;
  return tiled_bytes(rows, K);
}

int nvfp4_tile_weights(const uint8_t* packed, const uint8_t* sf_linear, int rows, int K, int interleave_rows,
                       uint8_t* tiled, cudaStream_t stream) {
  if (rows < 0 || K <= 0 || interleave_rows < 0) return MOE_ERR_INVALID;
  if (rows % 128 || K % 64) return MOE_ERR_SHAPE;
  if (interleave_rows > 0 && (interleave_rows % 256 || rows % interleave_rows)) return MOE_ERR_SHAPE;
  if (rows == 0) return MOE_OK;
  if (!packed || !sf_linear || !tiled) return MOE_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(packed) % 16 || reinterpret_cast<uintptr_t>(sf_linear) % 4 ||
      reinterpret_cast<uintptr_t>(tiled) % 16)
    return MOE_ERR_INVALID;
  return status_of(launch_tile(packed, sf_linear, rows, K, interleave_rows, tiled, stream));
}

int nvfp4_swizzle_block_scales(const uint8_t* linear, int N, int K, uint8_t* swizzled, cudaStream_t stream) {
  if (N < 0 || K <= 0) return MOE_ERR_INVALID;
  if (K % 64) return MOE_ERR_SHAPE;
  if (N == 0) return MOE_OK;
  if (!linear || !swizzled) return MOE_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(linear) % 4 || reinterpret_cast<uintptr_t>(swizzled) % 4) return MOE_ERR_INVALID;
  return status_of(launch_swizzle(linear, N, K, swizzled, stream));
}

}  // extern "C"
