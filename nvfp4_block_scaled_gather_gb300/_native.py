"""ctypes binding of libmoe_nvfp4.so (include/moe_nvfp4.h).

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are torch CUDA tensors (device memory and streams only); calls are
enqueued on the current torch stream. A nonzero status raises RuntimeError.
There is no fallback: if the library cannot be built or loaded, load()
raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

_LIB = None

c_int, c_size_t, c_void_p = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p

# token-scale layouts (include/moe_nvfp4.h)
SF_ATOM128 = 0   # per group, 128-row atoms, zero-padded (the pages' CUTLASS layout)
SF_CHUNK32 = 1   # per 32-row chunk, the layout nvfp4_grouped_gemm reads


class MoeGroups(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("counts", "group_offsets", "group_expert", "group_sf_block",
                                       "group_chunk", "chunk_info", "block_info", "row_slot", "slot_row")]


class MoeWeights(ctypes.Structure):
    _fields_ = [("E", c_int), ("w13_tiled", c_void_p), ("g_gate_up", c_void_p), ("w2_tiled", c_void_p),
                ("g_down", c_void_p)]


_SIGS = {
    "moe_nvfp4_error_string": (ctypes.c_char_p, [c_int]),
    "moe_nvfp4_check_status": (c_int, [c_void_p]),
    "moe_groups_bytes": (c_size_t, [c_int, c_int, c_int]),
    "moe_groups_carve": (c_int, [c_void_p, c_int, c_int, c_int, ctypes.POINTER(MoeGroups)]),
    "nvfp4_sf_bytes": (c_size_t, [c_int, c_int, c_int, c_int]),
    "moe_route_groups": (c_int, [c_void_p, c_int, c_int, c_int, ctypes.POINTER(MoeGroups), c_void_p]),
    "moe_gather_rows": (c_int, [c_void_p, c_int, c_int, c_void_p, c_int, c_int, ctypes.POINTER(MoeGroups),
                                c_void_p, c_void_p]),
    "nvfp4_quantize_rows": (c_int, [c_void_p, c_int, c_int, c_int, ctypes.POINTER(MoeGroups), c_int, c_void_p,
                                    c_void_p, c_void_p]),
    "moe_gather_quantize_rows": (c_int, [c_void_p, c_int, c_int, c_int, c_int, ctypes.POINTER(MoeGroups), c_int,
                                         c_void_p, c_void_p, c_void_p]),
    "nvfp4_grouped_gemm": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MoeGroups), c_int, c_void_p, c_int,
                                   c_int, c_int, c_int, c_void_p, c_void_p]),
    "nvfp4_grouped_gemm_swiglu": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MoeGroups), c_int, c_void_p,
                                          c_int, c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_route_gather_quantize": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_int, ctypes.POINTER(MoeGroups),
                                          c_void_p, c_void_p, c_void_p]),
    "moe_expert_gemms_gate_bytes": (ctypes.c_size_t, [c_int, c_int, c_int]),
    "nvfp4_moe_expert_gemms": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MoeGroups), c_int,
                                       ctypes.POINTER(MoeWeights), c_int, c_int, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p]),
    "swiglu_grouped": (c_int, [c_void_p, c_int, c_int, c_int, ctypes.POINTER(MoeGroups), c_void_p, c_void_p,
                               c_void_p]),
    "swiglu_quantize_grouped": (c_int, [c_void_p, c_int, c_int, c_int, ctypes.POINTER(MoeGroups), c_int,
                                        c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_scatter_add": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_int,
                                ctypes.POINTER(MoeGroups), c_void_p, c_void_p, c_void_p]),
    "moe_nvfp4_layer_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "moe_nvfp4_layer_sf_layout": (c_int, [c_int, c_int, c_int]),
    "moe_nvfp4_layer": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_int,
                                ctypes.POINTER(MoeWeights), c_void_p, c_size_t, c_void_p, c_void_p]),
    "nvfp4_swizzle_block_scales": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p]),
    "moe_nvfp4_layer_static": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_int,
                                       ctypes.POINTER(MoeWeights), c_void_p, c_void_p]),
    "nvfp4_grouped_gemv_w4a16": (c_int, [c_void_p, c_int, ctypes.POINTER(MoeGroups), c_int, c_void_p, c_int, c_int,
                                         c_int, c_int, c_void_p, c_void_p]),
    "moe_nvfp4_layer_w4a16_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "moe_nvfp4_layer_w4a16": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_int,
                                      ctypes.POINTER(MoeWeights), c_void_p, c_size_t, c_void_p, c_void_p]),
    "nvfp4_tiled_bytes": (c_size_t, [c_int, c_int]),
    "nvfp4_tile_weights": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p]),
}


def load():
    """Builds (if stale) and loads the library; raises if either fails."""
    global _LIB
    if _LIB is None:
        path = _build.ensure_built()
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _LIB = lib
    return _LIB


def library_path() -> str:
    return _build.LIB


def exported_symbols():
    return list(_SIGS)


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(name, status):
    if status != 0:
        msg = load().moe_nvfp4_error_string(status).decode()
        raise RuntimeError(f"{name} failed: {msg} (status {status})")


class Groups:
    """Device buffer holding the group metadata of T tokens, top-k, E experts,
    with torch views of its arrays for inspection."""

    def __init__(self, T: int, k: int, E: int, device="cuda"):
        import torch
        lib = load()
        self.T, self.k, self.E = T, k, E
        nbytes = lib.moe_groups_bytes(T, k, E)
        self.buffer = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        self.struct = MoeGroups()
        _check("moe_groups_carve", lib.moe_groups_carve(_ptr(self.buffer), T, k, E, ctypes.byref(self.struct)))

    def view(self, name: str, n: int):
        import torch
        off = getattr(self.struct, name) - self.buffer.data_ptr()
        return self.buffer[off:off + 4 * n].view(torch.int32)

    def host(self) -> dict:
        """Copies the metadata to the host (synchronizes)."""
        counts = self.view("counts", 5).cpu()
        G, R, maxmg, nblk, nchunk = (int(v) for v in counts)
        S = self.T * self.k
        return dict(G=G, R=R, max_mg=maxmg, blocks=nblk, chunks=nchunk,
                    group_offsets=self.view("group_offsets", G + 1).cpu(),
                    group_expert=self.view("group_expert", G).cpu(),
                    group_sf_block=self.view("group_sf_block", G + 1).cpu(),
                    group_chunk=self.view("group_chunk", G + 1).cpu(),
                    chunk_info=self.view("chunk_info", 4 * nchunk).cpu().reshape(-1, 4),
                    block_info=self.view("block_info", 4 * nblk).cpu().reshape(-1, 4),
                    row_slot=self.view("row_slot", R).cpu(),
                    slot_row=self.view("slot_row", S).cpu())


def sf_bytes(R_max: int, E: int, K: int, layout: int = SF_CHUNK32) -> int:
    return load().nvfp4_sf_bytes(R_max, E, K, layout)


def check_status(stream=None) -> int:
    return load().moe_nvfp4_check_status(_stream(stream))


def moe_route_groups(topk_ids, E: int, groups: Groups, stream=None):
    T, k = topk_ids.shape
    _check("moe_route_groups", load().moe_route_groups(_ptr(topk_ids), T, k, E, ctypes.byref(groups.struct),
                                                       _stream(stream)))


def moe_gather_rows(x, topk_ids, E: int, groups: Groups, xg, stream=None):
    T, H = x.shape
    k = topk_ids.shape[1]
    _check("moe_gather_rows", load().moe_gather_rows(_ptr(x), T, H, _ptr(topk_ids), k, E,
                                                     ctypes.byref(groups.struct), _ptr(xg), _stream(stream)))


def nvfp4_quantize_rows(rows, groups: Groups, packed, sf, layout: int = SF_CHUNK32, stream=None):
    R, K = rows.shape
    _check("nvfp4_quantize_rows", load().nvfp4_quantize_rows(_ptr(rows), R, K, groups.E,
                                                             ctypes.byref(groups.struct), layout, _ptr(packed),
                                                             _ptr(sf), _stream(stream)))


def moe_gather_quantize_rows(x, k: int, groups: Groups, packed, sf, layout: int = SF_CHUNK32, stream=None):
    T, H = x.shape
    _check("moe_gather_quantize_rows",
           load().moe_gather_quantize_rows(_ptr(x), T, H, k, groups.E, ctypes.byref(groups.struct), layout,
                                           _ptr(packed), _ptr(sf), _stream(stream)))


class TiledWeight:
    """One projection of all experts, [E, N, K], tiled for the grouped GEMM.
    interleave=True pairs rows of the two halves of N in every tile (the w13
    gate|up layout the fused SwiGLU epilogue reads)."""

    def __init__(self, packed, sf_linear, interleave: bool = False, stream=None):
        import torch
        self.E, self.N, K2 = packed.shape
        self.K = 2 * K2
        self.interleaved = interleave
        rows = self.E * self.N
        self.data = torch.empty(load().nvfp4_tiled_bytes(rows, self.K), dtype=torch.uint8, device=packed.device)
        _check("nvfp4_tile_weights",
               load().nvfp4_tile_weights(_ptr(packed.contiguous()), _ptr(sf_linear.contiguous()), rows, self.K,
                                         self.N if interleave else 0, _ptr(self.data), _stream(stream)))


def nvfp4_grouped_gemm(a_packed, a_sf, groups: Groups, w: TiledWeight, d, layout: int = SF_CHUNK32, stream=None):
    """a_sf in `layout`: the token block size the GEMM works in (32 or 128 rows)."""
    R_max = a_packed.shape[0]
    K = a_packed.shape[1] * 2
    assert K == w.K
    _check("nvfp4_grouped_gemm",
           load().nvfp4_grouped_gemm(_ptr(a_packed), _ptr(a_sf), layout, ctypes.byref(groups.struct), R_max,
                                     _ptr(w.data), int(w.interleaved), w.E, w.N, K, _ptr(d), _stream(stream)))


def nvfp4_grouped_gemm_swiglu(a_packed, a_sf, groups: Groups, w13: TiledWeight, g_gate_up, h_packed, h_sf,
                              layout: int = SF_CHUNK32, stream=None):
    R_max = a_packed.shape[0]
    K = a_packed.shape[1] * 2
    assert K == w13.K and w13.interleaved
    _check("nvfp4_grouped_gemm_swiglu",
           load().nvfp4_grouped_gemm_swiglu(_ptr(a_packed), _ptr(a_sf), layout, ctypes.byref(groups.struct), R_max,
                                            _ptr(w13.data), w13.E, w13.N // 2, K, _ptr(g_gate_up), _ptr(h_packed),
                                            _ptr(h_sf), _stream(stream)))


def moe_route_gather_quantize(topk_ids, x, E: int, groups: Groups, packed, sf, stream=None):
    """Route + gather + quantize (one launch for T*k <= 32), MOE_SF_CHUNK32 scales."""
    T, k = topk_ids.shape
    _check("moe_route_gather_quantize",
           load().moe_route_gather_quantize(_ptr(topk_ids), T, k, E, _ptr(x), x.shape[1],
                                            ctypes.byref(groups.struct), _ptr(packed), _ptr(sf), _stream(stream)))


def nvfp4_moe_expert_gemms(x_packed, x_sf, groups: Groups, W: "Weights", h_packed, h_sf, d2, gate,
                           layout: int = SF_CHUNK32, stream=None):
    """Both grouped GEMMs in one launch (w13 + SwiGLU + requantize, then w2);
    x_sf and h_sf in `layout`."""
    R_max = x_packed.shape[0]
    _check("nvfp4_moe_expert_gemms",
           load().nvfp4_moe_expert_gemms(_ptr(x_packed), _ptr(x_sf), layout, ctypes.byref(groups.struct), R_max,
                                         ctypes.byref(W.struct), W.H, W.I, _ptr(h_packed), _ptr(h_sf), _ptr(d2),
                                         _ptr(gate), _stream(stream)))


def expert_gemms_gate_bytes(R_max: int, E: int, I: int) -> int:
    return load().moe_expert_gemms_gate_bytes(R_max, E, I)


def swiglu_grouped(d13, groups: Groups, g_gate_up, h, stream=None):
    R_max, I2 = d13.shape
    _check("swiglu_grouped", load().swiglu_grouped(_ptr(d13), R_max, I2 // 2, groups.E, ctypes.byref(groups.struct),
                                                   _ptr(g_gate_up), _ptr(h), _stream(stream)))


def swiglu_quantize_grouped(d13, groups: Groups, g_gate_up, packed, sf, layout: int = SF_CHUNK32, stream=None):
    R_max, I2 = d13.shape
    _check("swiglu_quantize_grouped",
           load().swiglu_quantize_grouped(_ptr(d13), R_max, I2 // 2, groups.E, ctypes.byref(groups.struct), layout,
                                          _ptr(g_gate_up), _ptr(packed), _ptr(sf), _stream(stream)))


def moe_scatter_add(d2, topk_ids, topk_w, E: int, groups: Groups, g_down, y, stream=None):
    T, k = topk_ids.shape
    H = y.shape[1]
    _check("moe_scatter_add",
           load().moe_scatter_add(_ptr(d2), H, _ptr(topk_ids), _ptr(topk_w), T, k, E, ctypes.byref(groups.struct),
                                  _ptr(g_down), _ptr(y), _stream(stream)))


def nvfp4_swizzle_block_scales(linear, swizzled, stream=None):
    """linear [N, K/16] u8 -> swizzled (ceil(N/128)*128*K/16 bytes)."""
    N, Kc = linear.shape
    _check("nvfp4_swizzle_block_scales",
           load().nvfp4_swizzle_block_scales(_ptr(linear), N, Kc * 16, _ptr(swizzled), _stream(stream)))


def moe_nvfp4_layer_workspace_size(T: int, k: int, E: int, H: int, I: int) -> int:
    return load().moe_nvfp4_layer_workspace_size(T, k, E, H, I)


def layer_sf_layout(T: int, k: int, E: int) -> int:
    """The token-scale layout (token block size) moe_nvfp4_layer uses."""
    return load().moe_nvfp4_layer_sf_layout(T, k, E)


class Weights:
    """Device NVFP4 expert weights in the layout moe_nvfp4_layer reads.

    Built from packed nibbles, LINEAR block scales and globals; both
    projections are tiled for the grouped GEMM once here (load time, on the
    GPU). The inputs are not kept."""

    def __init__(self, w13_packed, w13_sf_linear, g_gate_up, w2_packed, w2_sf_linear, g_down, stream=None):
        import torch
        self.E, I2, H2 = w13_packed.shape
        self.H, self.I = H2 * 2, I2 // 2
        self.w13 = TiledWeight(w13_packed, w13_sf_linear, interleave=True, stream=stream)
        self.w2 = TiledWeight(w2_packed, w2_sf_linear, stream=stream)
        self.g_gate_up = g_gate_up.to(torch.float32).contiguous()
        self.g_down = g_down.to(torch.float32).contiguous()
        self.struct = MoeWeights(self.E, self.w13.data.data_ptr(), self.g_gate_up.data_ptr(),
                                 self.w2.data.data_ptr(), self.g_down.data_ptr())

    @property
    def nbytes(self) -> int:
        return self.w13.data.numel() + self.w2.data.numel()


def moe_nvfp4_layer(x, topk_ids, topk_w, weights: Weights, workspace, y, stream=None):
    T, H = x.shape
    k = topk_ids.shape[1]
    _check("moe_nvfp4_layer",
           load().moe_nvfp4_layer(_ptr(x), T, H, weights.I, _ptr(topk_ids), _ptr(topk_w), k,
                                  ctypes.byref(weights.struct), _ptr(workspace), workspace.numel(), _ptr(y),
                                  _stream(stream)))


def nvfp4_grouped_gemv_w4a16(a, groups: Groups, w: TiledWeight, d, src_k: int = 0, R_max: int = None, stream=None):
    """W4A16 grouped GEMV: bf16 rows a (gathered from token rows by slot when
    src_k > 0, else row r = a[r]) times the tiled NVFP4 weight, fp32 d."""
    K = a.shape[1]
    assert K == w.K
    if R_max is None:
        R_max = a.shape[0] * (src_k if src_k > 0 else 1)
    _check("nvfp4_grouped_gemv_w4a16",
           load().nvfp4_grouped_gemv_w4a16(_ptr(a), src_k, ctypes.byref(groups.struct), R_max, _ptr(w.data),
                                           int(w.interleaved), w.E, w.N, K, _ptr(d), _stream(stream)))


def moe_nvfp4_layer_w4a16_workspace_size(T: int, k: int, E: int, H: int, I: int) -> int:
    return load().moe_nvfp4_layer_w4a16_workspace_size(T, k, E, H, I)


def moe_nvfp4_layer_w4a16(x, topk_ids, topk_w, weights: Weights, workspace, y, stream=None):
    T, H = x.shape
    k = topk_ids.shape[1]
    _check("moe_nvfp4_layer_w4a16",
           load().moe_nvfp4_layer_w4a16(_ptr(x), T, H, weights.I, _ptr(topk_ids), _ptr(topk_w), k,
                                        ctypes.byref(weights.struct), _ptr(workspace), workspace.numel(), _ptr(y),
                                        _stream(stream)))


class MoeLayerW4A16:
    """The GEMV path (W4A16) of the step, with its own workspace for up to T_max tokens."""

    def __init__(self, weights: Weights, T_max: int, k: int):
        import torch
        self.weights, self.k, self.T_max = weights, k, T_max
        n = moe_nvfp4_layer_w4a16_workspace_size(T_max, k, weights.E, weights.H, weights.I)
        self.workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=weights.w13.data.device)

    def __call__(self, x, topk_ids, topk_w, y=None, stream=None):
        import torch
        assert x.shape[0] <= self.T_max and topk_ids.shape[1] == self.k
        if y is None:
            y = torch.empty_like(x)
        moe_nvfp4_layer_w4a16(x, topk_ids, topk_w, self.weights, self.workspace, y, stream)
        return y

    def capture(self, x, topk_ids, topk_w, y):
        """One GEMV-path step on these device buffers as a CUDA graph."""
        import torch
        self(x, topk_ids, topk_w, y)  # one-time lookups outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            moe_nvfp4_layer_w4a16(x, topk_ids, topk_w, self.weights, self.workspace, y)
        return graph


STATIC_SCRATCH_BYTES = 8 << 20  # MOE_NVFP4_STATIC_SCRATCH_BYTES


def moe_nvfp4_layer_static(x, topk_ids, topk_w, weights: Weights, y, stream=None):
    """The layer step with the library's own fixed scratch array instead of a
    caller workspace, for callers that may not allocate device memory. Calls
    that can overlap on the GPU share that array and must be serialized."""
    T, H = x.shape
    k = topk_ids.shape[1]
    _check("moe_nvfp4_layer_static",
           load().moe_nvfp4_layer_static(_ptr(x), T, H, weights.I, _ptr(topk_ids), _ptr(topk_w), k,
                                         ctypes.byref(weights.struct), _ptr(y), _stream(stream)))


class MoeLayer:
    """Holds the weights and a workspace sized for up to T_max tokens."""

    def __init__(self, weights: Weights, T_max: int, k: int):
        import torch
        self.weights, self.k, self.T_max = weights, k, T_max
        n = moe_nvfp4_layer_workspace_size(T_max, k, weights.E, weights.H, weights.I)
        # zeroed once: the step's work counters live here and every completed call leaves them zero
        self.workspace = torch.zeros(n, dtype=torch.uint8, device=weights.w13.data.device)

    def __call__(self, x, topk_ids, topk_w, y=None, stream=None):
        import torch
        assert x.shape[0] <= self.T_max and topk_ids.shape[1] == self.k
        if y is None:
            y = torch.empty_like(x)
        moe_nvfp4_layer(x, topk_ids, topk_w, self.weights, self.workspace, y, stream)
        return y

    def capture(self, x, topk_ids, topk_w, y):
        """Records one layer step on these device buffers as a CUDA graph (the
        buffers are baked into it; refill them and call .replay()). The first
        page's layer bench and verdict take the graph: it removes the host's
        per-launch cost, which matters when a step is tens of microseconds."""
        import torch
        self(x, topk_ids, topk_w, y)  # first call on the device does its one-time lookups outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            moe_nvfp4_layer(x, topk_ids, topk_w, self.weights, self.workspace, y)
        return graph
