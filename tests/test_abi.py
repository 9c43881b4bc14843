"""The C ABI without a GPU: the library builds and loads, exports every entry
point the header declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

from nvfp4_block_scaled_gather_gb300 import _native
from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe_nvfp4.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)


def test_header_declares_the_hot_path():
    names = set(declared_functions())
    for n in ("moe_gather_rows", "nvfp4_quantize_rows", "nvfp4_grouped_gemm", "swiglu_grouped",
              "moe_scatter_add", "moe_nvfp4_layer", "moe_nvfp4_layer_workspace_size",
              "nvfp4_swizzle_block_scales", "moe_route_groups", "nvfp4_grouped_gemv_w4a16",
              "moe_nvfp4_layer_w4a16", "moe_nvfp4_layer_w4a16_workspace_size"):
        assert n in names, n


def test_library_exports_every_declared_symbol(native):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(native, n), n
    assert set(names) == set(_native.exported_symbols())


def test_error_strings(native):
    for code in range(6):
        assert native.moe_nvfp4_error_string(code)
    assert native.moe_nvfp4_error_string(0) == b"ok"


def _fake_groups():
    g = _native.MoeGroups()
    for name, _ in g._fields_:
        setattr(g, name, 4096)
    return g


def test_host_side_validation(native):
    g = _fake_groups()
    s = None
    # unsupported GEMM shapes
    assert native.nvfp4_grouped_gemm(16, 16, 1, ctypes.byref(g), 8, 16, 0, 4, 100, 256, 16, s) == 2
    assert native.nvfp4_grouped_gemm(16, 16, 1, ctypes.byref(g), 8, 16, 0, 4, 128, 96, 16, s) == 2
    assert native.nvfp4_grouped_gemm(16, 16, 1, ctypes.byref(g), 8, 16, 1, 4, 384, 256, 16, s) == 2
    assert native.nvfp4_grouped_gemm_swiglu(16, 16, 1, ctypes.byref(g), 8, 16, 4, 192, 256, 16, 16, 16, s) == 2
    # token-scale layout must be one of the two
    assert native.nvfp4_grouped_gemm(16, 16, 2, ctypes.byref(g), 8, 16, 0, 4, 128, 256, 16, s) == 1
    assert native.nvfp4_grouped_gemm_swiglu(16, 16, -1, ctypes.byref(g), 8, 16, 4, 128, 256, 16, 16, 16, s) == 1
    # missing group arrays / bad sizes / misaligned weights
    assert native.nvfp4_grouped_gemm(16, 16, 1, None, 8, 16, 0, 4, 128, 256, 16, s) == 1
    assert native.nvfp4_grouped_gemm(16, 16, 1, ctypes.byref(g), 8, 24, 0, 4, 128, 256, 16, s) == 1
    assert native.nvfp4_quantize_rows(16, 8, 100, 4, ctypes.byref(g), 1, 16, 16, s) == 2
    assert native.nvfp4_quantize_rows(16, 8, 128, 0, ctypes.byref(g), 1, 16, 16, s) == 1
    assert native.nvfp4_quantize_rows(16, 8, 128, 4, ctypes.byref(g), 7, 16, 16, s) == 1
    assert native.nvfp4_tile_weights(16, 16, 100, 128, 0, 16, s) == 2
    assert native.nvfp4_tile_weights(16, 16, 128, 96, 0, 16, s) == 2
    assert native.nvfp4_tile_weights(16, 16, 384, 128, 384, 16, s) == 2
    assert native.moe_route_groups(16, 2, 2, 2000, ctypes.byref(g), s) == 1
    assert native.moe_route_groups(16, 2, 40, 8, ctypes.byref(g), s) == 1
    assert native.moe_scatter_add(16, 256, 16, 16, 2, 2, -1, ctypes.byref(g), 16, 16, s) == 1
    # device buffers must be 16-byte aligned
    assert native.moe_scatter_add(24, 256, 16, 16, 2, 2, 8, ctypes.byref(g), 16, 16, s) == 1
    assert native.moe_scatter_add(16, 256, 16, 16, 2, 2, 8, ctypes.byref(g), 16, 40, s) == 1
    assert native.nvfp4_quantize_rows(24, 8, 128, 4, ctypes.byref(g), 1, 16, 16, s) == 1
    assert native.swiglu_grouped(16, 8, 128, 4, ctypes.byref(g), 16, 8, s) == 1
    w = _native.MoeWeights(8, 16, 16, 16, 16)
    assert native.moe_nvfp4_layer(16, 4, 200, 128, 16, 16, 2, ctypes.byref(w), 256, 1 << 20, 16, s) == 2
    assert native.moe_nvfp4_layer(16, 4, 256, 96, 16, 16, 2, ctypes.byref(w), 256, 1 << 20, 16, s) == 2
    assert native.moe_nvfp4_layer(16, 4, 256, 128, 16, 16, 2, None, 256, 1 << 20, 16, s) == 1
    ws = native.moe_nvfp4_layer_workspace_size(4, 2, 8, 256, 128)
    assert native.moe_nvfp4_layer(16, 4, 256, 128, 16, 16, 2, ctypes.byref(w), 256, ws - 1, 16, s) == 5
    assert native.moe_nvfp4_layer(16, 4, 256, 128, 16, 16, 2, ctypes.byref(w), 300, ws, 16, s) == 1
    # the allocation-free entry checks its arguments like moe_nvfp4_layer, before its size limit:
    # a batch far beyond the scratch array still gets the shape / argument error first
    assert native.moe_nvfp4_layer_static(16, 4096, 200, 128, 16, 16, 8, ctypes.byref(w), 16, s) == 2
    assert native.moe_nvfp4_layer_static(16, 4096, 256, 96, 16, 16, 8, ctypes.byref(w), 16, s) == 2
    assert native.moe_nvfp4_layer_static(16, 4096, 256, 128, 16, 16, 33, ctypes.byref(w), 16, s) == 1
    assert native.moe_nvfp4_layer_static(16, 4096, 256, 128, 16, 16, 8, None, 16, s) == 1
    assert native.moe_nvfp4_layer_static(24, 4096, 256, 128, 16, 16, 8, ctypes.byref(w), 16, s) == 1
    assert native.moe_nvfp4_layer_static(16, 4096, 256, 128, 16, 16, 8, ctypes.byref(w), 16, s) == 5
    # the GEMV path: shapes (N % 128, K % 64, K <= 14336, interleaved N % 256), alignment, src_k
    assert native.nvfp4_grouped_gemv_w4a16(16, 2, ctypes.byref(g), 8, 16, 0, 4, 100, 256, 16, s) == 2
    assert native.nvfp4_grouped_gemv_w4a16(16, 2, ctypes.byref(g), 8, 16, 0, 4, 128, 96, 16, s) == 2
    assert native.nvfp4_grouped_gemv_w4a16(16, 2, ctypes.byref(g), 8, 16, 0, 4, 128, 14400, 16, s) == 2
    assert native.nvfp4_grouped_gemv_w4a16(16, 2, ctypes.byref(g), 8, 16, 1, 4, 384, 256, 16, s) == 2
    assert native.nvfp4_grouped_gemv_w4a16(24, 2, ctypes.byref(g), 8, 16, 0, 4, 128, 256, 16, s) == 1
    assert native.nvfp4_grouped_gemv_w4a16(16, -1, ctypes.byref(g), 8, 16, 0, 4, 128, 256, 16, s) == 1
    assert native.nvfp4_grouped_gemv_w4a16(16, 2, None, 8, 16, 0, 4, 128, 256, 16, s) == 1
    assert native.moe_nvfp4_layer_w4a16(16, 4, 200, 128, 16, 16, 2, ctypes.byref(w), 256, 1 << 20, 16, s) == 2
    assert native.moe_nvfp4_layer_w4a16(16, 4, 16384, 128, 16, 16, 2, ctypes.byref(w), 256, 1 << 20, 16, s) == 2
    ws16 = native.moe_nvfp4_layer_w4a16_workspace_size(4, 2, 8, 256, 128)
    assert ws16 > 0
    assert native.moe_nvfp4_layer_w4a16(16, 4, 256, 128, 16, 16, 2, ctypes.byref(w), 256, ws16 - 1, 16, s) == 5
    assert native.moe_nvfp4_layer_w4a16(16, 4, 256, 128, 16, 16, 2, ctypes.byref(w), 300, ws16, 16, s) == 1
    # empty problems are no-ops
    assert native.moe_nvfp4_layer_w4a16(None, 0, 256, 128, None, None, 2, ctypes.byref(w), None, 0, None, s) == 0
    assert native.moe_nvfp4_layer(None, 0, 256, 128, None, None, 2, ctypes.byref(w), None, 0, None, s) == 0
    assert native.nvfp4_swizzle_block_scales(None, 0, 64, None, s) == 0


def test_sizes(native):
    # tiled weights: one 18 KB block per 128 rows and 256 K values, K padded up
    assert native.nvfp4_tiled_bytes(288 * 4096, 4096) == 288 * 4096 * 4096 * 9 // 16
    assert native.nvfp4_tiled_bytes(256, 128) == 2 * 18432
    assert native.moe_groups_bytes(1, 8, 288) > 0
    # token-scale region bounds: (min(E, R) + ceil(R / 128 or 32)) * 128 * K / 16
    assert native.nvfp4_sf_bytes(8, 288, 4096, 0) == (8 + 1) * 128 * 256
    assert native.nvfp4_sf_bytes(2304, 288, 2048, 0) == (288 + 18) * 128 * 128
    assert native.nvfp4_sf_bytes(2304, 288, 2048, 1) == (288 + 72) * 128 * 128
    assert native.nvfp4_sf_bytes(8, 288, 4096, 5) == 0
    small = native.moe_nvfp4_layer_workspace_size(1, 8, 288, 4096, 2048)
    big = native.moe_nvfp4_layer_workspace_size(288, 8, 288, 4096, 2048)
    assert 0 < small < big


def test_groups_carve_is_host_only(native):
    buf = ctypes.create_string_buffer(native.moe_groups_bytes(3, 2, 5) + 512)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    g = _native.MoeGroups()
    assert native.moe_groups_carve(base, 3, 2, 5, ctypes.byref(g)) == 0
    assert g.counts == base and g.slot_row > g.row_slot > g.group_offsets
    assert native.moe_groups_carve(base + 4, 3, 2, 5, ctypes.byref(g)) == 1


def test_layer_token_block_rule(native):
    """The layer's token blocks: 32-row chunks for decode-sized and mid-sized
    batches, 128-row blocks once the batch routes 16 rows per expert on
    average (T*k >= 16*E), never for the one-launch decode front end."""
    assert native.moe_nvfp4_layer_sf_layout(1, 8, 288) == 1
    assert native.moe_nvfp4_layer_sf_layout(32, 8, 288) == 1
    assert native.moe_nvfp4_layer_sf_layout(288, 8, 288) == 1         # ~2300 rows, mean 8 per expert
    assert native.moe_nvfp4_layer_sf_layout(576, 8, 288) == 0         # mean 16 per expert
    assert native.moe_nvfp4_layer_sf_layout(1152, 8, 288) == 0        # prefill-sized, mean 32
    assert native.moe_nvfp4_layer_sf_layout(4, 8, 1) == 1             # decode front end (T*k <= 32)
    assert native.moe_nvfp4_layer_sf_layout(160, 2, 6) == 0
