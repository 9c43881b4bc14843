"""CPU oracle for the NVFP4 routed-expert MoE layer step (test infrastructure).

This module is the slow, plain definition the CUDA path is checked against.
Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
may import it; the product path never does. It shares no code with the CUDA
library and does not import it.

Arithmetic is numpy: fp32 where the method fixes fp32 (the quantizer's two
divisions), fp64 everywhere else, with a library matmul as the only borrowed
step. Every function cites the passage of the pages it follows:

  [P1] rocket blog, "The CUTLASS grouped GEMM beats the scalar GEMV loop at
       every M, M=1 included" (grouped-gemm-beats-gemv-at-every-m).
  [P2] rocket blog, "Fusing the MoE layer's two grouped GEMMs is worth 4%, and
       a CUDA graph already collects it" (moe-fusion-worth-4-percent).

Pipeline, [P1] "What changed": gather -> quantize -> grouped GEMM w13 (fused,
alpha = 1) -> SwiGLU with per-group gate/up weight_scale_2 -> quantize ->
grouped GEMM w2 -> scatter-add weighted by router weight * down
weight_scale_2.

Readings where the pages are silent (each is listed with its reason in the
design notes of the repository):
  * e2m1 values {0, .5, 1, 1.5, 2, 3, 4, 6}, round to nearest, ties to the even
    code, saturating at 6; a negative value that rounds to 0 keeps its sign
    (code 0x8).
  * e4m3 is E4M3FN (bias 7, max 448), round to nearest even, saturating.
  * activations carry no global scale: block scale = e4m3(amax / 6), element
    code = e2m1(x / scale), both divisions correctly rounded fp32; a block whose
    scale decodes to 0 is all-zero codes.
  * element 2j sits in bits 0-3 of byte j, element 2j+1 in bits 4-7.
  * packed activation rows are contiguous across groups; block scales are laid
    out per group in 128-row atoms, zero-padded to a multiple of 128 rows.
  * rows of a group ascend by slot index t*k + j; groups ascend by expert id.
  * GEMM outputs are fp32 on the device (fp64 here), h and y are bf16.
  * expert ids outside [0, E) mark unused slots.
Parity pins for every function live in tests/oracle_pins.py (run by tests/test_oracle.py).
"""
from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------
# Codecs
# --------------------------------------------------------------------------

E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def e2m1_decode(codes) -> np.ndarray:
    """Value of 4-bit e2m1 codes (bit 3 = sign). [P2] "Different globals on the
    two halves" names the e2m1 step (50% near 1.0); the value set is the
    standard FP4 E2M1 one."""
    codes = np.asarray(codes, dtype=np.uint8)
    mag = E2M1_MAGNITUDES[codes & 0x7]
    return np.where(codes & 0x8, -mag, mag)


def e2m1_encode(v) -> np.ndarray:
    """Round fp32 values to e2m1 codes: nearest, ties to even, saturate at 6.

    The grid has spacing 0.5 on [0, 2), 1 on [2, 4) and 2 on [4, 6]; rounding
    |v| to a multiple of the local spacing with numpy's half-to-even rint gives
    ties to the even code, because a code's last bit is the parity of its
    multiple of the spacing.
    """
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    r = np.minimum(np.rint(a / step) * step, 6.0)
    # value -> magnitude code: 0,.5,1,1.5 -> 0..3 ; 2,3 -> 4,5 ; 4,6 -> 6,7
    mag = np.where(r < 2.0, r * 2.0, np.where(r < 4.0, r + 2.0, r / 2.0 + 4.0)).astype(np.uint8)
    sign = np.signbit(v).astype(np.uint8) << 3
    return (mag | sign).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    """Value of E4M3FN codes: bias 7, subnormals m * 2^-9, 0x7F/0xFF are NaN."""
    c = np.asarray(codes, dtype=np.int64)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where(c & 0x80, -val, val)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def e4m3_encode(v) -> np.ndarray:
    """Round non-negative fp32 values to E4M3FN codes, nearest-even, saturating
    at 448. Used for block scales only, which are never negative."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    assert np.all(v >= 0), "block scales are non-negative"
    v = np.minimum(v, 448.0)
    _, ex = np.frexp(v)                     # v = f * 2^ex with f in [0.5, 1)
    e = np.maximum(ex - 1, -6)              # exponent of v, floored at the subnormal range
    q = np.exp2(e - 3.0)                    # spacing: 3 mantissa bits
    r = np.rint(v / q) * q                  # nearest, ties to even multiple
    r = np.minimum(r, 448.0)
    # code: subnormal part counts 2^-9 steps; normal part (E, m)
    _, rex = np.frexp(r)
    re = rex - 1
    normal = r >= 2.0 ** -6
    E = np.where(normal, re + 7, 0)
    m = np.where(normal, r / np.exp2(re) * 8.0 - 8.0, r / 2.0 ** -9)
    return (E * 8 + m).astype(np.uint8)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round fp64 values once to bf16 (8 significant bits), nearest-even."""
    x = np.asarray(x, dtype=np.float64)
    _, ex = np.frexp(x)
    e = np.maximum(ex - 1, -126)            # bf16 normals reach 2^-126
    q = np.exp2(e - 7.0)                    # spacing: 7 stored mantissa bits
    r = np.rint(x / q) * q
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


# --------------------------------------------------------------------------
# Block-scale layout
# --------------------------------------------------------------------------

def sf_atom_offset(m, c, Kc) -> np.ndarray:
    """Byte offset of scale column c (= k // 16) of row m in a region of 128-row
    atoms. [P1] "The seam CUTLASS forced open" and [P2] "Tiles below M=8" name
    the CUTLASS SFA/SFB swizzle with a 128-row atom shared by sm_100 and SM120.
    An atom covers 128 rows x 4 scale columns in 512 bytes: byte
    (m % 32) * 16 + ((m // 32) % 4) * 4 + (c % 4); atoms run along K first,
    then along rows."""
    m = np.asarray(m, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    assert Kc % 4 == 0
    atom = (m // 128) * (Kc // 4) + c // 4
    return atom * 512 + (m % 32) * 16 + ((m // 32) % 4) * 4 + (c % 4)


def swizzle_scales(linear: np.ndarray) -> np.ndarray:
    """Linear [N, Kc] scale bytes -> the 128-row atom layout (N padded up to a
    multiple of 128 with zero bytes). [P1] "The seam CUTLASS forced open":
    fuel::swizzle_block_scales, applied once per projection at load."""
    N, Kc = linear.shape
    Np = -(-N // 128) * 128
    out = np.zeros(Np * Kc, dtype=np.uint8)
    m, c = np.meshgrid(np.arange(N), np.arange(Kc), indexing="ij")
    out[sf_atom_offset(m, c, Kc)] = linear
    return out


def group_sf_blocks(group_offsets: np.ndarray) -> np.ndarray:
    """First 128-row scale block of each group (exclusive prefix of
    ceil(Mg / 128)); entry G is the total."""
    mg = np.diff(np.asarray(group_offsets, dtype=np.int64))
    return np.concatenate([[0], np.cumsum((mg + 127) // 128)]).astype(np.int64)


# --------------------------------------------------------------------------
# Pipeline steps
# --------------------------------------------------------------------------

def route_groups(topk_ids: np.ndarray, E: int):
    """Group routed slots by expert. [P1] "What changed": rows are grouped by
    expert id across the whole batch with an ordered map, so group order is a
    pure function of which experts fired; each expert is fetched once.

    Returns row_slot [R] (slot index t*k + j of each grouped row),
    group_offsets [G+1] and group_expert [G] (ascending expert ids).
    """
    ids = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    rows_of = {}
    for slot, e in enumerate(ids):          # slots visited in stream order
        if 0 <= e < E:
            rows_of.setdefault(int(e), []).append(slot)
    group_expert = sorted(rows_of)
    row_slot, offsets = [], [0]
    for e in group_expert:
        row_slot.extend(rows_of[e])
        offsets.append(len(row_slot))
    return (np.array(row_slot, dtype=np.int64), np.array(offsets, dtype=np.int64),
            np.array(group_expert, dtype=np.int64))


def gather_rows(x_bits: np.ndarray, row_slot: np.ndarray, k: int) -> np.ndarray:
    """[P1] "What changed", moe_gather_rows: one row per (stream, expert) slot,
    copied from the stream's normed activations. x_bits [T, H] bf16 bits."""
    return np.asarray(x_bits)[np.asarray(row_slot) // k]


def quantize_block(x16: np.ndarray):
    """NVFP4 codec for one 16-element block of fp32 values (activations).
    [P1] "What changed": quantize to NVFP4 (nvfp4_quantize_rows), one e4m3
    scale per 16 elements; alpha = 1 so no activation global exists.
    Returns (scale code, 16 e2m1 codes)."""
    x16 = np.asarray(x16, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x16)))
    s = e4m3_encode(np.float32(amax / np.float32(6.0)))
    d = np.float32(e4m3_decode(s))
    if d == 0:
        return np.uint8(0), np.zeros(16, dtype=np.uint8)
    return np.uint8(s), e2m1_encode(x16 / d)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Two e2m1 codes per byte along the last axis: element 2j low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def quantize_rows(rows_bits: np.ndarray, group_offsets: np.ndarray):
    """Quantize grouped bf16 rows [R, K] to NVFP4. [P1] "What changed" and
    "Proof" (test_kernels: packed nibbles and swizzled scale bytes, per group,
    group_m = {1, 130}). Returns packed [R, K/2] and the per-group padded
    scale region (bytes)."""
    rows = bf16_bits_to_f64(rows_bits).astype(np.float32)
    R, K = rows.shape
    Kc = K // 16
    # quantize_block, applied to every block at once
    blk = rows.reshape(R, Kc, 16)
    amax = np.max(np.abs(blk), axis=2).astype(np.float32)
    s = e4m3_encode(amax / np.float32(6.0))
    d = e4m3_decode(s).astype(np.float32)
    safe = np.where(d == 0, np.float32(1.0), d)
    codes = np.where((d == 0)[..., None], np.uint8(0), e2m1_encode(blk / safe[..., None]))
    # scale bytes into each group's zero-padded atom region
    offs = np.asarray(group_offsets, dtype=np.int64)
    blocks = group_sf_blocks(offs)
    sf = np.zeros(int(blocks[-1]) * 128 * Kc, dtype=np.uint8)
    for g in range(len(offs) - 1):
        m = np.arange(int(offs[g + 1] - offs[g]))
        mm, cc = np.meshgrid(m, np.arange(Kc), indexing="ij")
        sf[int(blocks[g]) * 128 * Kc + sf_atom_offset(mm, cc, Kc)] = s[int(offs[g]) + m]
    return pack_nibbles(codes.reshape(R, K)), sf


def dequantize_rows(packed: np.ndarray, sf: np.ndarray, group_offsets: np.ndarray) -> np.ndarray:
    """Values (fp64) of grouped NVFP4 rows, scales read from the atom layout."""
    packed = np.asarray(packed, dtype=np.uint8)
    R, K2 = packed.shape
    K, Kc = 2 * K2, K2 // 8
    offs = np.asarray(group_offsets, dtype=np.int64)
    blocks = group_sf_blocks(offs)
    vals = e2m1_decode(unpack_nibbles(packed))
    scale = np.zeros((R, Kc), dtype=np.float64)
    for g in range(len(offs) - 1):
        m = np.arange(int(offs[g + 1] - offs[g]))
        mm, cc = np.meshgrid(m, np.arange(Kc), indexing="ij")
        idx = int(blocks[g]) * 128 * Kc + sf_atom_offset(mm, cc, Kc)
        scale[int(offs[g]) + m] = e4m3_decode(np.asarray(sf)[idx])
    return vals * np.repeat(scale, 16, axis=1)


def dequantize_weight(packed: np.ndarray, sf_linear: np.ndarray) -> np.ndarray:
    """Values (fp64) of one expert's NVFP4 weight [N, K] without its global:
    [P2] "Bytes decide it": 0.5 B of e2m1 plus 1/16 B of e4m3 per element."""
    vals = e2m1_decode(unpack_nibbles(packed))
    return vals * np.repeat(e4m3_decode(sf_linear), 16, axis=1)


def grouped_gemm(a_packed, a_sf, group_offsets, group_expert, w_packed, w_sf_linear) -> np.ndarray:
    """D[r, n] = sum_k A[r, k] * W_e[n, k] per group, on dequantized values with
    no global (alpha = 1). [P1] "What changed": grouped GEMM (w13, fused)
    N=4096 K=4096 and grouped GEMM (w2) N=4096 K=2048, one call for all
    groups. Products of e2m1*e4m3 values are exact in fp64; the fp64 sum is
    the exact value to within fp64 rounding."""
    A = dequantize_rows(a_packed, a_sf, group_offsets)
    N = w_packed.shape[1]  # w_packed / w_sf_linear: anything indexable by expert id
    D = np.zeros((A.shape[0], N), dtype=np.float64)
    offs = np.asarray(group_offsets, dtype=np.int64)
    for g, e in enumerate(np.asarray(group_expert, dtype=np.int64)):
        r0, r1 = int(offs[g]), int(offs[g + 1])
        W = dequantize_weight(w_packed[e], w_sf_linear[e])
        D[r0:r1] = A[r0:r1] @ W.T
    return D


def swiglu(d13: np.ndarray, group_offsets, group_expert, g_gate_up) -> np.ndarray:
    """h = silu(gate * g_gate[e]) * (up * g_up[e]), rounded once to bf16.
    Gate is the first I columns of the fused w13 output, up the last I
    ([P1] "The seam CUTLASS forced open": gate_packed and up_packed back to
    back). Per-group globals applied here: [P2] "Different globals on the two
    halves", option (a). Returns bf16 bits [R, I]."""
    d13 = np.asarray(d13, dtype=np.float64)
    I = d13.shape[1] // 2
    gg = np.asarray(g_gate_up, dtype=np.float32).astype(np.float64)
    offs = np.asarray(group_offsets, dtype=np.int64)
    h = np.zeros((d13.shape[0], I), dtype=np.float64)
    for g, e in enumerate(np.asarray(group_expert, dtype=np.int64)):
        r0, r1 = int(offs[g]), int(offs[g + 1])
        gate = d13[r0:r1, :I] * gg[e, 0]
        up = d13[r0:r1, I:] * gg[e, 1]
        h[r0:r1] = gate / (1.0 + np.exp(-gate)) * up
    return f64_to_bf16_bits(h)


def scatter_add(d2: np.ndarray, row_slot, topk_ids, topk_w, g_down, T: int, E: int) -> np.ndarray:
    """y[t] = sum over t's rows, ascending row index, of topk_w * g_down[e] * D2[row].
    [P1] "What changed": scatter-add weighted by router weight * down
    weight_scale_2; "Proof": shared accumulator row, ordered-by-i
    accumulation. y is overwritten; a token with no rows gets 0.
    Returns bf16 bits [T, H]."""
    d2 = np.asarray(d2, dtype=np.float64)
    ids = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    w = np.asarray(topk_w, dtype=np.float32).reshape(-1).astype(np.float64)
    gd = np.asarray(g_down, dtype=np.float32).astype(np.float64)
    k = ids.size // T if T else 1
    y = np.zeros((T, d2.shape[1]), dtype=np.float64)
    for r, slot in enumerate(np.asarray(row_slot, dtype=np.int64)):  # ascending r
        t, e = int(slot) // k, int(ids[slot])
        y[t] += (w[slot] * gd[e]) * d2[r]
    return f64_to_bf16_bits(y)


def moe_layer(x_bits, topk_ids, topk_w, weights: dict, E: int) -> dict:
    """The whole routed-expert step, [P1] "What changed" (seven steps), with the
    weight globals applied after each GEMM ([P2] option (a) for w13, the
    scatter's router weight * down weight_scale_2 for w2). Returns every
    intermediate so each stage can be compared on its own."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    topk_ids = np.asarray(topk_ids)
    T, k = topk_ids.shape
    row_slot, offs, gexp = route_groups(topk_ids, E)
    xg = gather_rows(x_bits, row_slot, k)
    xq, xsf = quantize_rows(xg, offs)
    d13 = grouped_gemm(xq, xsf, offs, gexp, weights["w13_packed"], weights["w13_sf_linear"])
    h = swiglu(d13, offs, gexp, weights["g_gate_up"])
    hq, hsf = quantize_rows(h, offs)
    d2 = grouped_gemm(hq, hsf, offs, gexp, weights["w2_packed"], weights["w2_sf_linear"])
    y = scatter_add(d2, row_slot, topk_ids, topk_w, weights["g_down"], T, E)
    return dict(row_slot=row_slot, group_offsets=offs, group_expert=gexp, xg=xg, xq=xq,
                xsf=xsf, d13=d13, h=h, hq=hq, hsf=hsf, d2=d2, y=y)


# ---------------------------------------------------------------------------
# The GEMV path (W4A16): [P1] "Proof" (grouped vs GEMV at M=1) -- the pages keep it
# as an explicit override and fallback; it multiplies the exact bf16
# activations against the NVFP4 weights (no activation quantization), which is
# why its output differs materially from the W4A4 grouped path's.
# ---------------------------------------------------------------------------

def grouped_gemv_w4a16(a_bits, group_offsets, group_expert, w_packed, w_sf_linear) -> np.ndarray:
    """D[r, n] = sum_k a[r, k] * W_e[n, k] per group, with a[r, k] the exact
    value of the bf16 activation and W the dequantized NVFP4 weight without its
    global. Products of bf16 and e2m1*e4m3 values are exact in fp64."""
    A = bf16_bits_to_f64(np.asarray(a_bits, dtype=np.uint16))
    N = w_packed.shape[1]
    D = np.zeros((A.shape[0], N), dtype=np.float64)
    offs = np.asarray(group_offsets, dtype=np.int64)
    for g, e in enumerate(np.asarray(group_expert, dtype=np.int64)):
        r0, r1 = int(offs[g]), int(offs[g + 1])
        Wg = dequantize_weight(w_packed[e], w_sf_linear[e])  # [N, K]
        D[r0:r1] = A[r0:r1] @ Wg.T
    return D


def moe_layer_w4a16(x_bits, topk_ids, topk_w, weights: dict, E: int) -> dict:
    """The routed-expert step on the GEMV path: the same route, SwiGLU (h
    rounded once to bf16) and scatter-add as moe_layer, with both GEMMs taking
    bf16 activations as they are instead of their NVFP4 quantization."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    topk_ids = np.asarray(topk_ids)
    T, k = topk_ids.shape
    row_slot, offs, gexp = route_groups(topk_ids, E)
    xg = gather_rows(x_bits, row_slot, k)
    d13 = grouped_gemv_w4a16(xg, offs, gexp, weights["w13_packed"], weights["w13_sf_linear"])
    h = swiglu(d13, offs, gexp, weights["g_gate_up"])
    d2 = grouped_gemv_w4a16(h, offs, gexp, weights["w2_packed"], weights["w2_sf_linear"])
    y = scatter_add(d2, row_slot, topk_ids, topk_w, weights["g_down"], T, E)
    return dict(row_slot=row_slot, group_offsets=offs, group_expert=gexp, xg=xg, d13=d13, h=h, d2=d2, y=y)
