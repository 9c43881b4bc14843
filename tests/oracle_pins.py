"""Pins for the CPU oracle: each check takes the oracle module and raises
AssertionError when the oracle disagrees with what the pages or the
mathematics fix. The pins are plain functions so that the mutation tests can
run them against an oracle with a planted mistake and see them fail.

None of these checks re-types an oracle formula: each compares against an
independent route (brute-force search, a library routine, a closed form, a
figure printed on the pages, or a hand-worked example)."""
from fractions import Fraction

import numpy as np
import torch


# --------------------------------------------------------------------------
# e2m1
# --------------------------------------------------------------------------

def e2m1_value_from_bits(code: int) -> float:
    """FP4 E2M1 as a float format: 1 sign, 2 exponent (bias 1), 1 mantissa bit."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = m * 0.5 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


def check_e2m1_decode(O):
    for c in range(16):
        assert O.e2m1_decode(np.uint8(c)) == e2m1_value_from_bits(c), c


def check_e2m1_ties(O):
    # Hand table: ties between neighbours go to the code with mantissa bit 0.
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for v, want in ties.items():
        for sgn in (1.0, -1.0):
            got = O.e2m1_decode(O.e2m1_encode(np.float32(sgn * v)))
            assert got == sgn * want, (sgn * v, got)
    # saturation and signed zero
    assert O.e2m1_decode(O.e2m1_encode(np.float32(100.0))) == 6.0
    assert O.e2m1_encode(np.float32(-0.2)) == 0x8
    assert O.e2m1_encode(np.float32(0.2)) == 0x0


def brute_e2m1(v: float) -> int:
    """Nearest e2m1 value by exhaustive search; ties to the even code."""
    best = None
    for code in range(8):
        d = abs(abs(v) - e2m1_value_from_bits(code))
        key = (d, code & 1)
        if best is None or key < best[0]:
            best = (key, code)
    code = best[1]
    return code | (8 if np.signbit(v) else 0)


def e2m1_probe_values():
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)
    mids = (mags[:-1] + mags[1:]) / 2
    pts = np.concatenate([mags, mids, [6.5, 7.0, 9.0, 1e6]]).astype(np.float32)
    near = np.concatenate([pts, np.nextafter(pts, np.float32(-np.inf)),
                           np.nextafter(pts, np.float32(np.inf))])
    grid = np.arange(-8.0, 8.0, 1.0 / 64, dtype=np.float32)
    v = np.concatenate([near, -near, grid])
    return v[np.abs(v) < 1e7].astype(np.float32)


def check_e2m1_brute_force(O):
    v = e2m1_probe_values()
    got = O.e2m1_encode(v)
    want = np.array([brute_e2m1(float(x)) for x in v], dtype=np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(v[i]), int(got[i]), int(want[i])) for i in bad[:5]]


# --------------------------------------------------------------------------
# e4m3
# --------------------------------------------------------------------------

def torch_e4m3_values():
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def check_e4m3_decode_library(O):
    ref = torch_e4m3_values()
    got = O.e4m3_decode(np.arange(256))
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def e4m3_probe_values():
    vals = torch_e4m3_values()[:0x7F]  # 0 .. 448
    mids = (vals[:-1] + vals[1:]) / 2
    pts = np.concatenate([vals, mids]).astype(np.float32)
    near = np.concatenate([pts, np.nextafter(pts, np.float32(0)), np.nextafter(pts, np.float32(np.inf))])
    logs = np.exp2(np.linspace(-12, 8.9, 4000)).astype(np.float32)
    return np.unique(np.concatenate([near, logs, [0.0]]).astype(np.float32))


def check_e4m3_brute_force(O):
    vals = torch_e4m3_values()[:0x7F]
    v = e4m3_probe_values()
    v = v[v <= 448]
    got = O.e4m3_encode(v)
    d = np.abs(v.astype(np.float64)[:, None] - vals[None, :])
    dmin = d.min(axis=1, keepdims=True)
    cand = d == dmin
    # among equidistant codes keep the even one (codes are 0..126 here)
    even = cand & ((np.arange(0x7F) % 2) == 0)[None, :]
    want = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1)).astype(np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(v[i]), int(got[i]), int(want[i])) for i in bad[:5]]


def check_e4m3_library_cast(O):
    v = e4m3_probe_values()
    v = v[v <= 448]
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(v), lib)


def check_e4m3_saturation(O):
    for v in (448.0, 449.0, 463.9, 464.0, 500.0, 1e9):
        assert O.e4m3_encode(np.float32(v)) == 0x7E, v


def check_e4m3_fold_figures(O, pages):
    """Option (b) of the pages: fold the gate/up ratio into the e4m3 scales."""
    fig = pages["e4m3_fold"]
    codes = np.arange(1, 0x7F, dtype=np.uint8)
    assert codes.size == fig["codes"]
    want = (O.e4m3_decode(codes) * fig["ratio"]).astype(np.float32).astype(np.float64)
    got = O.e4m3_decode(O.e4m3_encode(want.astype(np.float32)))
    err = np.abs(got - want) / want
    assert round(float(err.mean()), 4) == fig["mean_rel_error"]
    assert round(float(err.max()), 4) == fig["max_rel_error"]
    assert int(np.sum(want > 448.0)) == fig["saturated_codes"]
    assert abs(fig["gate_global"] / fig["up_global"] - fig["ratio"]) < 5e-4


# --------------------------------------------------------------------------
# bf16
# --------------------------------------------------------------------------

def check_bf16_rounding(O):
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        [0.0, 1.0, -1.0, 1.00390625, 1.01171875]]).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f64_to_bf16_bits(x.astype(np.float64)), lib)
    # One rounding from fp64: 1 + 2^-8 + 2^-30 lies above the bf16 midpoint, so
    # it rounds up to 1 + 2^-7; rounding through fp32 first would give 1.0.
    assert O.bf16_bits_to_f64(O.f64_to_bf16_bits(np.float64(1 + 2.0 ** -8 + 2.0 ** -30))) == 1 + 2.0 ** -7
    assert O.bf16_bits_to_f64(O.f64_to_bf16_bits(np.float64(1 + 2.0 ** -8))) == 1.0


# --------------------------------------------------------------------------
# Block-scale layout and sizes
# --------------------------------------------------------------------------

def check_quantize_bytes(O, pages):
    """[P1] "Proof": 5728 bytes for group_m = {1, 130}."""
    fig = pages["quantize_bytes"]
    K = fig["K_reading"]
    mg = fig["group_m"]
    R = sum(mg)
    offs = np.concatenate([[0], np.cumsum(mg)])
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal((R, K)).astype(np.float32)).to(torch.bfloat16)
    packed, sf = O.quantize_rows(x.view(torch.int16).numpy().view(np.uint16), offs)
    assert packed.nbytes + sf.nbytes == fig["bytes"]
    # and the padding rows of each group carry zero scale bytes
    Kc = K // 16
    m_pad = np.arange(1, 128)
    mm, cc = np.meshgrid(m_pad, np.arange(Kc), indexing="ij")
    assert np.all(sf[O.sf_atom_offset(mm, cc, Kc)] == 0)


def check_sf_layout_points(O):
    # Hand-worked offsets: atom index (m // 128) * (Kc / 4) + c // 4, then
    # 16 bytes per row of the 32-row slab, 4 bytes per 32-row quarter.
    assert O.sf_atom_offset(0, 0, 8) == 0
    assert O.sf_atom_offset(33, 5, 8) == 512 + 16 + 4 + 1
    assert O.sf_atom_offset(130, 0, 8) == 1024 + 32
    assert O.sf_atom_offset(127, 3, 4) == 31 * 16 + 3 * 4 + 3
    assert O.sf_atom_offset(200, 9, 12) == (1 * 3 + 2) * 512 + 8 * 16 + 2 * 4 + 1


def check_sf_layout_structure(O):
    N, Kc = 256, 12
    m, c = np.meshgrid(np.arange(N), np.arange(Kc), indexing="ij")
    off = O.sf_atom_offset(m, c, Kc)
    assert np.array_equal(np.sort(off.ravel()), np.arange(N * Kc))   # bijection
    # chunk i (16 bytes) of an atom holds rows i, i+32, i+64, i+96, each with
    # the 4 scale columns of that atom in consecutive bytes
    for i in (0, 7, 31):
        for q in range(4):
            row = i + 32 * q
            assert list(off[row, 4:8]) == [512 + 16 * i + 4 * q + j for j in range(4)]


def check_fused_swizzle(O):
    """[P1] "The seam CUTLASS forced open": w13's scales = gate's swizzle
    followed by up's swizzle, bit-identical to swizzling the fused matrix
    because the intermediate size is a multiple of the 128-row atom."""
    rng = np.random.default_rng(5)
    for I, same in ((128, True), (256, True), (64, False)):
        gate = rng.integers(1, 255, (I, 8), dtype=np.uint8)
        up = rng.integers(1, 255, (I, 8), dtype=np.uint8)
        fused = O.swizzle_scales(np.concatenate([gate, up]))
        cat = np.concatenate([O.swizzle_scales(gate), O.swizzle_scales(up)])
        assert (fused.size == cat.size and np.array_equal(fused, cat)) == same, I


def expert_bytes(H, I):
    return 2 * I * H * 9 // 16 + H * I * 9 // 16


def check_sizes(pages):
    slot = pages["expert_slot"]
    H, I = slot["hidden"], slot["intermediate"]
    b = expert_bytes(H, I)
    assert b == 14_155_776
    assert b / 2 ** 20 == slot["one_scale_copy_mib"]
    sf = (2 * I * H + H * I) // 16
    assert (b + sf) / 2 ** 20 == slot["two_scale_copies_mib"]
    bud = pages["byte_budget"]
    E = bud["experts"]
    w13 = E * 2 * I * H * 9 / 16
    w2 = E * H * I * 9 / 16
    assert round(w13 / 1e9, 3) == bud["w13_gb"]
    assert round(w2 / 1e9, 3) == bud["w2_gb"]
    assert round((w13 + w2) / 1e9, 3) == bud["total_gb"]
    assert round((w13 + w2) / 238e9 * 1e3, 2) == bud["roofline_ms_at_238_gbs"]


# --------------------------------------------------------------------------
# Pipeline steps
# --------------------------------------------------------------------------

def bf16_bits(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def check_quantize_block_hand(O):
    # amax 6 -> scale e4m3(1.0) = 0x38; codes are then the e2m1 codes of x.
    x = np.array([6, -3, 1.5, 0.75, -0.25, 0.1, 4, -6, 2.5, 3.5, 0, -0.5, 1, -1.25, 5, 2], dtype=np.float32)
    s, q = O.quantize_block(x)
    assert s == 0x38
    want = [0x7, 0xD, 0x3, 0x2, 0x8, 0x0, 0x6, 0xF, 0x4, 0x6, 0x0, 0x9, 0x2, 0xA, 0x6, 0x4]
    assert list(q) == want
    # amax 0.3 -> 0.3 / 6 = 0.05 in fp32 = 1.6 * 2^-5 -> e4m3 1.625 * 2^-5
    # = 0.05078125 (exponent field 2, mantissa 5: code 0x15)
    y = np.full(16, 0.1, dtype=np.float32)
    y[3] = -0.3
    s, q = O.quantize_block(y)
    assert s == 0x15
    # 0.1 / 0.05078125 = 1.969 -> 2.0 (code 4); -0.3 / 0.05078125 = -5.9 -> -6 (0xF)
    assert q[3] == 0xF and q[0] == 0x4
    # all-zero and vanishing blocks: scale 0 and zero codes
    # (negative values too: an underflowed block is code 0, not signed zero)
    zero_blocks = (np.zeros(16, np.float32), np.full(16, 1e-6, np.float32), np.full(16, -1e-6, np.float32))
    for z in zero_blocks:
        s, q = O.quantize_block(z)
        assert s == 0 and not q.any()
    # the row quantizer gives the same hand-worked codes and scales
    row = np.concatenate([x, y] + list(zero_blocks) + [np.zeros(48, np.float32)]).astype(np.float32)
    packed, sf = O.quantize_rows(bf16_bits(row)[None, :], np.array([0, 1]))
    codes = O.unpack_nibbles(packed)[0]
    assert list(codes[:16]) == want and codes[19] == 0xF and not codes[32:].any()
    assert [sf[O.sf_atom_offset(0, c, 8)] for c in range(5)] == [0x38, 0x15, 0, 0, 0]


def check_pack_order(O):
    # element 2j in bits 0-3 of byte j
    codes = np.array([0x1, 0xF, 0x7, 0x8], dtype=np.uint8)
    assert list(O.pack_nibbles(codes)) == [0xF1, 0x87]
    assert list(O.unpack_nibbles(np.array([0xF1, 0x87], np.uint8))) == [0x1, 0xF, 0x7, 0x8]


def check_quantize_error_bound(O):
    """Property: every value lands on the nearest point of the scaled grid,
    so |deq - x| <= half the local grid step times the scale (x / scale <= 6
    when the scale did not round down; otherwise saturates at 6 * scale)."""
    rng = np.random.default_rng(11)
    R, K = 12, 256
    x = bf16_bits(rng.standard_normal((R, K)) * 3.0)
    offs = np.array([0, 5, 12])
    packed, sf = O.quantize_rows(x, offs)
    deq = O.dequantize_rows(packed, sf, offs)
    xv = O.bf16_bits_to_f64(x)
    scale = np.zeros((R, K // 16))
    blocks = O.group_sf_blocks(offs)
    for g in range(2):
        for m in range(offs[g + 1] - offs[g]):
            for c in range(K // 16):
                scale[offs[g] + m, c] = O.e4m3_decode(sf[blocks[g] * 128 * (K // 16) + O.sf_atom_offset(m, c, K // 16)])
    sc = np.repeat(scale, 16, axis=1)
    r = np.abs(xv) / sc
    step = np.where(r < 2, 0.5, np.where(r < 4, 1.0, 2.0))
    bound = np.where(r <= 6, step / 2 * sc, np.abs(xv) - 6 * sc)
    assert np.all(np.abs(deq - xv) <= bound * (1 + 1e-6) + 1e-30)
    # the block maximum maps close to the top of the grid
    amax = np.abs(xv).reshape(R, K // 16, 16).max(axis=2)
    # (scale within 1/16 relative of amax / 6 -> ratio within [6/(17/16), 6/(15/16)])
    ratio = amax / scale
    assert np.all((ratio >= 6 / (17 / 16) - 1e-9) & (ratio <= 6 / (15 / 16) + 1e-9))


def check_grouping_brute(O):
    rng = np.random.default_rng(13)
    for trial in range(20):
        T, k, E = int(rng.integers(1, 9)), int(rng.integers(1, 5)), int(rng.integers(2, 12))
        ids = np.stack([rng.permutation(E + 2)[:k] - 1 for _ in range(T)]).astype(np.int32)
        ids[ids >= E] = -1
        row_slot, offs, gexp = O.route_groups(ids, E)
        flat = ids.ravel()
        pairs = sorted((int(e), s) for s, e in enumerate(flat) if 0 <= e < E)
        assert list(row_slot) == [s for _, s in pairs]
        assert list(gexp) == sorted(set(e for e, _ in pairs))
        for g, e in enumerate(gexp):
            assert all(flat[s] == e for s in row_slot[offs[g]:offs[g + 1]])


def check_gather(O):
    x = np.arange(3 * 4, dtype=np.uint16).reshape(3, 4)
    row_slot = np.array([5, 0, 3, 4])
    assert np.array_equal(O.gather_rows(x, row_slot, 2), x[[2, 0, 1, 2]])


def tiny_gemm_case(seed=17, N=128, K=64, mg=(2, 1)):
    rng = np.random.default_rng(seed)
    R = sum(mg)
    E = 3
    x = bf16_bits(rng.standard_normal((R, K)))
    offs = np.concatenate([[0], np.cumsum(mg)])
    gexp = np.array([2, 0][:len(mg)])
    w = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    wsf = rng.integers(0x30, 0x7F, (E, N, K // 16), dtype=np.uint8)
    return x, offs, gexp, w, wsf


def check_gemm_brute_force(O):
    x, offs, gexp, w, wsf = tiny_gemm_case()
    a, asf = O.quantize_rows(x, offs)
    D = O.grouped_gemm(a, asf, offs, gexp, w, wsf)
    K = x.shape[1]
    Kc = K // 16
    blocks = O.group_sf_blocks(offs)

    def frac(v):
        return Fraction(float(v))

    e4m3_vals = torch_e4m3_values()
    rng = np.random.default_rng(1)
    for _ in range(24):
        r = int(rng.integers(0, len(x)))
        n = int(rng.integers(0, w.shape[1]))
        g = int(np.searchsorted(offs, r, side="right") - 1)
        m, e = r - offs[g], gexp[g]
        acc = Fraction(0)
        for kk in range(K):
            an = (a[r, kk // 2] >> (4 * (kk % 2))) & 0xF
            wn = (w[e, n, kk // 2] >> (4 * (kk % 2))) & 0xF
            s_a = asf[blocks[g] * 128 * Kc + O.sf_atom_offset(m, kk // 16, Kc)]
            acc += (frac(e2m1_value_from_bits(int(an))) * frac(e4m3_vals[s_a])
                    * frac(e2m1_value_from_bits(int(wn))) * frac(e4m3_vals[wsf[e, n, kk // 16]]))
        assert Fraction(float(D[r, n])) == acc, (r, n)


def check_gemm_invariants(O):
    """[P1] "Proof": row alone (Mg=1) == row paired (Mg=2); fused w13 ==
    separate gate-only and up-only GEMMs; repeated calls identical."""
    x, offs, gexp, w, wsf = tiny_gemm_case(seed=19, N=256, K=128, mg=(2,))
    a, asf = O.quantize_rows(x, offs)
    pair = O.grouped_gemm(a, asf, offs, gexp, w, wsf)
    for r in range(2):
        one = np.array([0, 1])
        a1, s1 = O.quantize_rows(x[r:r + 1], one)
        alone = O.grouped_gemm(a1, s1, one, gexp, w, wsf)
        assert np.array_equal(alone[0], pair[r])
    gate = O.grouped_gemm(a, asf, offs, gexp, w[:, :128], wsf[:, :128])
    up = O.grouped_gemm(a, asf, offs, gexp, w[:, 128:], wsf[:, 128:])
    assert np.array_equal(np.concatenate([gate, up], axis=1), pair)
    for _ in range(5):
        assert np.array_equal(O.grouped_gemm(a, asf, offs, gexp, w, wsf), pair)


def check_swiglu_closed_form(O):
    """silu(x) = x * sigmoid(x) and sigmoid(ln a) = a / (1 + a)."""
    I = 4
    gg = np.array([[2.0, 0.5]], dtype=np.float32)        # g_gate != g_up
    ln3 = np.log(3.0)
    gate = np.array([0.0, ln3 / 2, -ln3 / 2, 20.0])      # times g_gate=2 -> 0, ln3, -ln3, 40
    up = np.array([5.0, 4.0, 8.0, 0.25])                 # times g_up=0.5 -> 2.5, 2, 4, 0.125
    d13 = np.concatenate([gate, up])[None, :]
    h = O.bf16_bits_to_f64(O.swiglu(d13, [0, 1], [0], gg))[0]
    want = [0.0, ln3 * 0.75 * 2.0, -ln3 * 0.25 * 4.0, 40.0 * 0.125]
    assert np.array_equal(h, O.bf16_bits_to_f64(O.f64_to_bf16_bits(np.array(want))))
    assert I == d13.shape[1] // 2


def check_scatter_hand(O):
    """Two tokens, k = 2, E = 3. Hand-summed in ascending row order."""
    H = 2
    topk_ids = np.array([[2, 0], [0, -1]])
    topk_w = np.array([[0.5, 0.25], [1.0, 0.0]], dtype=np.float32)
    g_down = np.array([2.0, 8.0, 4.0], dtype=np.float32)
    # grouped rows: expert 0 -> slots 1, 2 (rows 0, 1); expert 2 -> slot 0 (row 2)
    row_slot = np.array([1, 2, 0])
    d2 = np.array([[1.0, -2.0], [3.0, 5.0], [0.5, 0.125]])
    y = O.bf16_bits_to_f64(O.scatter_add(d2, row_slot, topk_ids, topk_w, g_down, T=2, E=3))
    # token 0: 0.25*2*[1,-2] + 0.5*4*[0.5,0.125] = [0.5+1, -1+0.25]
    # token 1: 1.0*2*[3,5]
    assert np.array_equal(y, np.array([[1.5, -0.75], [6.0, 10.0]]))
    assert H == 2


def small_layer_inputs(T=6, E=5, H=64, I=128, k=2, seed=23):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    tw = rng.random((T, k)).astype(np.float32)
    x = bf16_bits(rng.standard_normal((T, H)))
    wts = dict(
        w13_packed=rng.integers(0, 256, (E, 2 * I, H // 2), dtype=np.uint8),
        w13_sf_linear=rng.integers(0x58, 0x7F, (E, 2 * I, H // 16), dtype=np.uint8),
        g_gate_up=np.stack([np.full(E, 4.65e-5), np.full(E, 4.65e-5 / 1.2308)], 1).astype(np.float32),
        w2_packed=rng.integers(0, 256, (E, H, I // 2), dtype=np.uint8),
        w2_sf_linear=rng.integers(0x58, 0x7F, (E, H, I // 16), dtype=np.uint8),
        g_down=np.full(E, 4.2e-5, dtype=np.float32))
    return x, ids, tw, wts


def check_layer_batch_invariance(O):
    """[P1] "Proof", batch parity: a stream's output is the same alone (M=1)
    or inside a batch (M=8)."""
    x, ids, tw, wts = small_layer_inputs()
    full = O.moe_layer(x, ids, tw, wts, E=5)["y"]
    for t in (0, 3, 5):
        alone = O.moe_layer(x[t:t + 1], ids[t:t + 1], tw[t:t + 1], wts, E=5)["y"]
        assert np.array_equal(alone[0], full[t]), t


def check_unused_slots(O):
    x, ids, tw, wts = small_layer_inputs()
    ids2 = ids.copy()
    ids2[:, 1] = -1
    y_masked = O.moe_layer(x, ids2, tw, wts, E=5)["y"]
    y_k1 = O.moe_layer(x, ids[:, :1], tw[:, :1], wts, E=5)["y"]
    assert np.array_equal(y_masked, y_k1)


# ---------------------------------------------------------------------------
# the GEMV path (W4A16): [P1] "Proof" (grouped vs GEMV at M=1)
# ---------------------------------------------------------------------------

def lossless_rows(rng, R, K):
    """bf16 rows whose NVFP4 quantization loses nothing: each 16-block is a
    power-of-two scale times e2m1 values, with one element at +-6 times it
    (so the block scale is that power of two exactly)."""
    vals = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    x = rng.choice(vals, size=(R, K)) * rng.choice([-1.0, 1.0], size=(R, K))
    x[:, ::16] = 6.0 * rng.choice([-1.0, 1.0], size=(R, K // 16))
    scale = np.exp2(rng.integers(-6, 4, size=(R, K // 16)).astype(np.float64)).repeat(16, axis=1)
    return bf16_bits(x * scale)


def check_gemv_w4a16_lossless(O):
    """Where quantizing the activations loses nothing, W4A16 and W4A4 are the
    same arithmetic: the GEMV path must equal the grouped GEMM exactly."""
    rng = np.random.default_rng(31)
    _, offs, gexp, w, wsf = tiny_gemm_case(seed=31)
    x = lossless_rows(rng, int(offs[-1]), 64)
    a, asf = O.quantize_rows(x, offs)
    exact = torch.tensor(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(O.dequantize_rows(a, asf, offs), exact)  # the construction holds
    assert np.array_equal(O.grouped_gemv_w4a16(x, offs, gexp, w, wsf), O.grouped_gemm(a, asf, offs, gexp, w, wsf))


def check_gemv_w4a16_brute_force(O):
    """Each output against the exact rational sum of bf16 activation times
    e2m1 code times e4m3 scale (values read through torch, not the oracle)."""
    x, offs, gexp, w, wsf = tiny_gemm_case(seed=37)
    D = O.grouped_gemv_w4a16(x, offs, gexp, w, wsf)
    xv = torch.tensor(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    e4m3_vals = torch_e4m3_values()
    rng = np.random.default_rng(2)
    for _ in range(24):
        r = int(rng.integers(0, len(x)))
        n = int(rng.integers(0, w.shape[1]))
        e = gexp[int(np.searchsorted(offs, r, side="right") - 1)]
        acc = Fraction(0)
        for kk in range(x.shape[1]):
            wn = (w[e, n, kk // 2] >> (4 * (kk % 2))) & 0xF
            acc += (Fraction(float(xv[r, kk])) * Fraction(e2m1_value_from_bits(int(wn)))
                    * Fraction(float(e4m3_vals[wsf[e, n, kk // 16]])))
        assert abs(Fraction(float(D[r, n])) - acc) <= abs(acc) * Fraction(1, 2 ** 50), (r, n)


def check_layer_w4a16(O):
    """The GEMV-path step is batch invariant, and on losslessly quantizable
    activations its first GEMM equals the grouped path's."""
    x, ids, tw, wts = small_layer_inputs()
    full = O.moe_layer_w4a16(x, ids, tw, wts, E=5)["y"]
    for t in (0, 3, 5):
        alone = O.moe_layer_w4a16(x[t:t + 1], ids[t:t + 1], tw[t:t + 1], wts, E=5)["y"]
        assert np.array_equal(alone[0], full[t]), t
    # the first GEMM of token 0's first slot, recomputed from the raw codes
    res = O.moe_layer_w4a16(x, ids, tw, wts, E=5)
    r = int(np.where(res["row_slot"] == 0)[0][0])
    e = int(ids[0, 0])
    xv = torch.tensor(x[0].view(np.int16)).view(torch.bfloat16).double().numpy()
    e4m3_vals = torch_e4m3_values()
    codes = np.stack([wts["w13_packed"][e] & 0xF, wts["w13_packed"][e] >> 4], axis=-1).reshape(len(wts["w13_packed"][e]), -1)
    wv = np.vectorize(e2m1_value_from_bits)(codes) * np.repeat(e4m3_vals[wts["w13_sf_linear"][e]], 16, axis=1)
    want = wv @ xv
    assert np.allclose(res["d13"][r], want, rtol=1e-12, atol=0.0)
    xl = lossless_rows(np.random.default_rng(41), x.shape[0], x.shape[1])
    a = O.moe_layer_w4a16(xl, ids, tw, wts, E=5)
    b = O.moe_layer(xl, ids, tw, wts, E=5)
    assert np.array_equal(a["d13"], b["d13"])
    assert np.array_equal(a["h"], b["h"])
