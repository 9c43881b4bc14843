"""Shared helpers of the GPU parity tests: conversions, the stage-by-stage run
through the C ABI, and lazy host copies of expert weights for the oracle."""
import numpy as np
import torch

from nvfp4_block_scaled_gather_gb300 import _native as N
from oracle import nvfp4_moe as O

GEMM_TOL = 1e-5   # grouped GEMM vs the oracle fed the same NVFP4 inputs (relative Frobenius)
LAYER_TOL = 1e-2  # layer output vs the oracle (relative Frobenius)


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def np_to_bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def rel_fro(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def bf16_ulps(got_bits, want_bits) -> np.ndarray:
    """Distance in bf16 units in the last place (same-sign ordering)."""
    def key(b):
        b = np.asarray(b, dtype=np.uint16).astype(np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(key(got_bits) - key(want_bits))


def assert_swiglu_close(h_gpu_bits, d13, offs, gexp, g_gate_up):
    """The device's SwiGLU (fp32, CUDA expf, one bf16 rounding) against the
    oracle's (fp64, one bf16 rounding) fed the same d13: within one bf16 ulp
    wherever fp32 can evaluate silu(gate) = gate / (1 + exp(-gate)), i.e.
    exp(-gate) and silu(gate) are both in fp32's normal range. Below that
    (gate < -ln(FLT_MAX) = -88.72, where exp(-gate) overflows to inf and the
    device's silu is -0, or |silu| below 2^-126) the device's h is 0 or within
    one ulp of the oracle's, and the oracle's |h| is below 2^-121 * |up|: what
    fp32 cannot hold."""
    d13 = np.asarray(d13, dtype=np.float64)
    with np.errstate(over="ignore"):
        h_ref = O.swiglu(d13, offs, gexp, g_gate_up)
    I = d13.shape[1] // 2
    gg = np.asarray(g_gate_up, dtype=np.float32).astype(np.float64)
    e_of_row = np.repeat(np.asarray(gexp, dtype=np.int64), np.diff(np.asarray(offs, dtype=np.int64)))
    gate = d13[:, :I] * gg[e_of_row, 0:1]
    up = d13[:, I:] * gg[e_of_row, 1:2]
    with np.errstate(over="ignore"):
        silu = gate / (1.0 + np.exp(-gate))
    out_of_fp32 = (-gate > np.log(float(np.finfo(np.float32).max))) | (np.abs(silu) < 2.0 ** -126)
    ulps = bf16_ulps(h_gpu_bits, h_ref)
    bad = np.nonzero((ulps > 1) & ~out_of_fp32)
    assert bad[0].size == 0, [(float(gate[i, j]), float(up[i, j]), int(ulps[i, j])) for i, j in zip(*bad)][:5]
    if out_of_fp32.any():
        got = O.bf16_bits_to_f64(np.asarray(h_gpu_bits)[out_of_fp32])
        want = O.bf16_bits_to_f64(h_ref[out_of_fp32])
        assert np.all((got == 0) | (ulps[out_of_fp32] <= 1))
        assert np.all(np.abs(want) <= 2.0 ** -121 * np.abs(up[out_of_fp32]) + 2.0 ** -133)
    return h_ref


def assert_scatter_close(y_gpu_bits, d2, row_slot, ids, tw, g_down, T, E):
    """The device's scatter-add (fp32 coefficient tw * g_down, fp32 fused
    multiply-adds in ascending row order, one bf16 rounding) against the
    oracle's (fp64, one bf16 rounding) fed the same d2: within one bf16 ulp,
    plus, where the token's terms cancel, the fp32 rounding of the sum itself:
    2 * k * 2^-24 * sum_i |coef_i * d2_i| (one rounding per coefficient and
    per multiply-add)."""
    d2 = np.asarray(d2, dtype=np.float64)
    y_ref = O.scatter_add(d2, row_slot, ids, tw, g_down, T, E)
    ids_f = np.asarray(ids, dtype=np.int64).reshape(-1)
    w = np.asarray(tw, dtype=np.float32).reshape(-1).astype(np.float64)
    gd = np.asarray(g_down, dtype=np.float32).astype(np.float64)
    k = ids_f.size // T if T else 1
    mag = np.zeros((T, d2.shape[1]))
    for r, slot in enumerate(np.asarray(row_slot, dtype=np.int64)):
        mag[slot // k] += np.abs(w[slot] * gd[ids_f[slot]] * d2[r])
    got = O.bf16_bits_to_f64(y_gpu_bits)
    want = O.bf16_bits_to_f64(y_ref)
    ulp = np.maximum(np.abs(want) * 2.0 ** -7, 2.0 ** -133)
    assert np.all(np.abs(got - want) <= ulp + 2 * k * 2.0 ** -24 * mag)
    return y_ref


class LazyExperts:
    """Indexable by expert id; copies that expert's tensor to the host on use."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, e):
        return self.t[int(e)].cpu().numpy()


def oracle_weights(w: dict) -> dict:
    """Weights dict the oracle reads: lazy per-expert host copies of the
    generator's tensors (packed nibbles, LINEAR scales, globals)."""
    out = {k: LazyExperts(w[k]) for k in ("w13_packed", "w13_sf_linear", "w2_packed", "w2_sf_linear")}
    out["g_gate_up"] = w["g_gate_up"].cpu().numpy()
    out["g_down"] = w["g_down"].cpu().numpy()
    return out


def row_scales(sf_atom: np.ndarray, offs: np.ndarray, K: int) -> np.ndarray:
    """Per-row scale codes [R, K/16] read out of the oracle's 128-row atom
    region (the oracle's own layout function)."""
    from oracle import nvfp4_moe as O
    Kc = K // 16
    blocks = O.group_sf_blocks(offs)
    out = np.zeros((int(offs[-1]), Kc), np.uint8)
    for g in range(len(offs) - 1):
        m = np.arange(int(offs[g + 1] - offs[g]))
        mm, cc = np.meshgrid(m, np.arange(Kc), indexing="ij")
        out[offs[g] + m] = sf_atom[int(blocks[g]) * 128 * Kc + O.sf_atom_offset(mm, cc, Kc)]
    return out


def chunk32_bytes(scales: np.ndarray, offs: np.ndarray, K: int) -> np.ndarray:
    """The MOE_SF_CHUNK32 token-scale region for these per-row scales, built
    from its definition: 32-row chunks per group, one 512-byte block per 64 K
    values, row i of a block = [chunk row i's 4 scales, 12 zero bytes]."""
    na = K // 64
    mg = np.diff(offs)
    nch = (mg + 31) // 32
    out = np.zeros(int(nch.sum()) * na * 512, np.uint8)
    c = 0
    for g in range(len(mg)):
        for q in range(int(nch[g])):
            rows = np.arange(offs[g] + 32 * q, min(offs[g + 1], offs[g] + 32 * q + 32))
            for i, r in enumerate(rows):
                for a in range(na):
                    o = (c * na + a) * 512 + i * 16
                    out[o:o + 4] = scales[r, 4 * a:4 * a + 4]
            c += 1
    return out


def chunk32_row_scales(region: np.ndarray, chunk_info: np.ndarray, rows, K: int) -> np.ndarray:
    """Per-row scale codes [len(rows), K/16] of grouped rows, read out of a
    MOE_SF_CHUNK32 region through the chunk table (row0, rows, expert, group
    per 32-row chunk): the inverse of chunk32_bytes for the rows asked for."""
    info = np.asarray(chunk_info, dtype=np.int64).reshape(-1, 4)
    region = np.asarray(region, dtype=np.uint8)
    na = K // 64
    out = np.zeros((len(rows), K // 16), np.uint8)
    for i, r in enumerate(rows):
        c = int(np.nonzero((info[:, 0] <= r) & (r < info[:, 0] + info[:, 1]))[0][0])
        m = int(r - info[c, 0])
        for a in range(na):
            o = (c * na + a) * 512 + m * 16
            out[i, 4 * a:4 * a + 4] = region[o:o + 4]
    return out


def run_stages(x, ids, tw, W: N.Weights, E: int) -> dict:
    """The layer through the separate entry points (unfused)."""
    T, H = x.shape
    k = ids.shape[1]
    S, I, dev = T * k, W.I, x.device
    G = N.Groups(T, k, E, dev)
    xg = torch.zeros(S, H, dtype=torch.bfloat16, device=dev)
    N.moe_gather_rows(x, ids, E, G, xg)
    xq = torch.zeros(S, H // 2, dtype=torch.uint8, device=dev)
    xsf = torch.zeros(N.sf_bytes(S, E, H), dtype=torch.uint8, device=dev)
    N.nvfp4_quantize_rows(xg, G, xq, xsf)
    d13 = torch.zeros(S, 2 * I, dtype=torch.float32, device=dev)
    N.nvfp4_grouped_gemm(xq, xsf, G, W.w13, d13)
    h = torch.zeros(S, I, dtype=torch.bfloat16, device=dev)
    N.swiglu_grouped(d13, G, W.g_gate_up, h)
    hq = torch.zeros(S, I // 2, dtype=torch.uint8, device=dev)
    hsf = torch.zeros(N.sf_bytes(S, E, I), dtype=torch.uint8, device=dev)
    N.nvfp4_quantize_rows(h, G, hq, hsf)
    d2 = torch.zeros(S, H, dtype=torch.float32, device=dev)
    N.nvfp4_grouped_gemm(hq, hsf, G, W.w2, d2)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    N.moe_scatter_add(d2, ids, tw, E, G, W.g_down, y)
    torch.cuda.synchronize()
    return dict(groups=G.host(), xg=xg, xq=xq, xsf=xsf, d13=d13, h=h, hq=hq, hsf=hsf, d2=d2, y=y)


def weights_from(w: dict) -> N.Weights:
    return N.Weights(w["w13_packed"], w["w13_sf_linear"], w["g_gate_up"], w["w2_packed"], w["w2_sf_linear"],
                     w["g_down"])


def small_case(device, seed=5):
    """Several tiles and ragged tails: E=6, H=512, I=384 (w13 N=768 K=512,
    w2 N=512 K=384 = one and a half K stages), 160 tokens top-2 with one
    expert taking 140 rows (two 128-row blocks), one taking 1, one none, and
    some unused slots."""
    g = torch.Generator().manual_seed(seed)
    E, H, I, T, k = 6, 512, 384, 160, 2
    ids = torch.full((T, k), -1, dtype=torch.int32)
    ids[:140, 0] = 0
    ids[140:, 0] = 3
    others = torch.tensor([1, 3, 4])
    ids[:, 1] = others[torch.randint(0, 3, (T,), generator=g)]
    ids[140:, 1] = 4
    ids[150, 1] = 5                      # expert 5: a single row
    ids[7, 1] = -1                       # unused slots
    ids[141, 0] = -1
    tw = torch.rand((T, k), generator=g)
    from nvfp4_block_scaled_gather_gb300.synthetic import make_activations, make_weights
    w = make_weights(E, H, I, seed=seed, device="cpu")
    x = make_activations(T, H, seed=seed + 1, device="cpu")
    return E, x, ids, tw, w


def edge_rows(R, K, seed=0):
    """bf16 rows mixing N(0,1), wide dynamic range, e2m1 ties, e4m3 subnormal
    and saturating scales, all-zero and underflowing (signed) blocks."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((R, K)).astype(np.float32)
    x *= np.exp2(rng.integers(-14, 12, (R, K // 16))).repeat(16, axis=1).astype(np.float32)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    for r in range(R):
        c = 16 * int(rng.integers(0, K // 16))
        x[r, c:c + 16] = np.tile(ties, 2) * rng.choice([-1, 1], 16)  # amax 6 -> scale 1, exact ties
    x[0, :16] = 0.0
    x[min(1, R - 1), :16] = -1e-7
    x[min(2, R - 1), 16:32] = 5000.0                                    # scale saturates at 448
    x[min(3, R - 1), 32:48] = 2.0 ** -9 * np.arange(16)                  # subnormal scale
    return np.asarray(O.f64_to_bf16_bits(x.astype(np.float64)))


def quotient_sweep_blocks() -> np.ndarray:
    """bf16 bits, 16-value blocks covering every nonzero e4m3 scale code c and,
    for each, every bf16 magnitude from d/8 to 6d (d the value of c) in both
    signs: element 0 of a block is +-6d, the block maximum, so the block scale
    is exactly c, and the other 15 carry the sweep, so v / d passes every
    e2m1 rounding threshold and its neighbours; the padding of the last
    block of each code alternates +0 and -0. Returns [n_blocks, 16]."""
    pos = np.arange(0x0001, 0x7F80, dtype=np.uint16)             # positive finite bf16
    mags = O.bf16_bits_to_f64(pos)
    out = []
    for c in range(1, 0x7F):
        d = float(O.e4m3_decode(np.array([c], np.uint8))[0])
        sel = pos[(mags >= d / 8) & (mags <= 6 * d)]
        sweep = np.concatenate([sel, sel | np.uint16(0x8000)])
        pad = (-sweep.size) % 15
        sweep = np.concatenate([sweep, np.where(np.arange(pad) % 2 == 0, 0x0000, 0x8000).astype(np.uint16)])
        body = sweep.reshape(-1, 15)
        top = O.f64_to_bf16_bits(np.array([6 * d]))[0]
        head = np.where(np.arange(body.shape[0]) % 2 == 0, top, top | 0x8000).astype(np.uint16)
        out.append(np.concatenate([head[:, None], body], axis=1))
    return np.concatenate(out)


def amax_sweep_blocks() -> np.ndarray:
    """bf16 bits, one 16-value block per positive finite bf16 value a (0x0001
    .. 0x7F7F): element 0 is +-a, the block maximum, so the block scale
    runs over e4m3(a / 6) for every a, through the subnormal scales, the
    zero-scale (underflow) blocks and the saturated ones; the other 15 are
    bf16(a j / 16), j = 1 .. 15, with alternating signs. Returns [32639, 16]."""
    a = np.arange(0x0001, 0x7F80, dtype=np.uint16)
    av = O.bf16_bits_to_f64(a)
    j = np.arange(1, 16, dtype=np.float64)
    body = O.f64_to_bf16_bits(av[:, None] * j[None, :] / 16.0)
    body = np.where(np.arange(15) % 2 == 1, body | np.uint16(0x8000), body).astype(np.uint16)
    head = np.where(np.arange(a.size) % 2 == 0, a, a | np.uint16(0x8000)).astype(np.uint16)
    return np.concatenate([head[:, None], body], axis=1)


def blocks_as_rows(blocks: np.ndarray, R: int, K: int) -> np.ndarray:
    """Lay 16-value blocks out row-major over [R, K] bf16 bits, zero-padded."""
    flat = blocks.reshape(-1)
    assert flat.size <= R * K
    return np.concatenate([flat, np.zeros(R * K - flat.size, np.uint16)]).reshape(R, K)


def check_groups(host, ref_row_slot, ref_offs, ref_gexp, S):
    G = len(ref_gexp)
    assert host["G"] == G and host["R"] == len(ref_row_slot)
    assert np.array_equal(host["group_expert"].numpy(), ref_gexp)
    assert np.array_equal(host["group_offsets"].numpy(), ref_offs)
    assert np.array_equal(host["row_slot"].numpy(), ref_row_slot)
    assert np.array_equal(host["group_sf_block"].numpy(), O.group_sf_blocks(ref_offs))
    chunks = np.concatenate([[0], np.cumsum((np.diff(ref_offs) + 31) // 32)])
    assert np.array_equal(host["group_chunk"].numpy(), chunks) and host["chunks"] == chunks[-1]
    info = [(ref_offs[g] + 32 * q, min(32, ref_offs[g + 1] - ref_offs[g] - 32 * q), ref_gexp[g], g)
            for g in range(G) for q in range(chunks[g + 1] - chunks[g])]
    assert np.array_equal(host["chunk_info"].numpy(), np.array(info, dtype=np.int64).reshape(-1, 4))
    blocks = O.group_sf_blocks(ref_offs)
    binfo = [(ref_offs[g] + 128 * q, min(128, ref_offs[g + 1] - ref_offs[g] - 128 * q), ref_gexp[g], g)
             for g in range(G) for q in range(blocks[g + 1] - blocks[g])]
    assert np.array_equal(host["block_info"].numpy(), np.array(binfo, dtype=np.int64).reshape(-1, 4))
    assert host["blocks"] == blocks[-1]
    assert host["max_mg"] == (int(np.diff(ref_offs).max()) if G else 0)
    slot_row = np.full(S, -1)
    slot_row[ref_row_slot] = np.arange(len(ref_row_slot))
    assert np.array_equal(host["slot_row"].numpy(), slot_row)


def check_stages_against_oracle(st, x_np, ids_np, tw_np, w_np, E, H, I):
    """Each stage of a run_stages() result against the oracle fed the GPU's
    own inputs for that stage."""
    T, k = ids_np.shape
    row_slot, offs, gexp = O.route_groups(ids_np, E)
    check_groups(st["groups"], row_slot, offs, gexp, T * k)
    R = len(row_slot)
    xg = O.gather_rows(x_np, row_slot, k)
    assert np.array_equal(bf16_to_np(st["xg"])[:R], xg)
    xq, xsf = O.quantize_rows(xg, offs)
    assert np.array_equal(st["xq"][:R].cpu().numpy(), xq)
    want = chunk32_bytes(row_scales(xsf, offs, H), offs, H)
    assert np.array_equal(st["xsf"][:want.size].cpu().numpy(), want)
    d13 = O.grouped_gemm(xq, xsf, offs, gexp, w_np["w13_packed"], w_np["w13_sf_linear"])
    assert rel_fro(st["d13"][:R].cpu().numpy(), d13) <= GEMM_TOL
    assert_swiglu_close(bf16_to_np(st["h"])[:R], st["d13"][:R].cpu().numpy(), offs, gexp, w_np["g_gate_up"])
    h_gpu = bf16_to_np(st["h"])[:R]
    hq, hsf = O.quantize_rows(h_gpu, offs)
    assert np.array_equal(st["hq"][:R].cpu().numpy(), hq)
    want = chunk32_bytes(row_scales(hsf, offs, I), offs, I)
    assert np.array_equal(st["hsf"][:want.size].cpu().numpy(), want)
    d2 = O.grouped_gemm(hq, hsf, offs, gexp, w_np["w2_packed"], w_np["w2_sf_linear"])
    assert rel_fro(st["d2"][:R].cpu().numpy(), d2) <= GEMM_TOL
    assert_scatter_close(bf16_to_np(st["y"]), st["d2"][:R].cpu().numpy(), row_slot, ids_np, tw_np, w_np["g_down"],
                         T, E)
