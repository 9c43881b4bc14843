"""CUDA path (through the C ABI) against the CPU oracle, step by step and end
to end, at the thresholds the layer is held to:
  * bit-exact: grouping (row order, offsets, group order), gathered rows,
    packed nibbles and scale bytes (padding included), requantized h;
  * grouped GEMM: relative Frobenius error <= 1e-5 against the oracle fed the
    same quantized inputs;
  * SwiGLU h and scatter y: within one bf16 unit in the last place of the
    oracle fed the same GEMM outputs (fp32 on the device, fp64 in the oracle);
  * layer output: relative Frobenius error <= 1e-2 (a 1-ulp difference in h can
    flip an e2m1 code at requantization).
"""
import numpy as np
import pytest
import torch

from nvfp4_block_scaled_gather_gb300 import _native as N
from nvfp4_block_scaled_gather_gb300.synthetic import CONFIGS, make_layer, make_weights, make_activations, \
    make_routing
from oracle import nvfp4_moe as O
from tests.gpu_cases import (GEMM_TOL, LAYER_TOL, assert_swiglu_close, bf16_to_np, check_groups,
                             check_stages_against_oracle, chunk32_bytes, chunk32_row_scales, edge_rows, np_to_bf16,
                             oracle_weights, rel_fro, row_scales, run_stages, small_case, weights_from)

pytestmark = pytest.mark.gpu


def np_inputs(x, ids, tw):
    return bf16_to_np(x), ids.cpu().numpy(), tw.cpu().numpy()


# ---------------------------------------------------------------------------
# tiny config (8 experts, hidden 256, intermediate 128)
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def tiny(cuda):
    cfg = CONFIGS["tiny"]
    inp = make_layer(cfg, device="cpu")
    w_np = {k: inp[k].numpy() for k in ("w13_packed", "w13_sf_linear", "g_gate_up", "w2_packed", "w2_sf_linear",
                                        "g_down")}
    x_np, ids_np, tw_np = np_inputs(inp["x"], inp["topk_ids"], inp["topk_w"])
    ref = O.moe_layer(x_np, ids_np, tw_np, w_np, E=cfg.E)
    gpu = {k: (v.to(cuda) if torch.is_tensor(v) else v) for k, v in inp.items()}
    W = weights_from(gpu)
    return cfg, gpu, W, w_np, (x_np, ids_np, tw_np), ref


def test_tiny_stages(tiny):
    cfg, g, W, w_np, (x_np, ids_np, tw_np), _ = tiny
    st = run_stages(g["x"], g["topk_ids"], g["topk_w"], W, cfg.E)
    check_stages_against_oracle(st, x_np, ids_np, tw_np, w_np, cfg.E, cfg.H, cfg.I)
    assert N.check_status() == 0


def test_tiny_layer_end_to_end(tiny):
    cfg, g, W, _, _, ref = tiny
    layer = N.MoeLayer(W, T_max=g["x"].shape[0], k=cfg.k)
    y = layer(g["x"], g["topk_ids"], g["topk_w"])
    torch.cuda.synchronize()
    assert rel_fro(O.bf16_bits_to_f64(bf16_to_np(y)), O.bf16_bits_to_f64(ref["y"])) <= LAYER_TOL
    assert N.check_status() == 0


def test_tiny_layer_equals_stages(tiny):
    cfg, g, W, *_ = tiny
    st = run_stages(g["x"], g["topk_ids"], g["topk_w"], W, cfg.E)
    y = N.MoeLayer(W, g["x"].shape[0], cfg.k)(g["x"], g["topk_ids"], g["topk_w"])
    assert torch.equal(y.view(torch.int16), st["y"].view(torch.int16))


def test_swizzle_matches_oracle(cuda):
    rng = np.random.default_rng(31)
    for n, kk in ((256, 256), (384, 512), (100, 128)):
        lin = rng.integers(0, 256, (n, kk // 16), dtype=np.uint8)
        out = torch.zeros(((n + 127) // 128) * 128 * kk // 16, dtype=torch.uint8, device=cuda)
        N.nvfp4_swizzle_block_scales(torch.from_numpy(lin).to(cuda), out)
        assert np.array_equal(out.cpu().numpy(), O.swizzle_scales(lin))


def expected_tiled(packed: np.ndarray, sf_linear: np.ndarray, K: int, interleave: int = 0) -> np.ndarray:
    """The GEMM tiling built independently on the host: per 128-row tile and
    256-value stage, rows' 16-byte chunks at chunk c ^ (r % 8), then the
    stage's scale atoms (the oracle's atom layout). interleave = n > 0 first
    reorders every n rows so that tile t holds rows 64t..64t+63 of the first
    half and the same rows of the second half."""
    rows = packed.shape[0]
    if interleave:
        src = []
        for b in range(rows // interleave):
            for t in range(interleave // 128):
                src += [b * interleave + 64 * t + j for j in range(64)]
                src += [b * interleave + interleave // 2 + 64 * t + j for j in range(64)]
        packed, sf_linear = packed[src], sf_linear[src]
    nk, kc4, rowb = (K + 255) // 256, K // 64, K // 2
    pad = np.zeros((rows, nk * 128), np.uint8)
    pad[:, :rowb] = packed
    sw = O.swizzle_scales(sf_linear)
    out = np.zeros(((rows // 128) * nk, 18432), np.uint8)
    r = np.arange(128)
    for t in range(rows // 128):
        for ks in range(nk):
            blk = out[t * nk + ks]
            tile = pad[t * 128:(t + 1) * 128, ks * 128:(ks + 1) * 128].reshape(128, 8, 16)
            img = np.zeros((128, 8, 16), np.uint8)
            for c in range(8):
                img[r, c ^ (r % 8)] = tile[:, c]
            blk[:16384] = img.reshape(-1)
            na = min(4, kc4 - 4 * ks)
            a0 = t * kc4 + 4 * ks
            blk[16384:16384 + na * 512] = sw[a0 * 512:(a0 + na) * 512]
    return out.reshape(-1)


@pytest.mark.parametrize("E,rows,K,il", [(1, 256, 256, False), (1, 128, 384, False), (1, 384, 128, False),
                                         (2, 256, 256, True), (3, 512, 192, True)])
def test_tile_weights_layout(cuda, E, rows, K, il):
    rng = np.random.default_rng(rows + K + E)
    packed = rng.integers(0, 256, (E, rows, K // 2), dtype=np.uint8)
    sfl = rng.integers(0, 256, (E, rows, K // 16), dtype=np.uint8)
    tw = N.TiledWeight(torch.from_numpy(packed).to(cuda), torch.from_numpy(sfl).to(cuda), interleave=il)
    want = expected_tiled(packed.reshape(E * rows, -1), sfl.reshape(E * rows, -1), K, rows if il else 0)
    assert np.array_equal(tw.data.cpu().numpy(), want)


# ---------------------------------------------------------------------------
# codec edge cases, and the pages' group_m = {1, 130} quantizer case
# ---------------------------------------------------------------------------

def _groups_for(mg, cuda):
    """Routing with k = 1 giving groups of the given sizes (experts 0..)."""
    ids = torch.cat([torch.full((m,), e, dtype=torch.int32) for e, m in enumerate(mg)]).reshape(-1, 1)
    G = N.Groups(ids.shape[0], 1, len(mg), cuda)
    N.moe_route_groups(ids.to(cuda), len(mg), G)
    return ids, G


@pytest.mark.parametrize("mg,K", [((1, 130), 64), ((3, 17, 1, 140), 256), ((1,), 4096), ((33, 64, 5), 1024)])
def test_quantize_rows_bit_exact(cuda, mg, K):
    """Both token-scale layouts, every byte (padding included) against the
    oracle; 0xAB fill shows that every byte of the region is written."""
    R = sum(mg)
    rows = edge_rows(R, K, seed=R + K)
    _, G = _groups_for(mg, cuda)
    offs = np.concatenate([[0], np.cumsum(mg)])
    ref_p, ref_sf = O.quantize_rows(rows, offs)
    for layout in (N.SF_ATOM128, N.SF_CHUNK32):
        packed = torch.zeros(R, K // 2, dtype=torch.uint8, device=cuda)
        sf = torch.full((N.sf_bytes(R, len(mg), K, layout),), 0xAB, dtype=torch.uint8, device=cuda)
        N.nvfp4_quantize_rows(np_to_bf16(rows, cuda), G, packed, sf, layout)
        assert np.array_equal(packed.cpu().numpy(), ref_p)
        want = ref_sf if layout == N.SF_ATOM128 else chunk32_bytes(row_scales(ref_sf, offs, K), offs, K)
        assert np.array_equal(sf[:want.size].cpu().numpy(), want), layout
    if mg == (1, 130):
        assert ref_p.nbytes + ref_sf.nbytes == 5728


def test_gather_quantize_fused_equals_separate(cuda):
    E, x, ids, tw, w = small_case("cpu")
    x, ids = x.to(cuda), ids.to(cuda)
    T, H = x.shape
    k, S = ids.shape[1], ids.numel()
    G = N.Groups(T, k, E, cuda)
    xg = torch.zeros(S, H, dtype=torch.bfloat16, device=cuda)
    N.moe_gather_rows(x, ids, E, G, xg)
    for layout in (N.SF_ATOM128, N.SF_CHUNK32):
        p1 = torch.zeros(S, H // 2, dtype=torch.uint8, device=cuda)
        s1 = torch.zeros(N.sf_bytes(S, E, H, layout), dtype=torch.uint8, device=cuda)
        p2, s2 = p1.clone(), s1.clone()
        N.nvfp4_quantize_rows(xg, G, p1, s1, layout)
        N.moe_gather_quantize_rows(x, k, G, p2, s2, layout)
        assert torch.equal(p1, p2) and torch.equal(s1, s2)


# ---------------------------------------------------------------------------
# several tiles, ragged tails, a group spanning two 128-row blocks
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def small(cuda):
    E, x, ids, tw, w = small_case("cpu")
    w_np = {k: v.numpy() for k, v in w.items()}
    gpu = {k: v.to(cuda) for k, v in w.items()}
    return E, x.to(cuda), ids.to(cuda), tw.to(cuda), weights_from(gpu), w_np, np_inputs(x, ids, tw)


def test_small_stages(small):
    E, x, ids, tw, W, w_np, (x_np, ids_np, tw_np) = small
    st = run_stages(x, ids, tw, W, E)
    check_stages_against_oracle(st, x_np, ids_np, tw_np, w_np, E, W.H, W.I)


def test_small_layer_end_to_end(small):
    E, x, ids, tw, W, w_np, (x_np, ids_np, tw_np) = small
    y = N.MoeLayer(W, x.shape[0], ids.shape[1])(x, ids, tw)
    ref = O.moe_layer(x_np, ids_np, tw_np, w_np, E)
    assert rel_fro(O.bf16_bits_to_f64(bf16_to_np(y)), O.bf16_bits_to_f64(ref["y"])) <= LAYER_TOL
    # a token with every slot unused gets zeros; check_status stays clean
    assert N.check_status() == 0


def test_gemm_row_invariance_and_fused_w13(small):
    """First page, "Proof": a row alone equals the same row paired; fused w13
    equals separate gate-only and up-only GEMMs; five calls bit-identical.
    Here also across MMA widths: the 140-row group runs a 128-wide and a
    16-wide MMA, the row alone a 16-wide one."""
    E, x, ids, tw, W, w_np, _ = small
    small_w = {k: torch.from_numpy(v).to(x.device) for k, v in w_np.items()}
    st = run_stages(x, ids, tw, W, E)
    dev = x.device
    I = W.I
    hostg = st["groups"]
    # rows of expert 0 (group 0, 140 rows): compare row 0, row 127, row 130 alone
    for r in (0, 127, 130, 139):
        xa = st["xg"][r:r + 1]
        G1 = N.Groups(1, 1, E, dev)
        N.moe_route_groups(torch.zeros((1, 1), dtype=torch.int32, device=dev), E, G1)
        q = torch.zeros(1, W.H // 2, dtype=torch.uint8, device=dev)
        s = torch.zeros(N.sf_bytes(1, E, W.H), dtype=torch.uint8, device=dev)
        N.nvfp4_quantize_rows(xa, G1, q, s)
        d = torch.zeros(1, 2 * I, dtype=torch.float32, device=dev)
        N.nvfp4_grouped_gemm(q, s, G1, W.w13, d)
        assert torch.equal(d[0], st["d13"][r]), r
    # fused w13 == gate-only and up-only GEMMs (each half tiled on its own)
    G = N.Groups(x.shape[0], ids.shape[1], E, dev)
    N.moe_route_groups(ids, E, G)
    R_max = ids.numel()
    w = small_w
    gate_w = N.TiledWeight(w["w13_packed"][:, :I].contiguous(), w["w13_sf_linear"][:, :I].contiguous())
    up_w = N.TiledWeight(w["w13_packed"][:, I:].contiguous(), w["w13_sf_linear"][:, I:].contiguous())
    gate = torch.zeros(R_max, I, dtype=torch.float32, device=dev)
    up = torch.zeros(R_max, I, dtype=torch.float32, device=dev)
    N.nvfp4_grouped_gemm(st["xq"], st["xsf"], G, gate_w, gate)
    N.nvfp4_grouped_gemm(st["xq"], st["xsf"], G, up_w, up)
    R = hostg["R"]
    assert torch.equal(torch.cat([gate, up], 1)[:R], st["d13"][:R])
    for _ in range(5):
        d = torch.zeros_like(st["d13"])
        N.nvfp4_grouped_gemm(st["xq"], st["xsf"], G, W.w13, d)
        assert torch.equal(d[:R], st["d13"][:R])


def test_swiglu_requant_fused_equals_separate(small):
    E, x, ids, tw, W, *_ = small
    st = run_stages(x, ids, tw, W, E)
    G = N.Groups(x.shape[0], ids.shape[1], E, x.device)
    N.moe_route_groups(ids, E, G)
    p = torch.zeros_like(st["hq"])
    s = torch.zeros_like(st["hsf"])
    N.swiglu_quantize_grouped(st["d13"], G, W.g_gate_up, p, s)
    R = st["groups"]["R"]
    assert torch.equal(p[:R], st["hq"][:R]) and torch.equal(s, st["hsf"])
    # the w13 GEMM with SwiGLU + requantization in its epilogue equals the
    # separate GEMM, SwiGLU and quantize kernels, nibbles and scales
    for _ in range(3):
        p2 = torch.zeros_like(st["hq"])
        s2 = torch.zeros_like(st["hsf"])
        N.nvfp4_grouped_gemm_swiglu(st["xq"], st["xsf"], G, W.w13, W.g_gate_up, p2, s2)
        assert torch.equal(p2[:R], st["hq"][:R]) and torch.equal(s2, st["hsf"])


@pytest.mark.parametrize("T,k,E,pattern", [(1, 8, 288, "topk"), (4, 8, 288, "topk"), (2, 8, 16, "topk"),
                                           (8, 4, 8, "one_expert"), (4, 8, 64, "unused"), (3, 2, 4, "all_unused"),
                                           (5, 8, 288, "topk"), (32, 1, 288, "one_expert")])
def test_route_gather_quantize_small_path(cuda, T, k, E, pattern):
    """T*k <= 32 takes the one-launch path (one warp routes, the CTA
    quantizes); its group tables, packed rows and token scales equal those of
    moe_route_groups + moe_gather_quantize_rows byte for byte. T*k = 40 runs
    the two-launch path inside the same entry point."""
    H = 256
    g = torch.Generator().manual_seed(T * 131 + k * 7 + E)
    if pattern == "topk":
        ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    elif pattern == "one_expert":
        ids = torch.full((T, k), 3, dtype=torch.int32)
    elif pattern == "unused":
        ids = torch.randint(-2, E + 3, (T, k), generator=g, dtype=torch.int32)
    else:
        ids = torch.full((T, k), -1, dtype=torch.int32)
    if pattern == "one_expert" and k > 1:
        ids[:, 1:] = torch.arange(1, k, dtype=torch.int32) + 3
    x = (torch.randn(T, H, generator=g) * 3).to(torch.bfloat16).to(cuda)
    ids = ids.to(cuda)
    S = T * k
    outs = []
    for one_launch in (True, False):
        G = N.Groups(T, k, E, cuda)
        xq = torch.full((S, H // 2), 0xAB, dtype=torch.uint8, device=cuda)
        xsf = torch.full((N.sf_bytes(S, E, H, N.SF_CHUNK32),), 0xCD, dtype=torch.uint8, device=cuda)
        if one_launch:
            N.moe_route_gather_quantize(ids, x, E, G, xq, xsf)
        else:
            N.moe_route_groups(ids, E, G)
            N.moe_gather_quantize_rows(x, k, G, xq, xsf)
        torch.cuda.synchronize()
        h = G.host()
        nbytes = h["chunks"] * (H // 64) * 512
        outs.append((h, xq[:h["R"]].cpu(), xsf[:nbytes].cpu()))
    (h1, q1, s1), (h2, q2, s2) = outs
    for key in ("G", "R", "max_mg", "blocks", "chunks"):
        assert h1[key] == h2[key], key
    for key in ("group_offsets", "group_expert", "group_sf_block", "group_chunk", "chunk_info", "row_slot",
                "slot_row"):
        assert torch.equal(h1[key], h2[key]), key
    assert torch.equal(q1, q2) and torch.equal(s1, s2)


def test_expert_gemms_one_launch_equals_two(small):
    """Both grouped GEMMs in one persistent launch (w2 units gated per chunk
    on h) give the same h and d2 bits as the two launches run one after the
    other; repeated calls agree (the work counters are re-zeroed per call)."""
    E, x, ids, tw, W, *_ = small
    st = run_stages(x, ids, tw, W, E)
    dev = x.device
    G = N.Groups(x.shape[0], ids.shape[1], E, dev)
    N.moe_route_groups(ids, E, G)
    R = st["groups"]["R"]
    gate = torch.zeros(N.expert_gemms_gate_bytes(st["xq"].shape[0], E, W.I), dtype=torch.uint8, device=dev)
    for _ in range(3):
        hq = torch.zeros_like(st["hq"])
        hsf = torch.zeros_like(st["hsf"])
        d2 = torch.zeros_like(st["d2"])
        N.nvfp4_moe_expert_gemms(st["xq"], st["xsf"], G, W, hq, hsf, d2, gate)
        torch.cuda.synchronize()
        assert torch.equal(hq[:R], st["hq"][:R]) and torch.equal(hsf, st["hsf"])
        assert torch.equal(d2[:R], st["d2"][:R])
    assert N.check_status() == 0


def test_128_row_token_blocks_equal_32_row_chunks(small):
    """The same GEMMs over 128-row token blocks (MOE_SF_ATOM128 scales: one
    unit per weight tile for the 140-row group's first 128 rows, MMA N = 128)
    give the bits of the 32-row chunks: plain w13 and w2, the fused SwiGLU
    epilogue (h scales written in the 128-row layout, equal to the quantizer's
    ATOM128 output), and the one-launch pair of GEMMs."""
    E, x, ids, tw, W, *_ = small
    st = run_stages(x, ids, tw, W, E)
    dev = x.device
    T, k = ids.shape
    S, R = T * k, st["groups"]["R"]
    G = N.Groups(T, k, E, dev)
    N.moe_route_groups(ids, E, G)
    A = N.SF_ATOM128
    xsf = torch.zeros(N.sf_bytes(S, E, W.H, A), dtype=torch.uint8, device=dev)
    xq = torch.zeros_like(st["xq"])
    N.nvfp4_quantize_rows(st["xg"], G, xq, xsf, A)
    hsf_ref = torch.zeros(N.sf_bytes(S, E, W.I, A), dtype=torch.uint8, device=dev)
    hq_ref = torch.zeros_like(st["hq"])
    N.nvfp4_quantize_rows(st["h"], G, hq_ref, hsf_ref, A)
    for _ in range(2):
        d13 = torch.zeros_like(st["d13"])
        N.nvfp4_grouped_gemm(xq, xsf, G, W.w13, d13, layout=A)
        d2 = torch.zeros_like(st["d2"])
        N.nvfp4_grouped_gemm(hq_ref, hsf_ref, G, W.w2, d2, layout=A)
        hq, hsf = torch.zeros_like(hq_ref), torch.full_like(hsf_ref, 0xAB)
        N.nvfp4_grouped_gemm_swiglu(xq, xsf, G, W.w13, W.g_gate_up, hq, hsf, layout=A)
        torch.cuda.synchronize()
        assert torch.equal(d13[:R], st["d13"][:R]) and torch.equal(d2[:R], st["d2"][:R])
        routed = G.host()["blocks"] * 128 * (W.I // 16)   # every byte of the routed blocks' regions
        assert torch.equal(hq[:R], st["hq"][:R]) and torch.equal(hsf[:routed], hsf_ref[:routed])
    gate = torch.zeros(N.expert_gemms_gate_bytes(S, E, W.I), dtype=torch.uint8, device=dev)
    for _ in range(3):
        hq, hsf, d2 = torch.zeros_like(hq_ref), torch.zeros_like(hsf_ref), torch.zeros_like(st["d2"])
        N.nvfp4_moe_expert_gemms(xq, xsf, G, W, hq, hsf, d2, gate, layout=A)
        torch.cuda.synchronize()
        assert torch.equal(hq[:R], st["hq"][:R]) and torch.equal(hsf, hsf_ref)
        assert torch.equal(d2[:R], st["d2"][:R])
    assert int(gate.sum()) == 0
    assert N.check_status() == 0


def test_bounded_wait_reports_timeout_and_the_context_survives(small):
    """Failure detection without a fault: start the two-GEMM launch's claim
    counter past every w13 unit, so no chunk's h is ever published and every
    w2 unit's wait runs out (about a second of clock64). The kernel records
    MOE_ERR_TIMEOUT, lets its own copies land, frees tensor memory and
    returns; moe_nvfp4_check_status reports it once, and the next call on the
    same context and counters is correct again."""
    E, x, ids, tw, W, *_ = small
    st = run_stages(x, ids, tw, W, E)
    dev = x.device
    G = N.Groups(x.shape[0], ids.shape[1], E, dev)
    N.moe_route_groups(ids, E, G)
    chunks = G.host()["chunks"]
    R = st["groups"]["R"]
    S = st["xq"].shape[0]
    gate = torch.zeros(N.expert_gemms_gate_bytes(S, E, W.I) // 4, dtype=torch.int32, device=dev)
    assert N.check_status() == 0
    gate[0] = chunks * (2 * W.I // 128)          # claims start at the first w2 unit
    hq, hsf, d2 = torch.zeros_like(st["hq"]), torch.zeros_like(st["hsf"]), torch.zeros_like(st["d2"])
    N.nvfp4_moe_expert_gemms(st["xq"], st["xsf"], G, W, hq, hsf, d2, gate)
    torch.cuda.synchronize()
    assert N.check_status() == 4                  # MOE_ERR_TIMEOUT, read and cleared
    assert N.check_status() == 0
    assert int(gate.abs().sum()) == 0             # the last CTA out left the counters zero
    N.nvfp4_moe_expert_gemms(st["xq"], st["xsf"], G, W, hq, hsf, d2, gate)
    torch.cuda.synchronize()
    assert torch.equal(hq[:R], st["hq"][:R]) and torch.equal(d2[:R], st["d2"][:R])
    assert N.check_status() == 0


def test_back_to_back_calls_share_a_workspace(small):
    """Layer calls queued back to back (no host sync) on one workspace,
    alternating the one-launch small-batch front end (T*k <= 32), the
    general one (route, then gather+quantize) with 32-row token chunks and
    with 128-row token blocks (the one-CTA-per-SM GEMM): every call's output
    equals the same call run alone. Kernels start before the one they depend on ends
    (programmatic dependent launch), so a read of an earlier kernel's output
    that could hit a stale cached line shows up here."""
    E, x, ids, tw, W, *_ = small
    cases = {n: (x[:n].contiguous(), ids[:n].contiguous(), tw[:n].contiguous()) for n in (3, 40, 60)}
    assert N.layer_sf_layout(60, ids.shape[1], E) == N.SF_ATOM128     # 128-row blocks, one CTA per SM
    assert N.layer_sf_layout(40, ids.shape[1], E) == N.SF_CHUNK32
    refs = {n: N.MoeLayer(W, n, ids.shape[1])(*c).clone() for n, c in cases.items()}
    torch.cuda.synchronize()
    ws = torch.zeros(max(N.moe_nvfp4_layer_workspace_size(n, ids.shape[1], E, W.H, W.I) for n in cases),
                     dtype=torch.uint8, device=x.device)
    outs = []
    for _ in range(5):
        for n in (40, 3, 60, 3, 40, 60, 60, 3):
            y = torch.empty_like(cases[n][0])
            N.moe_nvfp4_layer(*cases[n], W, ws, y)
            outs.append((n, y))
    torch.cuda.synchronize()
    for n, y in outs:
        assert torch.equal(y.view(torch.int16), refs[n].view(torch.int16)), n
    assert N.check_status() == 0


def test_layer_determinism_and_batch_invariance(small):
    E, x, ids, tw, W, *_ = small
    layer = N.MoeLayer(W, x.shape[0], ids.shape[1])
    y0 = layer(x, ids, tw).clone()
    for _ in range(4):
        assert torch.equal(layer(x, ids, tw).view(torch.int16), y0.view(torch.int16))
    for t in (0, 7, 100, 141, 150, 159):
        yt = layer(x[t:t + 1].contiguous(), ids[t:t + 1].contiguous(), tw[t:t + 1].contiguous())
        assert torch.equal(yt[0].view(torch.int16), y0[t].view(torch.int16)), t


@pytest.mark.parametrize("T,k,seed", [(1, 8, 0), (4, 8, 1), (32, 1, 2), (1, 32, 3), (3, 5, 4), (16, 2, 5)])
def test_decode_layer_equals_stages(small, T, k, seed):
    """Decode batches (T*k <= 32: the one-launch front end, in-kernel routing
    in the GEMM launch) give the separate entry points' bits for any routing:
    repeated experts in a token, unused slots, tokens with no rows, one slot
    per token or 32 for one."""
    E, _, _, _, W, *_ = small
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(100 + seed)
    ids = torch.randint(-1, E, (T, k), generator=g, dtype=torch.int32)
    if T > 1:
        ids[T - 1] = -1                  # a token with no rows
    tw = torch.rand((T, k), generator=g)
    x = (torch.randn((T, W.H), generator=g)).to(torch.bfloat16)
    x, ids, tw = x.to(dev), ids.to(dev), tw.to(dev)
    y = torch.full((T, W.H), 3.0, dtype=torch.bfloat16, device=dev)
    N.MoeLayer(W, T, k)(x, ids, tw, y)
    st = run_stages(x, ids, tw, W, E)
    assert torch.equal(y.view(torch.int16), st["y"].view(torch.int16))
    assert N.check_status() == 0


def test_graph_replay_matches_direct_call(small):
    """The layer step captured as a CUDA graph (PDL edges included) gives the
    same bits as the direct call, before and after its inputs are refilled."""
    E, x, ids, tw, W, *_ = small
    layer = N.MoeLayer(W, x.shape[0], ids.shape[1])
    want = layer(x, ids, tw).clone()
    xb, ib, wb, yb = x.clone(), ids.clone(), tw.clone(), torch.empty_like(x)
    g = layer.capture(xb, ib, wb, yb)
    yb.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(yb.view(torch.int16), want.view(torch.int16))
    xb.copy_(torch.flip(x, [0]))
    ib.copy_(torch.flip(ids, [0]))
    wb.copy_(torch.flip(tw, [0]))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(yb.view(torch.int16), torch.flip(want, [0]).view(torch.int16))


def test_unused_slots_and_empty(cuda, tiny):
    cfg, g, W, *_ = tiny
    x = g["x"]
    ids = torch.full_like(g["topk_ids"], -1)
    y = torch.full_like(x, 7.0)
    N.MoeLayer(W, x.shape[0], cfg.k)(x, ids, g["topk_w"], y)
    assert not y.float().abs().sum().item()
    # T = 0 is a no-op
    N.moe_nvfp4_layer(x[:0], g["topk_ids"][:0], g["topk_w"][:0], W, torch.empty(256, dtype=torch.uint8,
                                                                                   device=cuda), x[:0])
    assert N.check_status() == 0


# ---------------------------------------------------------------------------
# full-size layer (288 experts, hidden 4096, intermediate 2048): every step at
# the configs' sizes, checked on sampled tokens against the oracle run on those
# tokens alone (valid because a token's output does not depend on the batch)
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def full_weights(cuda):
    cfg = CONFIGS["decode_m1"]
    w = make_weights(cfg.E, cfg.H, cfg.I, device=cuda)
    return w, weights_from(w), oracle_weights(w)


def _token_check(t, x_np, ids_np, tw_np, w_or, E, gpu_y, gpu_st=None):
    ref = O.moe_layer(x_np[t:t + 1], ids_np[t:t + 1], tw_np[t:t + 1], w_or, E)
    assert rel_fro(O.bf16_bits_to_f64(bf16_to_np(gpu_y[t:t + 1])), O.bf16_bits_to_f64(ref["y"])) <= LAYER_TOL
    if gpu_st is not None:
        # every stage of the token's rows at full size: K = 4096 for w13 and
        # K = 2048 (eight stages, gated per stage on h in the layer) for w2
        k = ids_np.shape[1]
        H2, I2 = gpu_st["xq"].shape[1], gpu_st["hq"].shape[1]
        info = gpu_st["groups"]["chunk_info"].numpy()
        slot_row = gpu_st["groups"]["slot_row"].numpy()
        rows = [int(slot_row[t * k + s]) for s in ref["row_slot"]]
        offs1 = ref["group_offsets"]            # the token alone: one row per group
        assert np.array_equal(gpu_st["xq"][rows].cpu().numpy(), ref["xq"])
        assert np.array_equal(chunk32_row_scales(gpu_st["xsf"].cpu().numpy(), info, rows, 2 * H2),
                              row_scales(ref["xsf"], offs1, 2 * H2))
        assert rel_fro(gpu_st["d13"][rows].cpu().numpy(), ref["d13"]) <= GEMM_TOL
        # SwiGLU of the GPU's d13 within one bf16 ulp; requantization of the
        # GPU's h bit-exact; w2 against the oracle fed those NVFP4 rows
        h_gpu = bf16_to_np(gpu_st["h"])[rows]
        assert_swiglu_close(h_gpu, gpu_st["d13"][rows].cpu().numpy(), offs1, ref["group_expert"], w_or["g_gate_up"])
        hq, hsf = O.quantize_rows(h_gpu, offs1)
        assert np.array_equal(gpu_st["hq"][rows].cpu().numpy(), hq)
        assert np.array_equal(chunk32_row_scales(gpu_st["hsf"].cpu().numpy(), info, rows, 2 * I2),
                              row_scales(hsf, offs1, 2 * I2))
        d2 = O.grouped_gemm(hq, hsf, offs1, ref["group_expert"], w_or["w2_packed"], w_or["w2_sf_linear"])
        assert rel_fro(gpu_st["d2"][rows].cpu().numpy(), d2) <= GEMM_TOL


@pytest.mark.parametrize("name,tokens", [("decode_m1", (0,)), ("decode_m8", (0, 5)), ("decode_m32", (3, 31)),
                                         ("full_stream", (0, 40)), ("large_batch", (1, 150, 287)),
                                         ("prefill_m32", (0, 600, 1100))])
def test_full_size_layer(cuda, full_weights, name, tokens):
    cfg = CONFIGS[name]
    w, W, w_or = full_weights
    ids, tw = make_routing(cfg)
    x = make_activations(ids.shape[0], cfg.H, device=cuda)
    ids_d, tw_d = ids.to(cuda), tw.to(cuda)
    y = N.MoeLayer(W, ids.shape[0], cfg.k)(x, ids_d, tw_d)
    st = run_stages(x, ids_d, tw_d, W, cfg.E)
    assert torch.equal(y.view(torch.int16), st["y"].view(torch.int16))
    x_np, ids_np, tw_np = np_inputs(x, ids, tw)
    row_slot, offs, gexp = O.route_groups(ids_np, cfg.E)
    check_groups(st["groups"], row_slot, offs, gexp, ids.numel())
    for t in tokens:
        _token_check(t, x_np, ids_np, tw_np, w_or, cfg.E, y, st)
    assert N.check_status() == 0


@pytest.mark.parametrize("n", [1, 3, 40, 60])
def test_layer_reads_and_writes_pinned_host_buffers(small, n):
    """x, the routing, the router weights and y may sit in pinned host memory
    (unified addressing: the kernels read and write them over the CPU-GPU
    link): the same bits as the call on device buffers, for the one-launch
    decode front end (n = 1, 3) and the general path with 32-row (40) and
    128-row (60) token blocks."""
    E, x, ids, tw, W, *_ = small
    k = ids.shape[1]
    xd, idd, twd = x[:n].contiguous(), ids[:n].contiguous(), tw[:n].contiguous()
    layer = N.MoeLayer(W, n, k)
    want = layer(xd, idd, twd).clone()
    hx, hi, hw = xd.cpu().pin_memory(), idd.cpu().pin_memory(), twd.cpu().pin_memory()
    hy = torch.full_like(hx, 7.0).pin_memory()
    layer(hx, hi, hw, hy)
    torch.cuda.synchronize()
    assert torch.equal(hy.view(torch.int16), want.cpu().view(torch.int16))
    assert N.check_status() == 0


@pytest.mark.parametrize("n", [3, 40, 60])
def test_layer_ignores_workspace_contents(small, n):
    """The workspace may hold anything (the header's "any contents"): filled
    with 0xFF bytes first (NaN e4m3 scale codes, NaN-pattern codes and
    counters far past their ends), every call gives the bits of a call on a
    zeroed workspace; the token-scale padding a step never writes only feeds
    accumulator columns no result reads."""
    E, x, ids, tw, W, *_ = small
    k = ids.shape[1]
    c = (x[:n].contiguous(), ids[:n].contiguous(), tw[:n].contiguous())
    size = N.moe_nvfp4_layer_workspace_size(n, k, E, W.H, W.I)
    ws0 = torch.zeros(size, dtype=torch.uint8, device=x.device)
    want = torch.empty_like(c[0])
    N.moe_nvfp4_layer(*c, W, ws0, want)
    ws = torch.full((size,), 0xFF, dtype=torch.uint8, device=x.device)
    for _ in range(2):
        y = torch.empty_like(c[0])
        N.moe_nvfp4_layer(*c, W, ws, y)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), want.view(torch.int16))
        ws.fill_(0xFF)
    assert N.check_status() == 0


@pytest.mark.parametrize("E,H,I,T,k,seed", [(3, 256, 128, 1, 1, 0), (8, 384, 256, 5, 2, 1), (5, 640, 384, 17, 4, 2),
                                            (16, 256, 384, 40, 3, 3), (4, 512, 128, 70, 1, 4),
                                            (12, 384, 640, 9, 8, 5)])
def test_layer_over_shapes(cuda, E, H, I, T, k, seed):
    """The layer over a spread of shapes (K tails in both GEMMs, 1 to 12
    token blocks per expert, decode and general paths, top-1 to top-8):
    the separate entry points' bits and within 1e-2 of the oracle."""
    from nvfp4_block_scaled_gather_gb300.synthetic import make_weights as mw
    g = torch.Generator().manual_seed(1000 + seed)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    ids[torch.rand((T, k), generator=g) < 0.1] = -1                   # some unused slots
    tw = torch.rand((T, k), generator=g)
    x = torch.randn((T, H), generator=g).to(torch.bfloat16)
    w = mw(E, H, I, seed=seed)
    w_np = {kk: v.numpy() for kk, v in w.items()}
    W = weights_from({kk: v.to(cuda) for kk, v in w.items()})
    xd, idd, twd = x.to(cuda), ids.to(cuda), tw.to(cuda)
    y = N.MoeLayer(W, T, k)(xd, idd, twd)
    st = run_stages(xd, idd, twd, W, E)
    assert torch.equal(y.view(torch.int16), st["y"].view(torch.int16))
    ref = O.moe_layer(bf16_to_np(x), ids.numpy(), tw.numpy(), w_np, E=E)
    assert rel_fro(O.bf16_bits_to_f64(bf16_to_np(y)), O.bf16_bits_to_f64(ref["y"])) <= LAYER_TOL
    assert N.check_status() == 0
