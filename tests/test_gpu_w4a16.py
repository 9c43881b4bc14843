"""The GEMV path (W4A16: exact bf16 activations against NVFP4 weights),
through the C ABI, against the oracle's GEMV path; and how far the grouped
path's activation quantization (W4A4) moves the layer output from it.

Thresholds as for the grouped path: GEMV outputs within a relative Frobenius
error of 1e-5 of the oracle fed the same rows; the layer within 1e-2 (h may
differ from the oracle's by one bf16 ulp); a row's result bit-identical alone
and in its group, and call to call.
"""
import numpy as np
import pytest
import torch

from nvfp4_block_scaled_gather_gb300 import _native as N
from nvfp4_block_scaled_gather_gb300.synthetic import CONFIGS, make_activations, make_routing, make_weights
from oracle import nvfp4_moe as O
from tests.gpu_cases import bf16_to_np, oracle_weights, rel_fro, small_case, weights_from

pytestmark = pytest.mark.gpu

GEMV_TOL = 1e-5
LAYER_TOL = 1e-2


@pytest.fixture(scope="module")
def small(cuda):
    E, x, ids, tw, w = small_case("cpu")
    w_np = {k: v.numpy() for k, v in w.items()}
    gpu = {k: v.to(cuda) for k, v in w.items()}
    return E, x.to(cuda), ids.to(cuda), tw.to(cuda), weights_from(gpu), w_np


def routed(ids, E):
    T, k = ids.shape
    G = N.Groups(T, k, E, ids.device)
    N.moe_route_groups(ids, E, G)
    return G


def test_gemv_gathered_rows_against_oracle(small):
    """w13 (interleaved tiles, N = 2I, K = H) on rows gathered from x by slot:
    several tiles, a 140-row group (many passes), single-row groups."""
    E, x, ids, tw, W, w_np = small
    T, k = ids.shape
    G = routed(ids, E)
    d = torch.zeros(T * k, 2 * W.I, dtype=torch.float32, device=x.device)
    N.nvfp4_grouped_gemv_w4a16(x, G, W.w13, d, src_k=k)
    torch.cuda.synchronize()
    row_slot, offs, gexp = O.route_groups(ids.cpu().numpy(), E)
    R = len(row_slot)
    xg = O.gather_rows(bf16_to_np(x), row_slot, k)
    want = O.grouped_gemv_w4a16(xg, offs, gexp, w_np["w13_packed"], w_np["w13_sf_linear"])
    assert rel_fro(d[:R].cpu().numpy(), want) <= GEMV_TOL


def test_gemv_rows_in_place_and_k_tail(small):
    """w2 (plain tiles, K = I = 384: one and a half K stages) on rows read in
    place (src_k = 0)."""
    E, x, ids, tw, W, w_np = small
    T, k = ids.shape
    G = routed(ids, E)
    g = torch.Generator().manual_seed(3)
    h = (torch.randn((T * k, W.I), generator=g) * 0.1).to(torch.bfloat16).to(x.device)
    d = torch.zeros(T * k, W.H, dtype=torch.float32, device=x.device)
    N.nvfp4_grouped_gemv_w4a16(h, G, W.w2, d)
    torch.cuda.synchronize()
    row_slot, offs, gexp = O.route_groups(ids.cpu().numpy(), E)
    R = len(row_slot)
    want = O.grouped_gemv_w4a16(bf16_to_np(h)[:R], offs, gexp, w_np["w2_packed"], w_np["w2_sf_linear"])
    assert rel_fro(d[:R].cpu().numpy(), want) <= GEMV_TOL


def test_gemv_row_alone_equals_row_in_group(small):
    E, x, ids, tw, W, _ = small
    T, k = ids.shape
    G = routed(ids, E)
    d = torch.zeros(T * k, 2 * W.I, dtype=torch.float32, device=x.device)
    N.nvfp4_grouped_gemv_w4a16(x, G, W.w13, d, src_k=k)
    host = G.host()
    slot_row = host["slot_row"].numpy()
    for t in (0, 5, 139, 150):
        ids1 = ids[t:t + 1].contiguous()
        G1 = routed(ids1, E)
        d1 = torch.zeros(k, 2 * W.I, dtype=torch.float32, device=x.device)
        N.nvfp4_grouped_gemv_w4a16(x[t:t + 1].contiguous(), G1, W.w13, d1, src_k=k)
        h1 = G1.host()
        for j in range(k):
            if ids[t, j] >= 0:
                assert torch.equal(d1[int(h1["slot_row"][j])], d[int(slot_row[t * k + j])]), (t, j)


def test_layer_w4a16_against_oracle_deterministic_batch_invariant(small):
    E, x, ids, tw, W, w_np = small
    layer = N.MoeLayerW4A16(W, x.shape[0], ids.shape[1])
    y = layer(x, ids, tw).clone()
    ref = O.moe_layer_w4a16(bf16_to_np(x), ids.cpu().numpy(), tw.cpu().numpy(), w_np, E)
    assert rel_fro(O.bf16_bits_to_f64(bf16_to_np(y)), O.bf16_bits_to_f64(ref["y"])) <= LAYER_TOL
    for _ in range(3):
        assert torch.equal(layer(x, ids, tw).view(torch.int16), y.view(torch.int16))
    for t in (0, 7, 141, 150):
        yt = layer(x[t:t + 1].contiguous(), ids[t:t + 1].contiguous(), tw[t:t + 1].contiguous())
        assert torch.equal(yt[0].view(torch.int16), y[t].view(torch.int16)), t
    assert N.check_status() == 0


@pytest.fixture(scope="module")
def full_weights(cuda):
    cfg = CONFIGS["decode_m1"]
    w = make_weights(cfg.E, cfg.H, cfg.I, device=cuda)
    return w, weights_from(w), oracle_weights(w)


@pytest.mark.parametrize("name,tokens", [("decode_m1", (0,)), ("decode_m8", (0, 3, 7))])
def test_full_size_w4a16_and_the_grouped_path_against_it(cuda, full_weights, name, tokens):
    """288 experts, hidden 4096, intermediate 2048. The GEMV path against the
    oracle's; then the grouped (W4A4) path's output against the exact-
    activation result: the page measured the two paths' outputs apart
    (max relative logit difference 0.1395 over a whole model) and called the
    gap the arithmetic difference, not noise. Here the gap for one layer is
    printed and held to a loose bound."""
    cfg = CONFIGS[name]
    w, W, w_or = full_weights
    ids, tw = make_routing(cfg)
    x = make_activations(ids.shape[0], cfg.H, device=cuda)
    ids_d, tw_d = ids.to(cuda), tw.to(cuda)
    y16 = N.MoeLayerW4A16(W, ids.shape[0], cfg.k)(x, ids_d, tw_d)
    y4 = N.MoeLayer(W, ids.shape[0], cfg.k)(x, ids_d, tw_d)
    torch.cuda.synchronize()
    x_np, ids_np, tw_np = bf16_to_np(x), ids.numpy(), tw.numpy()
    gaps = []
    for t in tokens:
        ref = O.moe_layer_w4a16(x_np[t:t + 1], ids_np[t:t + 1], tw_np[t:t + 1], w_or, cfg.E)
        want = O.bf16_bits_to_f64(ref["y"])
        assert rel_fro(O.bf16_bits_to_f64(bf16_to_np(y16[t:t + 1])), want) <= LAYER_TOL
        gaps.append(rel_fro(O.bf16_bits_to_f64(bf16_to_np(y4[t:t + 1])), want))
    print(f"\n{name}: W4A4 layer output vs W4A16 (relative Frobenius, per token): "
          + ", ".join(f"{g:.4f}" for g in gaps))
    assert max(gaps) < 0.25
    assert N.check_status() == 0
