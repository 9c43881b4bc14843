"""The tcgen05 block-scaled GEMM on every scale value the e4m3 format has.

The first rocket blog page ("Proof") tests the grouped GEMM with constant and
random per-block scales, and its quantizer with the zero / underflow rule (a
block whose scale is 0 has zero codes). Here both GEMM operands carry the
edge cases: weight block-scale codes drawn over all of 0x00 .. 0x7E (zero,
the subnormals 0x01 .. 0x07, small normals, 448), and activation rows whose
token scales are zero, underflowing, subnormal and saturated. Shapes have a
K tail (K % 256 != 0) and groups larger than one 32-row chunk.

Thresholds: quantized codes and scales bit-exact, GEMM outputs within 1e-5
relative Frobenius error of the oracle fed the same NVFP4 inputs (and row by
row), SwiGLU within one bf16 ulp, the layer within 1e-2 and bit-equal to the
separate entry points.
"""
import numpy as np
import pytest
import torch

from nvfp4_block_scaled_gather_gb300 import _native as N
from nvfp4_block_scaled_gather_gb300.synthetic import make_edge_weights
from oracle import nvfp4_moe as O
from tests.gpu_cases import (GEMM_TOL, LAYER_TOL, amax_sweep_blocks, assert_swiglu_close, bf16_to_np, blocks_as_rows,
                             check_stages_against_oracle, chunk32_bytes, edge_rows, np_to_bf16, quotient_sweep_blocks,
                             rel_fro, row_scales, run_stages, weights_from)

pytestmark = pytest.mark.gpu


def _all_codes_present(sf: torch.Tensor):
    codes = set(np.unique(sf.cpu().numpy()).tolist())
    assert codes == set(range(0x7F)), sorted(set(range(0x7F)) - codes)


def _groups_for(mg, cuda):
    ids = torch.cat([torch.full((m,), e, dtype=torch.int32) for e, m in enumerate(mg)]).reshape(-1, 1)
    G = N.Groups(ids.shape[0], 1, len(mg), cuda)
    N.moe_route_groups(ids.to(cuda), len(mg), G)
    return G


def _rowwise_rel(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    num = np.linalg.norm(got - want, axis=1)
    den = np.linalg.norm(want, axis=1)
    zero = den == 0
    assert np.all(num[zero] == 0), "a row the oracle makes exactly zero must be zero"
    return float((num[~zero] / den[~zero]).max()) if (~zero).any() else 0.0


@pytest.mark.parametrize("mg,N_,K", [((40, 1, 140), 256, 320), ((33, 2), 512, 448), ((1,), 128, 64)])
def test_grouped_gemm_edge_scales(cuda, mg, N_, K):
    """Both operands on the edge scale codes; element by element (relative
    Frobenius over all rows, and over every row) against the oracle."""
    E = len(mg)
    R = sum(mg)
    w = make_edge_weights(E, K, N_ // 2, seed=11 + K)   # w13 draw: [E, N_, K]
    packed, sfl = w["w13_packed"], w["w13_sf_linear"]
    if E * N_ * K // 16 >= 4096:
        _all_codes_present(sfl)
    rows = edge_rows(R, K, seed=R + K)
    offs = np.concatenate([[0], np.cumsum(mg)])
    gexp = np.arange(E)
    xq_ref, xsf_ref = O.quantize_rows(rows, offs)
    scales = row_scales(xsf_ref, offs, K)
    assert {0} <= set(np.unique(scales).tolist())           # zero-scale blocks are there
    assert any(1 <= c <= 7 for c in np.unique(scales))      # and subnormal token scales
    assert 0x7E in scales                                   # and saturated ones
    G = _groups_for(mg, cuda)
    xq = torch.zeros(R, K // 2, dtype=torch.uint8, device=cuda)
    xsf = torch.zeros(N.sf_bytes(R, E, K), dtype=torch.uint8, device=cuda)
    N.nvfp4_quantize_rows(np_to_bf16(rows, cuda), G, xq, xsf)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    want_sf = chunk32_bytes(scales, offs, K)
    assert np.array_equal(xsf[:want_sf.size].cpu().numpy(), want_sf)
    ref = O.grouped_gemm(xq_ref, xsf_ref, offs, gexp, packed.numpy(), sfl.numpy())
    # the same rows in 128-row token blocks (the pages' ATOM128 scale layout)
    xq_a = torch.zeros_like(xq)
    xsf_a = torch.zeros(N.sf_bytes(R, E, K, N.SF_ATOM128), dtype=torch.uint8, device=cuda)
    N.nvfp4_quantize_rows(np_to_bf16(rows, cuda), G, xq_a, xsf_a, N.SF_ATOM128)
    assert torch.equal(xq_a, xq) and np.array_equal(xsf_a[:xsf_ref.size].cpu().numpy(), xsf_ref)
    for interleave in ((False, True) if N_ % 256 == 0 else (False,)):
        tw = N.TiledWeight(packed.to(cuda), sfl.to(cuda), interleave=interleave)
        d = torch.full((R, N_), 7.0, dtype=torch.float32, device=cuda)
        N.nvfp4_grouped_gemm(xq, xsf, G, tw, d)
        got = d.cpu().numpy()
        assert rel_fro(got, ref) <= GEMM_TOL, interleave
        assert _rowwise_rel(got, ref) <= GEMM_TOL, interleave
        d_a = torch.full((R, N_), 7.0, dtype=torch.float32, device=cuda)
        N.nvfp4_grouped_gemm(xq_a, xsf_a, G, tw, d_a, layout=N.SF_ATOM128)
        assert torch.equal(d_a, d), interleave
    assert N.check_status() == 0


def test_fused_swiglu_edge_scales(cuda):
    """The w13 GEMM with SwiGLU and requantization in its epilogue, on edge
    weights and edge rows: bit-equal to GEMM -> swiglu_grouped ->
    nvfp4_quantize_rows, and h within one bf16 ulp of the oracle's SwiGLU of
    the GPU's d13."""
    mg, I, K = (40, 1, 70), 256, 320
    E, R = len(mg), sum(mg)
    w = make_edge_weights(E, K, I, seed=5)
    rows = edge_rows(R, K, seed=77)
    offs = np.concatenate([[0], np.cumsum(mg)])
    G = _groups_for(mg, cuda)
    xq = torch.zeros(R, K // 2, dtype=torch.uint8, device=cuda)
    xsf = torch.zeros(N.sf_bytes(R, E, K), dtype=torch.uint8, device=cuda)
    N.nvfp4_quantize_rows(np_to_bf16(rows, cuda), G, xq, xsf)
    w13 = N.TiledWeight(w["w13_packed"].to(cuda), w["w13_sf_linear"].to(cuda), interleave=True)
    g_gate_up = w["g_gate_up"].to(cuda)
    d13 = torch.zeros(R, 2 * I, dtype=torch.float32, device=cuda)
    N.nvfp4_grouped_gemm(xq, xsf, G, w13, d13)
    h = torch.zeros(R, I, dtype=torch.bfloat16, device=cuda)
    N.swiglu_grouped(d13, G, g_gate_up, h)
    hq = torch.zeros(R, I // 2, dtype=torch.uint8, device=cuda)
    hsf = torch.zeros(N.sf_bytes(R, E, I), dtype=torch.uint8, device=cuda)
    N.nvfp4_quantize_rows(h, G, hq, hsf)
    hq2, hsf2 = torch.zeros_like(hq), torch.zeros_like(hsf)
    N.nvfp4_grouped_gemm_swiglu(xq, xsf, G, w13, g_gate_up, hq2, hsf2)
    torch.cuda.synchronize()
    assert torch.equal(hq2, hq) and torch.equal(hsf2, hsf)
    assert_swiglu_close(bf16_to_np(h), d13.cpu().numpy(), offs, np.arange(E), w["g_gate_up"].numpy())
    hq_ref, hsf_ref = O.quantize_rows(bf16_to_np(h), offs)
    assert np.array_equal(hq.cpu().numpy(), hq_ref)
    assert np.array_equal(hsf[:chunk32_bytes(row_scales(hsf_ref, offs, I), offs, I).size].cpu().numpy(),
                          chunk32_bytes(row_scales(hsf_ref, offs, I), offs, I))
    assert N.check_status() == 0


def test_layer_edge_scales(cuda):
    """The whole step on edge weights and edge activations: every stage
    against the oracle (bit-exact codecs, 1e-5 GEMMs, 1 ulp SwiGLU and
    scatter), the layer bit-equal to the stages and within 1e-2 of the
    oracle. Expert 0 takes 45 rows (two 32-row chunks), H and I have K
    tails, some slots are unused."""
    E, H, I, T, k = 4, 384, 384, 48, 2
    g = torch.Generator().manual_seed(9)
    ids = torch.randint(1, E, (T, k), generator=g, dtype=torch.int32)
    ids[:45, 0] = 0
    ids[:, 1] = torch.where(ids[:, 1] == ids[:, 0], (ids[:, 1] % (E - 1)) + 1, ids[:, 1])
    ids[3, 1] = -1
    ids[47, :] = -1
    tw = torch.rand((T, k), generator=g)
    w = make_edge_weights(E, H, I, seed=21)
    _all_codes_present(w["w13_sf_linear"])
    _all_codes_present(w["w2_sf_linear"])
    x_np = edge_rows(T, H, seed=123)
    w_np = {kk: v.numpy() for kk, v in w.items()}
    gpu = {kk: v.to(cuda) for kk, v in w.items()}
    W = weights_from(gpu)
    x, ids_d, tw_d = np_to_bf16(x_np, cuda), ids.to(cuda), tw.to(cuda)
    st = run_stages(x, ids_d, tw_d, W, E)
    check_stages_against_oracle(st, x_np, ids.numpy(), tw.numpy(), w_np, E, H, I)
    y = N.MoeLayer(W, T, k)(x, ids_d, tw_d)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), st["y"].view(torch.int16))
    with np.errstate(over="ignore"):
        ref = O.moe_layer(x_np, ids.numpy(), tw.numpy(), w_np, E)
    assert rel_fro(O.bf16_bits_to_f64(bf16_to_np(y)), O.bf16_bits_to_f64(ref["y"])) <= LAYER_TOL
    assert N.check_status() == 0


# ---------------------------------------------------------------------------
# The device codec does not divide: it converts with the hardware's e4m3 and
# e2m1 conversions, and forms each quotient from an approximate reciprocal
# and one fused multiply-add refinement (Markstein's method). The oracle
# divides (correctly rounded fp32 quotients) and rounds in software. Two
# sweeps hold the two against each other in each kernel that quantizes (the
# row quantizer, the one-launch decode front end, the SwiGLU requantizer):
#   "quotient": every nonzero scale code with every bf16 magnitude from d/8
#       to 6d, both signs and +-0 (every e2m1 threshold of every scale);
#   "amax": every positive finite bf16 block maximum (every e4m3 rounding
#       of amax / 6: subnormal, zero and saturated scales included).
# (The GEMM's fused epilogue calls the same device functions and is held
# bit-equal to the SwiGLU requantizer elsewhere.)
# ---------------------------------------------------------------------------

SWEEPS = {"quotient": quotient_sweep_blocks, "amax": amax_sweep_blocks}


def _sweep_case(sweep, K):
    blocks = SWEEPS[sweep]()
    R = -(-blocks.size // K)
    return blocks, blocks_as_rows(blocks, R, K), R


def _assert_scale_codes(scales, n_blocks, sweep):
    codes = set(np.asarray(scales).reshape(-1)[:n_blocks].tolist())
    assert codes == (set(range(1, 0x7F)) if sweep == "quotient" else set(range(0x7F))), sweep


@pytest.mark.parametrize("sweep", sorted(SWEEPS))
def test_quantizer_codec_sweep(cuda, sweep):
    K = 4096
    blocks, rows, R = _sweep_case(sweep, K)
    mg = (R // 3, R // 3 + 5, R - 2 * (R // 3) - 5)
    offs = np.concatenate([[0], np.cumsum(mg)])
    ref_p, ref_sf = O.quantize_rows(rows, offs)
    scales = row_scales(ref_sf, offs, K)
    _assert_scale_codes(scales, blocks.shape[0], sweep)
    G = _groups_for(mg, cuda)
    for layout in (N.SF_ATOM128, N.SF_CHUNK32):
        packed = torch.zeros(R, K // 2, dtype=torch.uint8, device=cuda)
        sf = torch.zeros(N.sf_bytes(R, len(mg), K, layout), dtype=torch.uint8, device=cuda)
        N.nvfp4_quantize_rows(np_to_bf16(rows, cuda), G, packed, sf, layout)
        assert np.array_equal(packed.cpu().numpy(), ref_p), layout
        want = ref_sf if layout == N.SF_ATOM128 else chunk32_bytes(scales, offs, K)
        assert np.array_equal(sf[:want.size].cpu().numpy(), want), layout
    assert N.check_status() == 0


@pytest.mark.parametrize("sweep", sorted(SWEEPS))
def test_decode_front_end_codec_sweep(cuda, sweep):
    """The one-launch route + gather + quantize (T*k <= 32) on the sweep: 8
    tokens, k = 1, token t routed to expert t, so routed row t is x[t]."""
    T, E = 8, 8
    blocks = SWEEPS[sweep]()
    H = -(-blocks.size // (T * 64)) * 64
    x_np = blocks_as_rows(blocks, T, H)
    offs = np.arange(T + 1)
    ref_p, ref_sf = O.quantize_rows(x_np, offs)
    scales = row_scales(ref_sf, offs, H)
    _assert_scale_codes(scales, blocks.shape[0], sweep)
    ids = torch.arange(T, dtype=torch.int32, device=cuda).reshape(T, 1)
    G = N.Groups(T, 1, E, cuda)
    xq = torch.zeros(T, H // 2, dtype=torch.uint8, device=cuda)
    xsf = torch.zeros(N.sf_bytes(T, E, H, N.SF_CHUNK32), dtype=torch.uint8, device=cuda)
    N.moe_route_gather_quantize(ids, np_to_bf16(x_np, cuda), E, G, xq, xsf)
    assert np.array_equal(xq.cpu().numpy(), ref_p)
    want = chunk32_bytes(scales, offs, H)
    assert np.array_equal(xsf[:want.size].cpu().numpy(), want)
    assert N.check_status() == 0


@pytest.mark.parametrize("sweep", sorted(SWEEPS))
def test_swiglu_requantizer_codec_sweep(cuda, sweep):
    """swiglu_quantize_grouped with gate = 32 and up = v / 32 (globals 1): in
    fp32 and in the oracle silu(32) * (v / 32) rounds to v, so h is the sweep
    itself and its codes must equal the oracle's quantization of the sweep."""
    I = 4096
    blocks, rows, R = _sweep_case(sweep, I)
    mg = (R // 2, R - R // 2)
    E = len(mg)
    offs = np.concatenate([[0], np.cumsum(mg)])
    v = O.bf16_bits_to_f64(rows).astype(np.float32)
    d13 = np.concatenate([np.full((R, I), 32.0, np.float32), v / np.float32(32.0)], axis=1)
    ones = np.ones((E, 2), np.float32)
    assert np.array_equal(O.swiglu(d13, offs, np.arange(E), ones), rows)
    ref_p, ref_sf = O.quantize_rows(rows, offs)
    scales = row_scales(ref_sf, offs, I)
    _assert_scale_codes(scales, blocks.shape[0], sweep)
    G = _groups_for(mg, cuda)
    d13_d, g_d = torch.from_numpy(d13).to(cuda), torch.from_numpy(ones).to(cuda)
    for layout in (N.SF_ATOM128, N.SF_CHUNK32):
        hq = torch.zeros(R, I // 2, dtype=torch.uint8, device=cuda)
        hsf = torch.zeros(N.sf_bytes(R, E, I, layout), dtype=torch.uint8, device=cuda)
        N.swiglu_quantize_grouped(d13_d, G, g_d, hq, hsf, layout)
        assert np.array_equal(hq.cpu().numpy(), ref_p), layout
        want = ref_sf if layout == N.SF_ATOM128 else chunk32_bytes(scales, offs, I)
        assert np.array_equal(hsf[:want.size].cpu().numpy(), want), layout
    assert N.check_status() == 0
