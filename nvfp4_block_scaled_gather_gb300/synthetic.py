"""Seeded synthetic workloads for the NVFP4 routed-expert MoE layer.

This module draws random inputs and nothing else: it holds no part of the
layer's arithmetic (no e2m1/e4m3 codec, no grouping, no GEMM). Both the CUDA
path and the CPU oracle are fed from here.

Workload shapes follow the two rocket blog pages:
  * "Fusing the MoE layer's two grouped GEMMs is worth 4%", table "Bytes decide
    it before the kernel runs": 288 experts, hidden 4096, intermediate 2048,
    w13 = 4096 x 4096 and w2 = 4096 x 2048 per expert, NVFP4 (0.5 + 1/16 B/elt).
  * same page, "Tiles below M=8": all 288 experts active with ragged row
    counts around means 2 / 4 / 8 (570 / 1145 / 2303 rows).
  * "Grouped GEMM beats GEMV at every M", "Numbers": M = 1..8 decode streams,
    each routed top-8.
  * same page 2, "Different globals on the two halves": gate and up
    weight_scale_2 differ, 4.650e-05 vs 3.778e-05 (ratio 1.2308).

Weights are drawn directly in NVFP4 code space: uniform e2m1 nibbles (all 16
codes), e4m3 block-scale codes uniform over 0x58..0x7E (16 .. 448), and
per-expert fp32 globals scattered around the pages' measured values. Drawing
codes (instead of quantizing Gaussian weights) keeps every codec out of this
shared module; the byte counts and layouts, which are what the weight stream
measures, are identical.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

# Global scale of the gate half on the pages' layer 10, and the gate/up ratio.
GATE_GLOBAL = 4.650e-05
GATE_UP_RATIO = 1.2308
DOWN_GLOBAL = 4.2e-05
SCALE_CODE_LO = 0x58  # e4m3 code of 16.0
SCALE_CODE_HI = 0x7E  # e4m3 code of 448.0 (largest finite)

SEED_WEIGHTS = 0
SEED_ACTIVATIONS = 1
SEED_ROUTING = 2


@dataclass(frozen=True)
class LayerConfig:
    name: str
    E: int
    H: int
    I: int
    k: int
    routing: str  # "topk": T streams routed top-k from N(0,1) logits
    #              "all_experts": every expert gets Mg ~ U{mg_lo..mg_hi} rows
    T: int = 0
    mg_lo: int = 1
    mg_hi: int = 1
    router_weights: str = "softmax"  # "softmax" over the top-k logits, or "uniform" U(0,1)


CONFIGS = {
    "tiny": LayerConfig("tiny", E=8, H=256, I=128, k=2, routing="topk", T=4),
    "decode_m1": LayerConfig("decode_m1", E=288, H=4096, I=2048, k=8, routing="topk", T=1),
    "decode_m8": LayerConfig("decode_m8", E=288, H=4096, I=2048, k=8, routing="topk", T=8),
    "full_stream": LayerConfig("full_stream", E=288, H=4096, I=2048, k=8, routing="all_experts",
                               mg_lo=1, mg_hi=3, router_weights="uniform"),
    "large_batch": LayerConfig("large_batch", E=288, H=4096, I=2048, k=8, routing="all_experts",
                               mg_lo=1, mg_hi=15, router_weights="uniform"),
    "decode_m32": LayerConfig("decode_m32", E=288, H=4096, I=2048, k=8, routing="topk", T=32),
    # prefill-sized: every expert Mg ~ U{16..48} rows (mean 32, ~9216 rows, ~1152 tokens)
    "prefill_m32": LayerConfig("prefill_m32", E=288, H=4096, I=2048, k=8, routing="all_experts",
                               mg_lo=16, mg_hi=48, router_weights="uniform"),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_weights(E: int, H: int, I: int, seed: int = SEED_WEIGHTS, device="cpu") -> dict:
    """NVFP4 expert weights with linear (row-major) block scales.

    w13_packed [E, 2I, H/2] u8: rows 0..I-1 are gate, I..2I-1 are up, two e2m1
        nibbles per byte.
    w13_sf_linear [E, 2I, H/16] u8: one e4m3 code per 16 elements of a row.
    g_gate_up [E, 2] f32: (gate global, up global).
    w2_packed [E, H, I/2] u8, w2_sf_linear [E, H, I/16] u8, g_down [E] f32.
    """
    g = _gen(seed, device)
    u8 = dict(dtype=torch.uint8, device=device, generator=g)
    w13 = torch.randint(0, 256, (E, 2 * I, H // 2), **u8)
    w13_sf = torch.randint(SCALE_CODE_LO, SCALE_CODE_HI + 1, (E, 2 * I, H // 16), **u8)
    w2 = torch.randint(0, 256, (E, H, I // 2), **u8)
    w2_sf = torch.randint(SCALE_CODE_LO, SCALE_CODE_HI + 1, (E, H, I // 16), **u8)
    z = torch.randn((E, 2), dtype=torch.float32, device=device, generator=g)
    g_gate = GATE_GLOBAL * torch.exp(0.05 * z[:, 0])
    g_gate_up = torch.stack([g_gate, g_gate / GATE_UP_RATIO], dim=1).contiguous()
    g_down = (DOWN_GLOBAL * torch.exp(0.05 * z[:, 1])).contiguous()
    return dict(w13_packed=w13, w13_sf_linear=w13_sf, g_gate_up=g_gate_up,
                w2_packed=w2, w2_sf_linear=w2_sf, g_down=g_down)


def make_edge_weights(E: int, H: int, I: int, seed: int = SEED_WEIGHTS, device="cpu") -> dict:
    """Expert weights as make_weights, but with e4m3 block-scale codes drawn
    uniformly over every finite non-negative code, 0x00 .. 0x7E: a zero scale
    (the whole 16-value block is zero), the subnormals 0x01 .. 0x07
    (m * 2^-9), the small normals and the largest value (448). The first
    rocket blog page ("Proof") tests with constant and random per-block
    scales; this draw puts every scale value the format has in front of the
    GEMM. Codes only: no codec runs here."""
    g = _gen(seed, device)
    u8 = dict(dtype=torch.uint8, device=device, generator=g)
    w13 = torch.randint(0, 256, (E, 2 * I, H // 2), **u8)
    w13_sf = torch.randint(0, SCALE_CODE_HI + 1, (E, 2 * I, H // 16), **u8)
    w2 = torch.randint(0, 256, (E, H, I // 2), **u8)
    w2_sf = torch.randint(0, SCALE_CODE_HI + 1, (E, H, I // 16), **u8)
    z = torch.randn((E, 2), dtype=torch.float32, device=device, generator=g)
    g_gate = GATE_GLOBAL * torch.exp(0.05 * z[:, 0])
    g_gate_up = torch.stack([g_gate, g_gate / GATE_UP_RATIO], dim=1).contiguous()
    g_down = (DOWN_GLOBAL * torch.exp(0.05 * z[:, 1])).contiguous()
    return dict(w13_packed=w13, w13_sf_linear=w13_sf, g_gate_up=g_gate_up,
                w2_packed=w2, w2_sf_linear=w2_sf, g_down=g_down)


def make_activations(T: int, H: int, seed: int = SEED_ACTIVATIONS, device="cpu") -> torch.Tensor:
    """x [T, H] bf16 drawn N(0, 1)."""
    g = _gen(seed, device)
    return torch.randn((T, H), dtype=torch.float32, device=device, generator=g).to(torch.bfloat16)


def make_topk_routing(T: int, E: int, k: int, seed: int = SEED_ROUTING, router_weights="softmax"):
    """T streams routed top-k from N(0,1) logits (ties go to the lower expert id).

    Returns topk_ids [T, k] int32 (descending logit order) and topk_w [T, k] f32:
    softmax over the k selected logits, or U(0,1) draws.
    """
    g = _gen(seed, "cpu")
    logits = torch.randn((T, E), dtype=torch.float32, generator=g)
    order = torch.sort(-logits, dim=1, stable=True).indices[:, :k]
    ids = order.to(torch.int32).contiguous()
    if router_weights == "softmax":
        sel = torch.gather(logits, 1, order)
        w = torch.softmax(sel.to(torch.float64), dim=1).to(torch.float32)
    else:
        w = torch.rand((T, k), dtype=torch.float32, generator=g)
    return ids, w.contiguous()


def make_all_expert_routing(E: int, k: int, mg_lo: int, mg_hi: int, seed: int = SEED_ROUTING):
    """Every expert active with Mg ~ U{mg_lo..mg_hi} rows; R = sum(Mg) rows.

    Rows are laid out by ascending expert; row r belongs to token r mod T with
    T = ceil(R / k), so a token's slots hold distinct experts. Slots a token
    does not fill carry expert id -1 (unused). Router weights are U(0,1).
    Returns (topk_ids [T, k] int32, topk_w [T, k] f32, mg [E] int64).
    """
    assert mg_hi < max(1, (E * mg_lo) // k), "token rule needs Mg < T"
    g = _gen(seed, "cpu")
    mg = torch.randint(mg_lo, mg_hi + 1, (E,), generator=g)
    R = int(mg.sum())
    T = math.ceil(R / k)
    row_expert = torch.repeat_interleave(torch.arange(E, dtype=torch.int32), mg)
    ids = torch.full((T, k), -1, dtype=torch.int32)
    for j in range(k):
        rows = torch.arange(j * T, min((j + 1) * T, R))
        ids[rows - j * T, j] = row_expert[rows]
    w = torch.rand((T, k), dtype=torch.float32, generator=g)
    return ids.contiguous(), w.contiguous(), mg


def make_routing(cfg: LayerConfig, seed: int = SEED_ROUTING):
    """(topk_ids, topk_w) for a config; T is implied by ids.shape[0]."""
    if cfg.routing == "topk":
        return make_topk_routing(cfg.T, cfg.E, cfg.k, seed, cfg.router_weights)
    ids, w, _ = make_all_expert_routing(cfg.E, cfg.k, cfg.mg_lo, cfg.mg_hi, seed)
    return ids, w


def make_layer(cfg: LayerConfig, device="cpu", seed_offset: int = 0) -> dict:
    """Weights, activations and routing for one config (routing on the host)."""
    ids, w = make_routing(cfg, SEED_ROUTING + seed_offset)
    T = ids.shape[0]
    out = make_weights(cfg.E, cfg.H, cfg.I, SEED_WEIGHTS, device)
    out["x"] = make_activations(T, cfg.H, SEED_ACTIVATIONS + seed_offset, device)
    out["topk_ids"] = ids.to(device)
    out["topk_w"] = w.to(device)
    out["cfg"] = cfg
    return out
