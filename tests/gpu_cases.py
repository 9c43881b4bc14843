"""Shared helpers of the GPU parity tests: conversions, the stage-by-stage run
through the C ABI, and lazy host copies of expert weights for the oracle."""
import numpy as np
import torch

from nvfp4_block_scaled_gather_gb300 import _native as N


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
