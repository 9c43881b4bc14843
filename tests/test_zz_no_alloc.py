"""moe_nvfp4_layer_static: the layer step for callers that cannot allocate
device memory (a host that owns every allocation, code that must not
synchronize the device). Its output must equal the workspace entry point's on
the same inputs, call after call, with the scratch array shared between calls.

This file is collected last on purpose: a failure here leaves every other
test already run."""
import dataclasses

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_gather_gb300 import _native as N
from nvfp4_block_scaled_gather_gb300.synthetic import CONFIGS, make_layer, make_activations, make_routing, \
    make_weights
from tests.gpu_cases import bf16_to_np, rel_fro, weights_from

pytestmark = pytest.mark.gpu

LAYER_TOL = 1e-2


def _check_against_workspace_entry(x, ids, tw, W, k):
    ref = N.MoeLayer(W, x.shape[0], k)(x, ids, tw)
    for _ in range(2):                       # two calls in a row share the scratch array
        y = torch.full_like(x, 3.0)
        N.moe_nvfp4_layer_static(x, ids, tw, W, y)
        torch.cuda.synchronize()
        got, want = bf16_to_np(y).view(np.uint16), bf16_to_np(ref)
        g = torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).double().numpy()
        r = torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).double().numpy()
        assert rel_fro(g, r) <= LAYER_TOL
        assert np.array_equal(got, want)      # the same kernels on the same inputs: identical bits
    assert N.check_status() == 0


def test_static_layer_tiny(cuda):
    cfg = CONFIGS["tiny"]
    inp = make_layer(cfg, device=cuda)
    W = weights_from(inp)
    _check_against_workspace_entry(inp["x"], inp["topk_ids"], inp["topk_w"], W, cfg.k)


def test_static_layer_decode_sizes(cuda):
    cfg = CONFIGS["decode_m8"]
    w = make_weights(cfg.E, cfg.H, cfg.I, device=cuda)
    W = weights_from(w)
    del w
    for name in ("decode_m1", "decode_m8"):
        ids, tw = make_routing(CONFIGS[name])
        x = make_activations(ids.shape[0], cfg.H, device=cuda)
        _check_against_workspace_entry(x, ids.to(cuda), tw.to(cuda), W, cfg.k)
    # beyond the fixed scratch: rejected on the host with MOE_ERR_WORKSPACE (status 5)
    ids, tw = make_routing(CONFIGS["decode_m32"])
    x = make_activations(ids.shape[0], cfg.H, device=cuda)
    assert N.load().moe_nvfp4_layer_workspace_size(32, 8, cfg.E, cfg.H, cfg.I) > N.STATIC_SCRATCH_BYTES
    with pytest.raises(RuntimeError, match="workspace too small"):
        N.moe_nvfp4_layer_static(x, ids.to(cuda), tw.to(cuda), W, torch.empty_like(x))


def test_static_layer_at_its_size_limit(cuda):
    """The largest decode batch whose workspace fits the scratch array runs and
    equals the workspace entry point; one more token is rejected on the host
    with MOE_ERR_WORKSPACE (status 5). The limit is derived from
    moe_nvfp4_layer_workspace_size, the same function the entry point uses."""
    cfg = CONFIGS["decode_m8"]
    lib = N.load()
    fits = [T for T in range(1, 64)
            if lib.moe_nvfp4_layer_workspace_size(T, cfg.k, cfg.E, cfg.H, cfg.I) <= N.STATIC_SCRATCH_BYTES]
    T_max = max(fits)
    assert fits == list(range(1, T_max + 1))
    assert lib.moe_nvfp4_layer_workspace_size(T_max + 1, cfg.k, cfg.E, cfg.H, cfg.I) > N.STATIC_SCRATCH_BYTES
    w = make_weights(cfg.E, cfg.H, cfg.I, device=cuda)
    W = weights_from(w)
    del w
    for T in (T_max, T_max + 1):
        ids, tw = make_routing(dataclasses.replace(cfg, T=T))
        x = make_activations(T, cfg.H, device=cuda)
        if T == T_max:
            _check_against_workspace_entry(x, ids.to(cuda), tw.to(cuda), W, cfg.k)
        else:
            with pytest.raises(RuntimeError, match="workspace too small"):
                N.moe_nvfp4_layer_static(x, ids.to(cuda), tw.to(cuda), W, torch.empty_like(x))
