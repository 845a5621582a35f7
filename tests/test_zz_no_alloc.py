"""moe_forward_noalloc: the layer for callers that cannot allocate device memory (engines
that reserve all of HBM for their own pools, hosts whose device allocator belongs to another
framework).  Its workspace is a fixed 64 MiB array inside the
library, so these tests call it through the C ABI and hold it to the same results as
moe_forward with a caller workspace, on two calls in a row (the second call finds the
first call's data in the shared array and must not depend on it)."""
import ctypes

import numpy as np
import pytest
import torch

from deepseek_moe_layer_gb300 import binding, inputs

from support import check_layer

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _noalloc(layer, x):
    T, d = x.shape
    K = layer.params.top_k
    y = torch.empty(T, d, dtype=torch.bfloat16, device=DEV)
    inds = torch.empty(T, K, dtype=torch.int32, device=DEV)
    scores = torch.empty(T, K, dtype=torch.float32, device=DEV)
    logits = torch.empty(T, layer.E, dtype=torch.float32, device=DEV)
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = binding.lib().moe_forward_noalloc(
        P(x), T, d, layer.I, layer.E, P(layer.w_router), P(layer.bias), P(layer.logit_offset),
        ctypes.byref(layer.params), ctypes.byref(layer.ew),
        None if layer.sw is None else ctypes.byref(layer.sw), P(y), P(inds), P(scores),
        P(logits), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == binding.MOE_OK, binding.lib().moe_last_error().decode()
    return y, inds, scores, logits


def _compare(w, seed):
    data = inputs.gen_layer(w, DEV, seed=seed)
    layer = binding.MoELayer(data["w_router"], data["bias"], data["experts"], data["shared"],
                             w.top_k, w.n_group, w.topk_group, w.norm_topk_prob,
                             w.routed_scaling_factor, data["logit_offset"])
    xs = [data["x"], inputs.gen_tokens(w, DEV, seed=seed + 1)]
    for x in xs:  # two calls in a row, different tokens
        ref = layer(x, want_intermediates=True)
        got = _noalloc(layer, x)
        torch.cuda.synchronize()
        assert torch.equal(got[1], ref[1])                                   # experts
        assert torch.allclose(got[2], ref[2], rtol=1e-6, atol=0)             # weights
        assert torch.allclose(got[3], ref[3], rtol=1e-5, atol=1e-5)          # logits
        check_layer(got[0].float().cpu().numpy(), ref[0].float().cpu().numpy())
    binding.device_status()


def test_noalloc_matches_forward_tiny():
    _compare(inputs.WORKLOADS["tiny_T64_E16"], seed=11)


def test_noalloc_matches_forward_decode_shape():
    w = inputs.Workload("decode_small", T=100, d=1024, E=64, I=512, top_k=8, n_group=8,
                        topk_group=4, norm_topk_prob=True, routed_scaling_factor=2.5,
                        bias_var=0.05)
    _compare(w, seed=12)


def test_noalloc_rejects_oversized_layer():
    w = inputs.WORKLOADS["dsv3_T8192_zipf"]
    p = binding.route_params(w.top_k, w.n_group, w.topk_group, True, 2.5)
    fake = ctypes.c_void_p(0x1000)
    ew = binding.ExpertWeights(16, 0, 0x1000, 0x1000, 0x1000, None, None, None, None, None, None)
    y = torch.full((4, 4), 3.0, device=DEV)
    rc = binding.lib().moe_forward_noalloc(fake, w.T, w.d, w.I, w.E, fake, fake, None,
                                           ctypes.byref(p), ctypes.byref(ew), ctypes.byref(ew),
                                           ctypes.c_void_p(y.data_ptr()), None, None, None,
                                           None)
    assert rc == binding.MOE_ERR_INVALID
    assert "fixed scratch" in binding.lib().moe_last_error().decode()
    torch.cuda.synchronize()
    assert torch.all(y == 3.0)
