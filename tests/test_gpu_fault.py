"""Host-side fault injection through the C ABI (MOE_FAULT / moe_set_fault): a launch that
the hook fails returns MOE_ERR_CUDA with a message naming the step, nothing after it runs,
and outputs that no earlier launch writes stay as they were (the gate's ownership contract,
"feat(engine): E1 DeepSeek-style MoE gate (sigmoid, group top-k, bias) (#108)", review
section "What looks solid": outputs unchanged on failure).  No GPU is made to fail: the
hook decides on the host, before the launch."""
import ctypes

import pytest
import torch

from deepseek_moe_layer_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")

# moe_forward's launches in order (from 8192 pairs the dispatch is still one launcher call)
STEPS = ["router GEMM", "route kernel", "permute kernel", "gather rows", "gate/up GEMM",
         "down GEMM", "combine kernel"]


def _forward(layer, x, y, inds, scores, logits):
    ws = layer.workspace(x.shape[0])
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    L = binding.lib()
    rc = L.moe_forward(P(x), x.shape[0], layer.d, layer.I, layer.E, P(layer.w_router),
                       P(layer.bias), None, ctypes.byref(layer.params), ctypes.byref(layer.ew),
                       ctypes.byref(layer.sw), P(y), P(inds), P(scores), P(logits), P(ws),
                       ws.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, L.moe_last_error().decode()


@pytest.mark.parametrize("T", [64, 2048])
def test_injected_launch_fault_leaves_later_outputs_untouched(T):
    w = inputs.scaled(inputs.WORKLOADS["tiny_T64_E16"], T=T)
    data = inputs.gen_layer(w, DEV, seed=31)
    layer = binding.MoELayer(data["w_router"], data["bias"], data["experts"], data["shared"],
                             w.top_k, w.n_group, w.topk_group, w.norm_topk_prob,
                             w.routed_scaling_factor)
    x = data["x"]
    ref = layer(x, want_intermediates=True)
    torch.cuda.synchronize()
    before = binding.get_fault()
    try:
        for at, step in enumerate(STEPS):
            y = torch.full((T, w.d), 7.0, dtype=torch.bfloat16, device=DEV)
            inds = torch.full((T, w.top_k), -5, dtype=torch.int32, device=DEV)
            scores = torch.full((T, w.top_k), -5.0, device=DEV)
            logits = torch.full((T, w.E), -5.0, device=DEV)
            binding.set_fault(binding.MOE_FAULT_LAUNCH, at)
            rc, err = _forward(layer, x, y, inds, scores, logits)
            torch.cuda.synchronize()
            assert rc == binding.MOE_ERR_CUDA, (at, rc, err)
            assert step in err and "injected launch fault" in err
            assert torch.all(y == 7.0), step          # only the combine writes y
            if at <= 1:                               # the gate writes the routing outputs
                assert torch.all(inds == -5) and torch.all(scores == -5.0)
                assert torch.all(logits == -5.0)
            else:
                assert torch.equal(inds, ref[1]) and torch.equal(scores, ref[2])
            binding.device_status()
        # with the hook off, the same call succeeds and matches the earlier result
        binding.set_fault(binding.MOE_FAULT_NONE, 0)
        y = torch.empty(T, w.d, dtype=torch.bfloat16, device=DEV)
        rc, err = _forward(layer, x, y, inds, scores, logits)
        torch.cuda.synchronize()
        assert rc == binding.MOE_OK, err
        assert torch.equal(y, ref[0]) and torch.equal(inds, ref[1])
    finally:
        binding.set_fault(*before)
