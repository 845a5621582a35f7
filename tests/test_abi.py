"""The C ABI on a machine without a GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any CUDA call (the gate's
validation matrix: "feat(engine): E1 DeepSeek-style MoE gate (sigmoid, group top-k, bias)
(#108)", review findings L1/L2 and the author's reply)."""
import ctypes
import os
import re
import subprocess
import sys

import pytest
import torch

from deepseek_moe_layer_gb300 import binding
from deepseek_moe_layer_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe_gb300.h")
FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails its host checks


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_header_matches_binding_exports():
    assert _declared() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol():
    so = B.build()
    out = subprocess.run(["nm", "-D", "--defined-only", so], capture_output=True, text=True,
                         check=True).stdout
    syms = {l.split()[-1] for l in out.splitlines() if l.strip()}
    for name in _declared():
        assert name in syms, name
    L = binding.lib()
    for name in _declared():
        assert hasattr(L, name)
    assert L.moe_version() >= 100


def _route(E=8, top_k=2, n_group=1, topk_group=1, logits=FAKE, bias=FAKE, rows=4, dtype=0):
    p = binding.route_params(top_k, n_group, topk_group, True, 1.0)
    L = binding.lib()
    rc = L.moe_route_deepseek(logits, dtype, rows, E, bias, ctypes.byref(p), FAKE, FAKE, None)
    return rc, L.moe_last_error().decode()


@pytest.mark.parametrize("kw,msg", [
    (dict(logits=None), "NULL"),
    (dict(bias=None), "NULL"),
    (dict(top_k=0), "top_k = 0 < 1"),
    (dict(top_k=9), "top_k = 9 > E"),
    (dict(E=64, top_k=33), "top_k = 33 > 32"),
    (dict(n_group=3), "not divisible"),
    (dict(n_group=2, topk_group=0), "topk_group"),
    (dict(n_group=2, topk_group=3), "topk_group"),
    (dict(n_group=1, topk_group=2), "topk_group"),
    (dict(n_group=8, topk_group=1), "expert(s) per group"),
    (dict(n_group=0), "n_group = 0"),
    (dict(E=0, top_k=1), "E = 0"),
    (dict(E=2048, top_k=2), "E = 2048"),
    (dict(rows=-1), "rows"),
    (dict(dtype=7), "dtype"),
])
def test_route_validation_matrix(kw, msg):
    rc, err = _route(**kw)
    assert rc == binding.MOE_ERR_INVALID
    assert msg in err


def test_valid_route_without_gpu_fails_loudly():
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, err = _route()
    assert rc == binding.MOE_ERR_NODEVICE and err


def test_empty_route_is_noop():
    rc, _ = _route(rows=0)
    assert rc == binding.MOE_OK


def _forward(T=4, d=256, I=128, E=16, bits=16, group=64, ws_bytes=None, shared=True, **pk):
    L = binding.lib()
    p = binding.route_params(pk.get("top_k", 4), pk.get("n_group", 4), pk.get("topk_group", 2),
                             True, 2.5)
    ew = binding.ExpertWeights(bits, group, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000,
                               0x1000, 0x1000, 0x1000)
    sw = binding.ExpertWeights(16, 0, 0x1000, 0x1000, 0x1000, None, None, None, None, None, None)
    need = L.moe_forward_workspace_bytes(T, d, I, E, p.top_k, 1)
    rc = L.moe_forward(FAKE, T, d, I, E, FAKE, FAKE, None, ctypes.byref(p), ctypes.byref(ew),
                       ctypes.byref(sw) if shared else None, FAKE, None, None, None,
                       ctypes.c_void_p(0x10000), need if ws_bytes is None else ws_bytes, None)
    return rc, L.moe_last_error().decode()


@pytest.mark.parametrize("kw,msg", [
    (dict(d=200), "d = 200"),
    (dict(I=100), "I = 100"),
    (dict(T=-1), "T = -1"),
    (dict(bits=2), "bits = 2"),
    (dict(bits=4, group=16), "group_size = 16"),
    (dict(bits=8, group=256), "group_size = 256"),
    (dict(ws_bytes=1024), "ws_bytes"),
    (dict(top_k=0), "top_k"),
    (dict(n_group=16, topk_group=1), "expert(s) per group"),
])
def test_forward_validation_matrix(kw, msg):
    rc, err = _forward(**kw)
    assert rc == binding.MOE_ERR_INVALID
    assert msg in err


def test_workspace_grows_with_tokens():
    L = binding.lib()
    a = L.moe_forward_workspace_bytes(128, 7168, 2048, 256, 8, 1)
    b = L.moe_forward_workspace_bytes(8192, 7168, 2048, 256, 8, 1)
    assert 0 < a < b
    assert b % 256 == 0
    # x_perm [P, d] + h [P+T, I] + expert_out [P+T, d] in bf16 at least
    P, T = 8192 * 8, 8192
    assert b >= 2 * (P * 7168 + (P + T) * 2048 + (P + T) * 7168)


def test_permute_and_combine_validation():
    L = binding.lib()
    assert L.moe_permute(None, 4, 2, 8, FAKE, FAKE, FAKE, FAKE, None) == binding.MOE_ERR_INVALID
    assert L.moe_permute(FAKE, 4, 0, 8, FAKE, FAKE, FAKE, FAKE, None) == binding.MOE_ERR_INVALID
    assert L.moe_permute(FAKE, 4, 2, 0, FAKE, FAKE, FAKE, FAKE, None) == binding.MOE_ERR_INVALID
    assert L.moe_combine(FAKE, FAKE, FAKE, None, 4, 2, 12, FAKE, None) == binding.MOE_ERR_INVALID
    assert L.moe_combine(None, FAKE, FAKE, None, 4, 2, 16, FAKE, None) == binding.MOE_ERR_INVALID
    assert L.moe_router_logits(FAKE, 4, 100, FAKE, 8, None, FAKE, None) == binding.MOE_ERR_INVALID


def test_binding_rejects_bad_bias_rank():
    lg = torch.zeros(2, 8)
    with pytest.raises(ValueError):
        binding.route_deepseek(lg, torch.zeros(1, 8), 2, 1, 1, True, 1.0)
    with pytest.raises(ValueError):
        binding.route_deepseek(lg, torch.zeros(7), 2, 1, 1, True, 1.0)


def _forward_ex(route_kind=binding.MOE_ROUTE_SOFTMAX, bias=True, shared=True, gate=True,
                top_k=4, E=16, ws_bytes=None):
    L = binding.lib()
    a = binding.LayerArgs()
    a.route_kind, a.x, a.T, a.d, a.I, a.E = route_kind, 0x1000, 4, 256, 128, E
    a.w_router = 0x1000
    a.bias = 0x1000 if bias else None
    a.params = binding.route_params(top_k, 4, 2, True, 2.5)
    ew = binding.ExpertWeights(16, 0, 0x1000, 0x1000, 0x1000, None, None, None, None, None, None)
    a.experts = ctypes.pointer(ew)
    a.shared = ctypes.pointer(ew) if shared else None
    a.w_shared_gate = 0x1000 if gate else None
    a.y = 0x1000
    need = L.moe_forward_ex_workspace_bytes(ctypes.byref(a))
    rc = L.moe_forward_ex(ctypes.byref(a), ctypes.c_void_p(0x10000),
                          need if ws_bytes is None else ws_bytes, None)
    return rc, L.moe_last_error().decode(), need


@pytest.mark.parametrize("kw,msg", [
    (dict(route_kind=7), "route_kind 7"),
    (dict(route_kind=binding.MOE_ROUTE_DEEPSEEK, bias=False), "NULL"),
    (dict(top_k=17), "top_k = 17"),
    (dict(E=2048, top_k=2), "E = 2048"),
    (dict(shared=False), "without a shared expert"),
    (dict(ws_bytes=4096), "ws_bytes"),
])
def test_forward_ex_validation_matrix(kw, msg):
    rc, err, _ = _forward_ex(**kw)
    assert rc == binding.MOE_ERR_INVALID
    assert msg in err


def test_forward_ex_workspace_counts_the_gate():
    _, _, with_gate = _forward_ex(gate=True, ws_bytes=0)
    _, _, without = _forward_ex(gate=False, ws_bytes=0)
    assert with_gate == without + 256  # T = 4 fp32 gates, 256-byte aligned
    assert without == binding.lib().moe_forward_workspace_bytes(4, 256, 128, 16, 4, 1)


def test_softmax_gate_watchdog_validation():
    L = binding.lib()
    assert L.moe_route_softmax(FAKE, 0, 4, 16, 17, FAKE, FAKE, None) == binding.MOE_ERR_INVALID
    assert "top_k = 17" in L.moe_last_error().decode()
    assert L.moe_route_softmax(FAKE, 5, 4, 16, 2, FAKE, FAKE, None) == binding.MOE_ERR_INVALID
    assert L.moe_route_softmax(None, 0, 4, 16, 2, FAKE, FAKE, None) == binding.MOE_ERR_INVALID
    assert L.moe_route_softmax(None, 0, 0, 16, 2, None, None, None) == binding.MOE_OK
    assert L.moe_shared_gate(FAKE, 4, 100, FAKE, FAKE, None) == binding.MOE_ERR_INVALID
    assert L.moe_shared_gate(FAKE, 4, 256, None, FAKE, None) == binding.MOE_ERR_INVALID
    assert L.moe_combine_gated(FAKE, FAKE, FAKE, FAKE, None, 4, 2, 256, FAKE,
                               None) == binding.MOE_ERR_INVALID
    for bad in (0, 999, 2_000_000_000):
        assert L.moe_watchdog_selftest(bad, None) == binding.MOE_ERR_INVALID
        assert "limit_ns" in L.moe_last_error().decode()


def _align256(v):
    return (v + 255) // 256 * 256


@pytest.mark.parametrize("T,d,I,E,K", [(128, 7168, 2048, 256, 8), (8192, 7168, 2048, 256, 8),
                                       (64, 256, 128, 16, 4), (33, 640, 128, 24, 6)])
def test_forward_workspace_layout_and_router_split_bound(T, d, I, E, K):
    """The workspace is the documented pieces, with room for the router's partial logits of
    at most max(1, d/512) K-splits: the router keeps at least 8 of its d/64 k-blocks per
    split, so no device's plan splits further."""
    P = T * K
    S = max(1, d // 512)
    want = (_align256(S * T * E * 4) + 2 * _align256(P * 4) + _align256(E * 4)
            + _align256((E + 1) * 4) + 2 * _align256(P * 4) + _align256((P + T) * d * 2)
            + _align256(P * d * 2) + _align256((P + T) * I * 2))
    assert binding.lib().moe_forward_workspace_bytes(T, d, I, E, K, 1) == want


def test_fault_hook_state_and_validation():
    L = binding.lib()
    before = binding.get_fault()
    try:
        binding.set_fault(binding.MOE_FAULT_LAUNCH, 3)
        assert binding.get_fault() == (binding.MOE_FAULT_LAUNCH, 3)
        assert L.moe_set_fault(7, 0) == binding.MOE_ERR_INVALID
        assert "fault kind 7" in L.moe_last_error().decode()
        assert L.moe_set_fault(binding.MOE_FAULT_LAUNCH, -1) == binding.MOE_ERR_INVALID
        assert binding.get_fault() == (binding.MOE_FAULT_LAUNCH, 3)  # rejected: unchanged
        assert L.moe_get_fault(None, None) == binding.MOE_ERR_INVALID
        # argument checks still come first: a bad call is rejected as invalid, not faulted
        binding.set_fault(binding.MOE_FAULT_LAUNCH, 0)
        rc, err = _route(top_k=0)
        assert rc == binding.MOE_ERR_INVALID and "top_k" in err
        if not torch.cuda.is_available():  # and so is the device check, before any launch
            rc, err = _route()
            assert rc == binding.MOE_ERR_NODEVICE
    finally:
        binding.set_fault(*before)


@pytest.mark.parametrize("env,want", [("launch", (1, 0)), ("launch:5", (1, 5)),
                                      ("bogus", (0, 0)), ("", (0, 0))])
def test_fault_hook_reads_environment(env, want):
    code = ("import sys; sys.path.insert(0, %r); from deepseek_moe_layer_gb300 import binding; "
            "print(*binding.get_fault())" % os.path.dirname(os.path.dirname(__file__)))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       env={**os.environ, "MOE_FAULT": env}, check=True)
    assert tuple(int(v) for v in r.stdout.split()) == want
