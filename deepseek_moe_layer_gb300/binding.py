"""Python binding of the C ABI in ``include/moe_gb300.h``.

Argument marshalling only: every function takes torch tensors (device memory from
PyTorch), checks dtype / shape / device, and passes raw pointers plus the current CUDA
stream to the library of the same name.  All arithmetic runs in the CUDA kernels of
``libmoe_gb300.so``; there is no other implementation behind these calls, and the
library must be built (``deepseek_moe_layer_gb300.build``) before use.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

MOE_OK, MOE_ERR_INVALID, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_NODEVICE = 0, -1, -2, -3, -4
MOE_DTYPE_F32, MOE_DTYPE_BF16 = 0, 1

# Every symbol the public header declares.
EXPORTS = ("moe_last_error", "moe_version", "moe_device_status", "moe_route_deepseek",
           "moe_permute", "moe_router_logits", "moe_grouped_swiglu",
           "moe_grouped_swiglu_workspace_bytes", "moe_combine", "moe_forward",
           "moe_forward_workspace_bytes", "moe_set_phase_events", "moe_forward_noalloc",
           "moe_route_softmax", "moe_shared_gate", "moe_combine_gated", "moe_forward_ex",
           "moe_forward_ex_workspace_bytes", "moe_watchdog_selftest", "moe_indexer_topk",
           "moe_set_fault", "moe_get_fault")
MOE_ROUTE_DEEPSEEK, MOE_ROUTE_SOFTMAX = 0, 1


class MoeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{msg} (code {code})")
        self.code = code


class RouteParams(ctypes.Structure):
    _fields_ = [("top_k", ctypes.c_int32), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("norm_topk_prob", ctypes.c_int32),
                ("routed_scaling_factor", ctypes.c_float)]


class ExpertWeights(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p),
                ("gate_scale", ctypes.c_void_p), ("gate_bias", ctypes.c_void_p),
                ("up_scale", ctypes.c_void_p), ("up_bias", ctypes.c_void_p),
                ("down_scale", ctypes.c_void_p), ("down_bias", ctypes.c_void_p)]


class LayerArgs(ctypes.Structure):
    _fields_ = [("route_kind", ctypes.c_int32), ("x", ctypes.c_void_p), ("T", ctypes.c_int64),
                ("d", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("w_router", ctypes.c_void_p), ("logit_offset", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("params", RouteParams),
                ("experts", ctypes.POINTER(ExpertWeights)),
                ("shared", ctypes.POINTER(ExpertWeights)), ("w_shared_gate", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("inds_out", ctypes.c_void_p),
                ("scores_out", ctypes.c_void_p), ("logits_out", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def lib(path: str | None = None):
    """The loaded CUDA library (built on first use if the sources are newer)."""
    global _lib
    with _lock:
        if _lib is None:
            so = path or _build.build()
            if not os.path.exists(so):
                raise MoeError(MOE_ERR_NODEVICE, f"CUDA library missing: {so}")
            L = ctypes.CDLL(so)
            P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            L.moe_last_error.restype = ctypes.c_char_p
            L.moe_version.restype = i32
            L.moe_device_status.argtypes = [i32, P]
            L.moe_route_deepseek.argtypes = [P, ctypes.c_int, i64, i32, P,
                                             ctypes.POINTER(RouteParams), P, P, P]
            L.moe_permute.argtypes = [P, i64, i32, i32, P, P, P, P, P]
            L.moe_router_logits.argtypes = [P, i64, i32, P, i32, P, P, P]
            L.moe_grouped_swiglu.argtypes = [P, i64, i32, i32, i32, i32, P, P,
                                             ctypes.POINTER(ExpertWeights),
                                             ctypes.POINTER(ExpertWeights), P, P, sz, P]
            L.moe_grouped_swiglu_workspace_bytes.argtypes = [i64, i32, i32, i32, i32, i32]
            L.moe_grouped_swiglu_workspace_bytes.restype = sz
            L.moe_combine.argtypes = [P, P, P, P, i64, i32, i32, P, P]
            L.moe_forward.argtypes = [P, i64, i32, i32, i32, P, P, P,
                                      ctypes.POINTER(RouteParams), ctypes.POINTER(ExpertWeights),
                                      ctypes.POINTER(ExpertWeights), P, P, P, P, P, sz, P]
            L.moe_forward_workspace_bytes.argtypes = [i64, i32, i32, i32, i32, i32]
            L.moe_forward_workspace_bytes.restype = sz
            L.moe_set_phase_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32]
            L.moe_forward_noalloc.argtypes = [P, i64, i32, i32, i32, P, P, P,
                                              ctypes.POINTER(RouteParams),
                                              ctypes.POINTER(ExpertWeights),
                                              ctypes.POINTER(ExpertWeights), P, P, P, P, P]
            L.moe_route_softmax.argtypes = [P, ctypes.c_int, i64, i32, i32, P, P, P]
            L.moe_shared_gate.argtypes = [P, i64, i32, P, P, P]
            L.moe_combine_gated.argtypes = [P, P, P, P, P, i64, i32, i32, P, P]
            L.moe_forward_ex.argtypes = [ctypes.POINTER(LayerArgs), P, sz, P]
            L.moe_forward_ex_workspace_bytes.argtypes = [ctypes.POINTER(LayerArgs)]
            L.moe_forward_ex_workspace_bytes.restype = sz
            L.moe_watchdog_selftest.argtypes = [i64, P]
            L.moe_indexer_topk.argtypes = [P, ctypes.c_int, i64, i32, i64, P, i32, P, P, i64, P]
            L.moe_set_fault.argtypes = [i32, i32]
            L.moe_get_fault.argtypes = [ctypes.POINTER(i32), ctypes.POINTER(i32)]
            for name in ("moe_device_status", "moe_route_deepseek", "moe_permute",
                         "moe_router_logits", "moe_grouped_swiglu", "moe_combine",
                         "moe_forward", "moe_set_phase_events", "moe_forward_noalloc",
                         "moe_route_softmax", "moe_shared_gate", "moe_combine_gated",
                         "moe_forward_ex", "moe_watchdog_selftest", "moe_indexer_topk",
                         "moe_set_fault", "moe_get_fault"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def _check(rc):
    if rc != MOE_OK:
        raise MoeError(rc, lib().moe_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, name, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def route_params(top_k, n_group, topk_group, norm_topk_prob, routed_scaling_factor):
    return RouteParams(int(top_k), int(n_group), int(topk_group), int(bool(norm_topk_prob)),
                       float(routed_scaling_factor))


def expert_weights(w: dict | None):
    """ExpertWeights from a dict: bits 16 -> gate/up/down bf16; bits 8 or 4 -> gate/up/down
    int32 (packed uint32 words) plus gate_s/gate_b/up_s/up_b/down_s/down_b fp16 and an
    optional 'group' (inputs per scale: 32, 64 or 128; default 64)."""
    if w is None:
        return None
    bits = int(w.get("bits", 16))
    if bits == 16:
        for k in ("gate", "up", "down"):
            _need(w[k], torch.bfloat16, k)
        return ExpertWeights(16, 0, w["gate"].data_ptr(), w["up"].data_ptr(), w["down"].data_ptr(),
                             None, None, None, None, None, None)
    for k in ("gate", "up", "down"):
        _need(w[k], torch.int32, k)
    for k in ("gate_s", "gate_b", "up_s", "up_b", "down_s", "down_b"):
        _need(w[k], torch.float16, k)
    if bits not in (4, 8):
        raise ValueError(f"bits = {bits}: expert weights are bf16 (16) or affine 8 / 4-bit")
    return ExpertWeights(bits, int(w.get("group", 64)), w["gate"].data_ptr(), w["up"].data_ptr(),
                         w["down"].data_ptr(), w["gate_s"].data_ptr(), w["gate_b"].data_ptr(),
                         w["up_s"].data_ptr(), w["up_b"].data_ptr(), w["down_s"].data_ptr(),
                         w["down_b"].data_ptr())


def _ref(s):
    return None if s is None else ctypes.byref(s)


# ---------------------------------------------------------------------------------------
# the calls
# ---------------------------------------------------------------------------------------

def route_deepseek(logits, bias, top_k, n_group, topk_group, norm_topk_prob,
                   routed_scaling_factor, inds=None, scores=None, stream=None):
    """logits [..., E] fp32/bf16, bias [E] fp32 -> (inds int32 [..., K], scores fp32 [..., K])."""
    if logits.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("logits must be fp32 or bf16")
    _need(logits, logits.dtype, "logits")
    if bias.dim() != 1 or bias.shape[0] != logits.shape[-1]:
        raise ValueError("bias must have rank 1 and length E (the last dim of logits)")
    _need(bias, torch.float32, "bias", logits.device)
    E = logits.shape[-1]
    rows = logits.numel() // E if E else 0
    shape = tuple(logits.shape[:-1]) + (int(top_k),)
    if inds is None:
        inds = torch.empty(shape, dtype=torch.int32, device=logits.device)
    if scores is None:
        scores = torch.empty(shape, dtype=torch.float32, device=logits.device)
    p = route_params(top_k, n_group, topk_group, norm_topk_prob, routed_scaling_factor)
    dt = MOE_DTYPE_F32 if logits.dtype == torch.float32 else MOE_DTYPE_BF16
    _check(lib().moe_route_deepseek(_ptr(logits), dt, rows, E, _ptr(bias), ctypes.byref(p),
                                    _ptr(inds), _ptr(scores), _stream(stream)))
    return inds, scores


def route_softmax(logits, top_k, inds=None, scores=None, stream=None):
    """Softmax route: logits [..., E] fp32/bf16 -> (inds int32, scores fp32) [..., K]."""
    if logits.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("logits must be fp32 or bf16")
    _need(logits, logits.dtype, "logits")
    E = logits.shape[-1]
    rows = logits.numel() // E if E else 0
    shape = tuple(logits.shape[:-1]) + (int(top_k),)
    if inds is None:
        inds = torch.empty(shape, dtype=torch.int32, device=logits.device)
    if scores is None:
        scores = torch.empty(shape, dtype=torch.float32, device=logits.device)
    dt = MOE_DTYPE_F32 if logits.dtype == torch.float32 else MOE_DTYPE_BF16
    _check(lib().moe_route_softmax(_ptr(logits), dt, rows, E, int(top_k), _ptr(inds),
                                   _ptr(scores), _stream(stream)))
    return inds, scores


def shared_gate(x, w_gate, stream=None):
    """gate[t] = sigmoid(x[t] . w_gate): bf16 x [T, d], w_gate [d] -> fp32 [T]."""
    _need(x, torch.bfloat16, "x")
    _need(w_gate, torch.bfloat16, "w_gate", x.device)
    T, d = x.shape
    g = torch.empty(T, dtype=torch.float32, device=x.device)
    _check(lib().moe_shared_gate(_ptr(x), T, d, _ptr(w_gate), _ptr(g), _stream(stream)))
    return g


def combine_gated(expert_out, scores, inv_perm, shared_out, gate, stream=None):
    """y[t] = sum_k scores[t,k] expert_out[inv_perm[t*K+k]] + gate[t] shared_out[t]."""
    _need(expert_out, torch.bfloat16, "expert_out")
    _need(scores, torch.float32, "scores")
    _need(inv_perm, torch.int32, "inv_perm")
    _need(gate, torch.float32, "gate")
    T, K = scores.shape
    d = expert_out.shape[1]
    y = torch.empty(T, d, dtype=torch.bfloat16, device=expert_out.device)
    _check(lib().moe_combine_gated(_ptr(expert_out), _ptr(scores), _ptr(inv_perm),
                                   _ptr(shared_out), _ptr(gate), T, K, d, _ptr(y),
                                   _stream(stream)))
    return y


def indexer_topk(scores, k, lengths=None, want_mask=False, inds=None, mask=None,
                 stream=None):
    """DSA indexer selection: scores [rows, n] fp32/bf16 (rows may be strided: the row
    stride is taken from the tensor) -> int32 [rows, k] ascending positions padded with -1,
    and with want_mask also the uint8 [rows, n] selection mask."""
    if scores.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("scores must be fp32 or bf16")
    if scores.dim() != 2 or (scores.shape[1] > 1 and scores.stride(1) != 1):
        raise ValueError("scores must be [rows, n] with unit stride along n")
    rows, n = scores.shape
    ld = scores.stride(0) if rows > 1 else n
    if lengths is not None:
        _need(lengths, torch.int32, "lengths", scores.device)
        if lengths.shape != (rows,):
            raise ValueError("lengths must be [rows]")
    if inds is None:
        inds = torch.empty(rows, int(k), dtype=torch.int32, device=scores.device)
    if want_mask and mask is None:
        mask = torch.empty(rows, n, dtype=torch.uint8, device=scores.device)
    dt = MOE_DTYPE_F32 if scores.dtype == torch.float32 else MOE_DTYPE_BF16
    _check(lib().moe_indexer_topk(_ptr(scores), dt, rows, n, ld, _ptr(lengths), int(k),
                                  _ptr(inds), _ptr(mask), n if mask is not None else 0,
                                  _stream(stream)))
    return (inds, mask) if want_mask else inds


def permute(inds, E, stream=None):
    """inds int32 [T, K] -> (counts [E], offsets [E+1], perm [P], inv_perm [P]), int32."""
    _need(inds, torch.int32, "inds")
    T, K = inds.shape
    dev = inds.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * K, dtype=torch.int32, device=dev)
    inv = torch.empty(T * K, dtype=torch.int32, device=dev)
    _check(lib().moe_permute(_ptr(inds), T, K, E, _ptr(counts), _ptr(offsets), _ptr(perm),
                             _ptr(inv), _stream(stream)))
    return counts, offsets, perm, inv


def router_logits(x, w_router, logit_offset=None, stream=None):
    """x bf16 [T, d], w_router bf16 [E, d] -> fp32 logits [T, E]."""
    _need(x, torch.bfloat16, "x")
    _need(w_router, torch.bfloat16, "w_router", x.device)
    T, d = x.shape
    E = w_router.shape[0]
    if logit_offset is not None:
        _need(logit_offset, torch.float32, "logit_offset", x.device)
    out = torch.empty(T, E, dtype=torch.float32, device=x.device)
    _check(lib().moe_router_logits(_ptr(x), T, d, _ptr(w_router), E, _ptr(logit_offset),
                                   _ptr(out), _stream(stream)))
    return out


def grouped_swiglu_workspace_bytes(T, d, I, E, K, has_shared):
    return lib().moe_grouped_swiglu_workspace_bytes(T, d, I, E, K, int(bool(has_shared)))


def grouped_swiglu(x, offsets, perm, K, experts, shared=None, I=None, ws=None, stream=None):
    """Expert SwiGLU over the dispatched tokens; returns bf16 [P (+T), d] in slot order."""
    _need(x, torch.bfloat16, "x")
    T, d = x.shape
    E = offsets.numel() - 1
    I = I if I is not None else (experts["gate"].shape[1])
    ew, sw = expert_weights(experts), expert_weights(shared)
    P = T * K
    out = torch.empty(P + (T if shared is not None else 0), d, dtype=torch.bfloat16,
                      device=x.device)
    need = grouped_swiglu_workspace_bytes(T, d, I, E, K, shared is not None)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    _check(lib().moe_grouped_swiglu(_ptr(x), T, d, I, E, K, _ptr(offsets), _ptr(perm),
                                    ctypes.byref(ew), _ref(sw), _ptr(out), _ptr(ws),
                                    ws.numel(), _stream(stream)))
    return out


def combine(expert_out, scores, inv_perm, shared_out=None, stream=None):
    """y[t] = sum_k scores[t,k] expert_out[inv_perm[t*K+k]] (+ shared_out[t]), bf16 [T, d]."""
    _need(expert_out, torch.bfloat16, "expert_out")
    _need(scores, torch.float32, "scores")
    _need(inv_perm, torch.int32, "inv_perm")
    T, K = scores.shape
    d = expert_out.shape[1]
    y = torch.empty(T, d, dtype=torch.bfloat16, device=expert_out.device)
    _check(lib().moe_combine(_ptr(expert_out), _ptr(scores), _ptr(inv_perm), _ptr(shared_out),
                             T, K, d, _ptr(y), _stream(stream)))
    return y


def forward_workspace_bytes(T, d, I, E, top_k, has_shared):
    return lib().moe_forward_workspace_bytes(T, d, I, E, top_k, int(bool(has_shared)))


class MoELayer:
    """The whole layer on device-resident weights: ``layer(x) -> y``.

    Holds the weights, the gate parameters and a reusable workspace; each call is one
    ``moe_forward`` on the current stream.  With ``want_intermediates`` it also returns the
    selected experts, their weights and the router logits.
    """

    def __init__(self, w_router, bias, experts, shared, top_k, n_group, topk_group,
                 norm_topk_prob, routed_scaling_factor, logit_offset=None,
                 route_kind=MOE_ROUTE_DEEPSEEK, w_shared_gate=None):
        _need(w_router, torch.bfloat16, "w_router")
        self.dev = w_router.device
        if bias is not None:
            _need(bias, torch.float32, "bias", self.dev)
        if w_shared_gate is not None:
            _need(w_shared_gate, torch.bfloat16, "w_shared_gate", self.dev)
        self.route_kind, self.w_shared_gate = int(route_kind), w_shared_gate
        # the DeepSeek body goes through moe_forward, anything else through moe_forward_ex
        self.ex = self.route_kind != MOE_ROUTE_DEEPSEEK or w_shared_gate is not None
        self.w_router, self.bias, self.logit_offset = w_router, bias, logit_offset
        self.experts, self.shared = experts, shared
        self.E, self.d = w_router.shape
        self.I = experts["gate"].shape[1]
        self.params = route_params(top_k, n_group, topk_group, norm_topk_prob,
                                   routed_scaling_factor)
        self.ew, self.sw = expert_weights(experts), expert_weights(shared)
        self.ws = None

    def _args(self, x, y, inds, scores, logits):
        a = LayerArgs()
        a.route_kind = self.route_kind
        a.x, a.T, a.d, a.I, a.E = x.data_ptr(), x.shape[0], self.d, self.I, self.E
        a.w_router = self.w_router.data_ptr()
        a.logit_offset = None if self.logit_offset is None else self.logit_offset.data_ptr()
        a.bias = None if self.bias is None else self.bias.data_ptr()
        a.params = self.params
        a.experts = ctypes.pointer(self.ew)
        a.shared = ctypes.pointer(self.sw) if self.sw is not None else None
        a.w_shared_gate = None if self.w_shared_gate is None else self.w_shared_gate.data_ptr()
        a.y = None if y is None else y.data_ptr()
        a.inds_out = None if inds is None else inds.data_ptr()
        a.scores_out = None if scores is None else scores.data_ptr()
        a.logits_out = None if logits is None else logits.data_ptr()
        return a

    def workspace(self, T):
        if self.ex:
            a = LayerArgs()
            a.route_kind, a.T, a.d, a.I, a.E = self.route_kind, T, self.d, self.I, self.E
            a.params = self.params
            a.shared = ctypes.pointer(self.sw) if self.sw is not None else None
            a.w_shared_gate = None if self.w_shared_gate is None else 1
            need = lib().moe_forward_ex_workspace_bytes(ctypes.byref(a))
        else:
            need = forward_workspace_bytes(T, self.d, self.I, self.E, self.params.top_k,
                                           self.shared is not None)
        if self.ws is None or self.ws.numel() < need:
            self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.dev)
        return self.ws

    def __call__(self, x, y=None, want_intermediates=False, stream=None):
        _need(x, torch.bfloat16, "x", self.dev)
        T, d = x.shape
        K = self.params.top_k
        ws = self.workspace(T)
        if y is None:
            y = torch.empty(T, d, dtype=torch.bfloat16, device=self.dev)
        inds = scores = logits = None
        if want_intermediates:
            inds = torch.empty(T, K, dtype=torch.int32, device=self.dev)
            scores = torch.empty(T, K, dtype=torch.float32, device=self.dev)
            logits = torch.empty(T, self.E, dtype=torch.float32, device=self.dev)
        if self.ex:
            a = self._args(x, y, inds, scores, logits)
            _check(lib().moe_forward_ex(ctypes.byref(a), _ptr(ws), ws.numel(), _stream(stream)))
            return (y, inds, scores, logits) if want_intermediates else y
        _check(lib().moe_forward(_ptr(x), T, d, self.I, self.E, _ptr(self.w_router),
                                 _ptr(self.bias), _ptr(self.logit_offset),
                                 ctypes.byref(self.params), ctypes.byref(self.ew), _ref(self.sw),
                                 _ptr(y), _ptr(inds), _ptr(scores), _ptr(logits), _ptr(ws),
                                 ws.numel(), _stream(stream)))
        if want_intermediates:
            return y, inds, scores, logits
        return y


PHASES = ("router", "route", "permute", "gather", "gate_up", "down", "combine")


def set_phase_events(events):
    """Record torch.cuda.Event objects (8: start + one after each of PHASES) inside the
    next moe_forward calls on their stream; None stops recording."""
    if not events:
        _check(lib().moe_set_phase_events(None, 0))
        return
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event at its first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib().moe_set_phase_events(arr, len(events)))


def device_status(clear=True, stream=None):
    """MOE_OK, or raises MoeError(MOE_ERR_TIMEOUT) if a kernel gave up a wait."""
    _check(lib().moe_device_status(int(bool(clear)), _stream(stream)))


def watchdog_selftest(limit_ns=20_000_000, stream=None):
    """Launches a wait that nothing completes, bounded by limit_ns; afterwards
    device_status() raises MoeError(MOE_ERR_TIMEOUT)."""
    _check(lib().moe_watchdog_selftest(int(limit_ns), _stream(stream)))


MOE_FAULT_NONE, MOE_FAULT_LAUNCH = 0, 1


def set_fault(kind=MOE_FAULT_NONE, at=0):
    """Test hook: with MOE_FAULT_LAUNCH the at-th kernel launch of every later call reports
    MOE_ERR_CUDA instead of launching; MOE_FAULT_NONE turns it off."""
    _check(lib().moe_set_fault(int(kind), int(at)))


def get_fault():
    """(kind, at) of the fault hook (MOE_FAULT in the environment sets the initial state)."""
    k, a = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().moe_get_fault(ctypes.byref(k), ctypes.byref(a)))
    return k.value, a.value
