"""CPU oracle for the DeepSeek-style MoE FFN forward.

TEST INFRASTRUCTURE ONLY.  The product path (the ``deepseek_moe_layer_gb300`` package and
its CUDA library) never imports, links or runs anything here.  Only the tests, the smoke
check and the CPU-baseline leg of the bench may use it.  It shares no code with the CUDA
path; both sides meet only through the seeded input generators, which hold none of the
method's arithmetic.

The arithmetic lives in ``moe_oracle.c`` (plain C, one function per step, each citing the
page and section it follows).  This module compiles it with gcc and exposes it through
ctypes on numpy arrays.

Parity of every function here is pinned by ``tests/test_oracle.py`` against brute force,
closed forms, invariants the pages state, and independent numpy evaluations.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, -O2, OpenMP, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            P = ctypes.c_void_p
            i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
            lib.oracle_route.argtypes = [P, i64, i32, P, i32, i32, i32, i32, f32, P, P]
            lib.oracle_route.restype = ctypes.c_int
            lib.oracle_permute.argtypes = [P, i64, i32, i32, P, P, P, P]
            lib.oracle_permute.restype = ctypes.c_int
            lib.oracle_router_logits.argtypes = [P, i64, i32, P, i32, P, P]
            lib.oracle_router_logits.restype = None
            lib.oracle_dequant_q4.argtypes = [P, P, P, i64, i64, i32, P]
            lib.oracle_dequant_q4.restype = None
            lib.oracle_dequant.argtypes = [ctypes.c_int, P, P, P, i64, i64, i32, P]
            lib.oracle_dequant.restype = None
            lib.oracle_moe_layer_rows.argtypes = (
                [P, i64, i32, i32, i32, i32, P, P, i32, i32] + [P] * 9 + [i32] + [P] * 9
                + [P, P, i64, P])
            lib.oracle_route_softmax.argtypes = [P, i64, i32, i32, P, P]
            lib.oracle_route_softmax.restype = ctypes.c_int
            lib.oracle_moe_layer_rows.restype = ctypes.c_int
            lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f32.restype = f32
            lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f32.restype = f32
            lib.oracle_indexer_topk.argtypes = [P, i64, i32, i64, P, i32, P, P, i64]
            lib.oracle_indexer_topk.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return _load().oracle_num_threads()


def route(logits, bias, top_k, n_group, topk_group, norm_topk_prob, routed_scaling_factor):
    """DeepSeek gate on fp32 logits [..., E] with bias [E]; returns (inds int32, scores fp32)."""
    lib = _load()
    lg = _c(logits, np.float32)
    E = lg.shape[-1]
    rows = lg.size // E if E else 0
    b = _c(bias, np.float32)
    inds = np.zeros(lg.shape[:-1] + (top_k,), np.int32)
    scores = np.zeros(lg.shape[:-1] + (top_k,), np.float32)
    rc = lib.oracle_route(_ptr(lg), rows, E, _ptr(b), top_k, n_group, topk_group,
                          int(bool(norm_topk_prob)), float(routed_scaling_factor),
                          _ptr(inds), _ptr(scores))
    if rc != 0:
        raise ValueError("oracle_route rejected its arguments")
    return inds, scores


def permute(inds, E):
    """Stable token->expert dispatch: (counts[E], offsets[E+1], perm[P], inv_perm[P])."""
    lib = _load()
    ind = _c(inds, np.int32)
    T, K = ind.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * K, np.int32)
    inv = np.zeros(T * K, np.int32)
    rc = lib.oracle_permute(_ptr(ind), T, K, E, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv))
    if rc != 0:
        raise ValueError("oracle_permute: expert index out of range")
    return counts, offsets, perm, inv


def router_logits(x_bf16_bits, w_router_bf16_bits, logit_offset=None):
    """fp32 logits [T, E] of bf16 x [T, d] against bf16 router weight [E, d] (uint16 bits)."""
    lib = _load()
    x = _c(x_bf16_bits, np.uint16)
    w = _c(w_router_bf16_bits, np.uint16)
    T, d = x.shape
    E = w.shape[0]
    off = None if logit_offset is None else _c(logit_offset, np.float32)
    out = np.zeros((T, E), np.float32)
    lib.oracle_router_logits(_ptr(x), T, d, _ptr(w), E, _ptr(off), _ptr(out))
    return out


def dequant_q4(q, scale_f16_bits, bias_f16_bits, cols, group=64):
    """Affine 4-bit rows [rows, cols/8] uint32 -> fp32 [rows, cols]."""
    lib = _load()
    qq = _c(q, np.uint32)
    rows = qq.size // (cols // 8)
    s = _c(scale_f16_bits, np.uint16)
    b = _c(bias_f16_bits, np.uint16)
    out = np.zeros((rows, cols), np.float32)
    lib.oracle_dequant_q4(_ptr(qq), _ptr(s), _ptr(b), rows, cols, group, _ptr(out))
    return out


def dequant(q, scale_f16_bits, bias_f16_bits, cols, bits, group=64):
    """Affine `bits`-bit rows [rows, cols*bits/32] uint32 -> fp32 [rows, cols] (4 or 8)."""
    if bits not in (4, 8):
        raise ValueError("bits must be 4 or 8")
    lib = _load()
    qq = _c(q, np.uint32)
    rows = qq.size // (cols * bits // 32)
    s = _c(scale_f16_bits, np.uint16)
    b = _c(bias_f16_bits, np.uint16)
    out = np.zeros((rows, cols), np.float32)
    lib.oracle_dequant(bits, _ptr(qq), _ptr(s), _ptr(b), rows, cols, group, _ptr(out))
    return out


def route_softmax(logits, top_k):
    """Softmax route on fp32 logits [..., E]: (inds int32, scores fp32) [..., K], weights
    renormalised over the selected experts (always)."""
    lib = _load()
    lg = _c(logits, np.float32)
    E = lg.shape[-1]
    rows = lg.size // E if E else 0
    inds = np.zeros(lg.shape[:-1] + (top_k,), np.int32)
    scores = np.zeros(lg.shape[:-1] + (top_k,), np.float32)
    if lib.oracle_route_softmax(_ptr(lg), rows, E, top_k, _ptr(inds), _ptr(scores)) != 0:
        raise ValueError("oracle_route_softmax rejected its arguments")
    return inds, scores


def indexer_topk(scores, k, lengths=None, want_mask=False):
    """DSA indexer selection on fp32 scores [rows, n]: int32 [rows, k] positions of the
    min(k, n_r) largest valid scores (positions j < n_r, n_r = lengths[r] or n), ascending,
    padded with -1; with want_mask also the uint8 [rows, n] mask of the selection."""
    lib = _load()
    sc = _c(scores, np.float32)
    if sc.ndim != 2:
        raise ValueError("scores must be [rows, n]")
    rows, n = sc.shape
    ln = None if lengths is None else _c(lengths, np.int32)
    inds = np.zeros((rows, k), np.int32)
    mask = np.zeros((rows, n), np.uint8) if want_mask else None
    if lib.oracle_indexer_topk(_ptr(sc), rows, n, n, _ptr(ln), k, _ptr(inds), _ptr(mask),
                               n) != 0:
        raise ValueError("oracle_indexer_topk rejected its arguments")
    return (inds, mask) if want_mask else inds


def moe_layer(x_bits, inds, scores, experts, shared=None, rows=None, group=64,
              shared_gate=None):
    """Dense per-token MoE layer; returns fp32 y for the listed token rows.

    x_bits: uint16 bf16 bits [T, d].  experts: dict with 'bits' (16, 8 or 4) and, for 16,
    'gate','up','down' uint16 bf16 bits ([E,I,d],[E,I,d],[E,d,I]); for 8 / 4, 'gate','up',
    'down' uint32 packed plus 'gate_s','gate_b',... fp16 bits, and optionally 'group' (the
    inputs per scale; default `group`).  shared: dict of bf16 bits 'gate','up','down'
    ([I,d],[I,d],[d,I]) or None.
    """
    lib = _load()
    x = _c(x_bits, np.uint16)
    T, d = x.shape
    ind = _c(inds, np.int32)
    sc = _c(scores, np.float32)
    K = ind.shape[1]
    bits = int(experts["bits"])
    group = int(experts.get("group", group))
    if bits == 16:
        g, u, dn = (_c(experts[k], np.uint16) for k in ("gate", "up", "down"))
        E, I = g.shape[0], g.shape[1]
        gs = gb = us = ub = ds = db = None
    else:
        g, u, dn = (_c(experts[k], np.uint32) for k in ("gate", "up", "down"))
        E, I = g.shape[0], g.shape[1]
        gs, gb, us, ub, ds, db = (_c(experts[k], np.uint16) for k in
                                  ("gate_s", "gate_b", "up_s", "up_b", "down_s", "down_b"))
    if shared is not None:
        sg, su, sd = (_c(shared[k], np.uint16) for k in ("gate", "up", "down"))
    else:
        sg = su = sd = None
    rws = np.arange(T, dtype=np.int64) if rows is None else _c(rows, np.int64)
    sgv = None if shared_gate is None else _c(shared_gate, np.uint16)
    y = np.zeros((len(rws), d), np.float32)
    rc = lib.oracle_moe_layer_rows(
        _ptr(x), T, d, I, E, K, _ptr(ind), _ptr(sc), bits, group,
        _ptr(g), _ptr(gs), _ptr(gb), _ptr(u), _ptr(us), _ptr(ub), _ptr(dn), _ptr(ds), _ptr(db),
        1 if shared is not None else 0,
        _ptr(sg), None, None, _ptr(su), None, None, _ptr(sd), None, None,
        _ptr(sgv), _ptr(rws), len(rws), _ptr(y))
    if rc != 0:
        raise ValueError("oracle_moe_layer_rows: bad expert index or allocation failure")
    return y


def bf16_to_f32(h: int) -> float:
    return _load().oracle_bf16_to_f32(h)


def f16_to_f32(h: int) -> float:
    return _load().oracle_f16_to_f32(h)
