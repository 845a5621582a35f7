"""Throughput of the DeepSeek-V3-shaped MoE layer forward on GB300.

One step = one moe_forward call (router linear, gate, dispatch, token gather, gate/up
GEMM with SwiGLU, down GEMM, combine; shared expert included) on one batch of synthetic
tokens with device-resident random-init weights.  Default workload: DeepSeek-V3 shape,
decode T=128 (d=7168, 256 routed experts + 1 shared, I=2048, top-8 of 8 groups keep 4);
the prefill shape (T=8192, Zipf-skewed routing) is measured in the same run and reported
under "prefill".  Timing: CUDA events on the launch stream, W untimed warm-up steps, steps
summed between their own events; every step streams 0.9 - 10 GB of expert weights from HBM
(inputs larger than the 129 MB L2), and --l2-flush adds a 256 MB write before each step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs N independent replicas (the layer has no exchange step), one per rank under
torchrun; value = tokens of all ranks / max over ranks of the timed time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from deepseek_moe_layer_gb300 import binding, inputs  # noqa: E402

METRIC = "MoE-layer tokens/s (DSv3 shape, T=128 & T=8192); % of HBM/tensor roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the dominant kernel per
# algorithmic byte, from single-pass ncu captures of the full-size launches of these
# workloads (routing is deterministic, so a launch's traffic is fixed), keyed by workload
# with the hash of the GEMM sources the capture ran; a stale hash reports null.
NCU_TRAFFIC = {
    "dsv3_T128": {"src": "766546b89d3431a7", "ratio": 4619120854 / 4601413632},
    "dsv3_T8192_zipf": {"src": "766546b89d3431a7", "ratio": 10454055765 / 7935623168},
    "dsv3_q4_T32": {"src": "766546b89d3431a7", "ratio": 961363115 / 922812416},
    "dsv3_q8_T32": {"src": "766546b89d3431a7", "ratio": 1743873238 / 1686175744},
    "dsv3_q4_T4096_zipf": {"src": "766546b89d3431a7", "ratio": 3130795051 / 2521825280},
    "dsv3_q8_T4096_zipf": {"src": "766546b89d3431a7", "ratio": 5094885461 / 4107272192},
}


NEAR_TIE = 1e-6


def near_tie_count(logits, bias, top_k, n_group, topk_group):
    """Rows of fp32 router logits [rows, E] whose K-th and (K+1)-th biased scores, or whose
    topk_group-th and next group scores, differ by a nonzero amount under 1e-6: two fp32
    sigmoid implementations (device expf, host libm) may order such candidates differently,
    so the parity rules count them and leave them out of the bit-exact verdict.  Evaluated
    in float64 on the host from the device's own logits."""
    lg = np.asarray(logits, np.float32).astype(np.float64)
    b = 1.0 / (1.0 + np.exp(-lg)) + np.asarray(bias, np.float32).astype(np.float64)[None, :]
    rows, E = b.shape
    flag = np.zeros(rows, bool)
    if n_group > 1 and n_group - topk_group > 0:
        eg = E // n_group
        srt = np.sort(b.reshape(rows, n_group, eg), axis=2)
        gs = srt[:, :, -1] + srt[:, :, -2]
        order = np.sort(gs, axis=1)[:, ::-1]
        gap = order[:, topk_group - 1] - order[:, topk_group]
        flag |= (gap > 0) & (gap < NEAR_TIE)
        keep = np.zeros_like(gs, bool)
        np.put_along_axis(keep, np.argsort(-gs, axis=1, kind="stable")[:, :topk_group], True,
                          axis=1)
        b = np.where(np.repeat(keep, eg, axis=1), b, 0.0)
    if top_k < E:
        srt = np.sort(b, axis=1)[:, ::-1]
        gap = srt[:, top_k - 1] - srt[:, top_k]
        flag |= (gap > 0) & (gap < NEAR_TIE)
    return int(flag.sum())


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("gemm.cu", "common.cuh"):
        with open(os.path.join(ROOT, "deepseek_moe_layer_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 100 ms while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev):
        self.proc = None
        self.path = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
        except Exception:
            uuid = str(dev.index or 0)
        self.uuid = uuid

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        sm = np.array([r[0] for r in rows])
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3][1:5])
                          if v.lower() == "active"})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(r[1] for r in rows)),
                "power_w_max": float(max(r[2] for r in rows)), "samples": len(rows),
                "reasons": reasons}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(times, dev=None):
    """Element-wise maximum of this rank's timings over all ranks (identity without a process
    group): the slowest replica sets the job's time."""
    t = torch.tensor([float(v) for v in times], dtype=torch.float64)
    if torch.distributed.is_available() and torch.distributed.is_initialized() and \
            torch.distributed.get_world_size() > 1:
        backend = torch.distributed.get_backend()
        t = t.to(dev if backend == "nccl" else "cpu")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        t = t.cpu()
    return [float(v) for v in t]


def replica_throughput(world_size, steps, tokens_per_step, total_ms):
    """Whole-job tokens/s of `world_size` replicas, each timing `steps` steps of
    `tokens_per_step` tokens: all ranks' tokens over the slowest rank's time."""
    return world_size * steps * tokens_per_step / (total_ms / 1e3)


def algorithmic(w, counts):
    """Algorithmic bytes and FLOPs of one forward, from the measured expert loads."""
    T, d, I, E, K = w.T, w.d, w.I, w.E, w.top_k
    P = T * K
    hit = int((counts > 0).sum())
    nsh = 1 if w.shared else 0
    rows = P + (T if w.shared else 0)
    if w.bits == 16:
        wmat = I * d * 2                     # bytes of one [I, d] bf16 matrix
    else:                                    # codes + fp16 scale and bias per group
        wmat = I * d * w.bits // 8 + 2 * (I * d // w.group) * 2
    shmat = I * d * 2
    gate_up_w = hit * 2 * wmat + nsh * 2 * shmat
    down_w = hit * wmat + nsh * shmat
    out = {
        "experts_hit": hit,
        "gate_up_bytes": gate_up_w + rows * d * 2 + rows * I * 2,
        "down_bytes": down_w + rows * I * 2 + rows * d * 2,
        "gate_up_flops": 2.0 * rows * d * 2 * I,
        "down_flops": 2.0 * rows * I * d,
        "router_flops": 2.0 * T * d * E,
        "layer_bytes": gate_up_w + down_w + E * d * 2 + 2 * T * d * 2,
    }
    out["layer_flops"] = out["gate_up_flops"] + out["down_flops"] + out["router_flops"]
    return out


def time_routing(dev, replays=50):
    """The gate alone on the routing workload (16384 rows x 256 experts, fp32 logits): per
    pass, a CUDA graph of 16 route launches, each on its own copy of the logits (16 x 16.8 MB
    > L2, so every launch reads its logits from HBM), replayed `replays` times between CUDA
    events on the launch stream.  Launch overhead is comparable with the ~3 us kernel, which
    is why the launches are replayed from a graph."""
    logits, bias = inputs.gen_routing(device=dev, seed=0)
    rows, E = logits.shape
    nbuf = 16
    bufs = [logits] + [logits.clone() for _ in range(nbuf - 1)]
    out = {}
    stream = torch.cuda.Stream(dev)
    for p, name in zip(inputs.ROUTING["passes"], ("grouped", "flat")):
        K = p["top_k"]
        inds = torch.empty(rows, K, dtype=torch.int32, device=dev)
        scores = torch.empty(rows, K, dtype=torch.float32, device=dev)
        args = (K, p["n_group"], p["topk_group"], p["norm_topk_prob"],
                p["routed_scaling_factor"])
        with torch.cuda.stream(stream):
            for b in bufs[:3]:  # warm-up (loads the module, checks the device)
                binding.route_deepseek(b, bias, *args, inds=inds, scores=scores)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for b in bufs:
                binding.route_deepseek(b, bias, *args, inds=inds, scores=scores)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(replays):
                g.replay()
            z.record(stream)
        stream.synchronize()
        us = a.elapsed_time(z) * 1e3 / (replays * nbuf)
        nbytes = rows * E * 4 + rows * K * 8
        rf = roofline("hbm", nbytes / (us * 1e-6), load_peaks()[0], False)
        out[name] = {"us_per_launch": round(us, 3), "rows_per_s": round(rows / (us * 1e-6), 1),
                     "bytes": nbytes, "launches": replays * nbuf, "roofline": rf,
                     "roofline_frac": rf["frac"],
                     "near_ties": near_tie_count(logits.cpu().numpy(), bias.cpu().numpy(), K,
                                                 p["n_group"], p["topk_group"])}
    del bufs
    torch.cuda.empty_cache()
    return {"workload": f"routing_{rows}x{E}", "l2": "16 rotating copies of the logits "
            "(269 MB > L2); launches replayed from a CUDA graph",
            "kernel": "gate_kernel<8, 8, GC, 32> (GC = 8 grouped, 0 flat)", **out}


def time_indexer(dev, reps=20):
    """The DSA indexer selection on its decode (64 rows x 131072 positions) and causal
    prefill (8192 x 8192, with the mask) workloads: launches over rotating score copies
    whose total exceeds L2, timed with CUDA events on the launch stream."""
    out = {}
    peaks = load_peaks()[0]
    for name, want_mask in (("dsa_decode_B64_N131072", False), ("dsa_prefill_L8192", True)):
        w = inputs.INDEXER_WORKLOADS[name]
        sc = inputs.gen_indexer_scores(w, dev, seed=0)
        ln = inputs.indexer_lengths(w, dev)
        nbuf = max(2, -(-(160 << 20) // (sc.numel() * 4)))
        bufs = [sc] + [sc.clone() for _ in range(nbuf - 1)]
        inds = torch.empty(w.rows, w.k, dtype=torch.int32, device=dev)
        mask = torch.empty(w.rows, w.n, dtype=torch.uint8, device=dev) if want_mask else None
        stream = torch.cuda.current_stream(dev)
        for b in bufs[:3]:
            binding.indexer_topk(b, w.k, lengths=ln, want_mask=want_mask, inds=inds, mask=mask)
        torch.cuda.synchronize(dev)
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(reps):
            binding.indexer_topk(bufs[i % nbuf], w.k, lengths=ln, want_mask=want_mask,
                                 inds=inds, mask=mask)
        z.record(stream)
        torch.cuda.synchronize(dev)
        us = a.elapsed_time(z) * 1e3 / reps
        valid = w.rows * w.n if ln is None else int(ln.clamp(max=w.n).long().sum())
        nbytes = valid * 4 + w.rows * w.k * 4 + (w.rows * w.n if want_mask else 0)
        out[name] = {"rows": w.rows, "n": w.n, "k": w.k, "causal": w.causal, "mask": want_mask,
                     "us_per_launch": round(us, 2), "rows_per_s": round(w.rows / (us * 1e-6), 1),
                     "bytes": nbytes, "launches": reps,
                     "roofline": roofline("hbm", nbytes / (us * 1e-6), peaks, False)}
        del bufs, sc
        torch.cuda.empty_cache()
    out["kernel"] = "indexer_topk_kernel<false> (fp32 scores)"
    out["l2"] = "rotating score copies totalling > 160 MB (> L2) between launches"
    return out


def make_layer(w, data):
    return binding.MoELayer(data["w_router"], data["bias"], data["experts"], data["shared"],
                            w.top_k, w.n_group, w.topk_group, w.norm_topk_prob,
                            w.routed_scaling_factor, data["logit_offset"])


def time_layer(w, data, steps, warmup, dev, sampler=None, flush_l2=False):
    """Device time of `steps` forwards, then per-kernel times from `steps` more.

    The first loop is the measurement: CUDA events recorded on the launch stream between
    consecutive forwards, nothing inside them, so the layer's kernels overlap their
    neighbours' tails as in use (programmatic dependent launch).  The second loop records
    the library's phase events between the kernels (which serialises them) for the
    per-kernel durations the roofline uses.  Every step streams its expert weights (0.9 - 10
    GB) from HBM, far more than the 129 MB L2, so no flush is needed; with flush_l2 a 256 MB
    write precedes each step (its dirty lines are then written back to HBM during the next
    step, a cost that is not the layer's)."""
    layer = make_layer(w, data)
    x = data["x"]
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    y = torch.empty(w.T, w.d, dtype=torch.bfloat16, device=dev)
    for _ in range(warmup):
        layer(x, y=y)
    torch.cuda.synchronize(dev)
    binding.device_status()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
    if torch.distributed.is_initialized():
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    for s in range(steps):
        if flush_l2:
            flush.zero_()
        marks[2 * s].record(stream)
        layer(x, y=y)
        marks[2 * s + 1].record(stream)
    torch.cuda.synchronize(dev)
    if torch.distributed.is_initialized():
        torch.distributed.barrier()
    binding.device_status()
    per_step = np.array([marks[2 * s].elapsed_time(marks[2 * s + 1]) for s in range(steps)])
    # per-kernel times: the same steps with the phase events
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(steps)]
    for s in range(steps):
        if flush_l2:
            flush.zero_()
        binding.set_phase_events(evs[s])
        layer(x, y=y)
    binding.set_phase_events(None)
    torch.cuda.synchronize(dev)
    binding.device_status()
    phased = np.array([evs[s][0].elapsed_time(evs[s][7]) for s in range(steps)])
    phases = {name: float(np.mean([evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(steps)]))
              for i, name in enumerate(binding.PHASES)}
    _, inds, _, logits = layer(x, want_intermediates=True)
    torch.cuda.synchronize(dev)
    counts = np.bincount(inds.cpu().numpy().reshape(-1), minlength=w.E)
    ties = near_tie_count(logits.cpu().numpy(), data["bias"].cpu().numpy(), w.top_k, w.n_group,
                          w.topk_group)
    # seven kernels per forward; from 8192 token-expert pairs the dispatch is two launches
    per_fwd = 7 + (1 if w.T * w.top_k >= 8192 else 0)
    return dict(total_ms=float(per_step.sum()), ms=float(per_step.mean()), phases=phases,
                phased_ms=float(phased.mean()), counts=counts, launches=per_fwd * steps,
                near_ties=ties)


def time_e2e(w, data, steps, warmup, dev):
    """Same forward through the public API with the tokens in pinned host memory: each
    step copies x host->device, runs the layer, copies y device->host."""
    layer = make_layer(w, data)
    xh = data["x"].cpu().pin_memory()
    yh = torch.empty(w.T, w.d, dtype=torch.bfloat16).pin_memory()
    xd = torch.empty_like(data["x"])
    yd = torch.empty(w.T, w.d, dtype=torch.bfloat16, device=dev)

    def step():
        xd.copy_(xh, non_blocking=True)
        layer(xd, y=yd)
        yh.copy_(yd, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        step()
    b.record()
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b)
    return dict(ms=ms, h2d=xh.numel() * 2, d2h=yh.numel() * 2)


def roofline(kind, achieved_per_s, peaks, sustained, traffic=None):
    if kind == "hbm":
        peak = peaks["hbm_gbs"]
        a = achieved_per_s / 1e9
        unit = "GB/s"
    else:
        peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        a = achieved_per_s / 1e12
        unit = "TFLOP/s"
    return {"bound": kind, "achieved": round(a, 1), "peak": peak, "unit": unit,
            "frac": round(a / peak, 4), "traffic": traffic}


def kernel_roofline(w, t, alg, peaks, src):
    """Roofline of the dominant kernel (the gate/up GEMM): HBM-bound when its bytes at
    peak bandwidth take longer than its FLOPs at peak tensor rate, else tensor-bound."""
    sec = t["phases"]["gate_up"] / 1e3
    t_hbm = alg["gate_up_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg["gate_up_flops"] / (peaks["bf16_tflops_sustained"] * 1e12)
    tr = NCU_TRAFFIC.get(w.name)
    traffic = (int(tr["ratio"] * alg["gate_up_bytes"])
               if tr and tr.get("src") == src else None)
    if t_hbm >= t_tc:
        r = roofline("hbm", alg["gate_up_bytes"] / sec, peaks, True, traffic)
        r["algorithmic"] = alg["gate_up_bytes"]
    else:
        r = roofline("tensor", alg["gate_up_flops"] / sec, peaks, True, traffic)
        r["algorithmic"] = alg["gate_up_flops"]
    r["kernel"] = "moe_gemm_kernel<kGateUp> (gate/up GEMM + SwiGLU)"
    r["ms"] = round(t["phases"]["gate_up"], 4)
    return r


def layer_roofline(alg, ms, peaks):
    sec = ms / 1e3
    t_hbm = alg["layer_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg["layer_flops"] / (peaks["bf16_tflops_sustained"] * 1e12)
    if t_hbm >= t_tc:
        return roofline("hbm", alg["layer_bytes"] / sec, peaks, True)
    return roofline("tensor", alg["layer_flops"] / sec, peaks, True)


# ---------------------------------------------------------------------------------------
# CPU oracle timing (baseline and the reference arm)
# ---------------------------------------------------------------------------------------

def _bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def oracle_inputs(w, data, rows):
    """Host copies of what the oracle needs for `rows` (only the experts they route to)."""
    import oracle
    xb = _bits(data["x"][torch.as_tensor(rows, device=data["x"].device)])
    wr = _bits(data["w_router"])
    off = None if data["logit_offset"] is None else data["logit_offset"].cpu().numpy()
    bias = data["bias"].cpu().numpy()
    lg = oracle.router_logits(xb, wr, off)
    inds, _ = oracle.route(lg, bias, w.top_k, w.n_group, w.topk_group, w.norm_topk_prob,
                           w.routed_scaling_factor)
    used = np.unique(inds)
    idx = torch.as_tensor(used, device=data["w_router"].device)
    ex = {"bits": data["experts"]["bits"]}
    for k, v in data["experts"].items():
        if isinstance(v, torch.Tensor):
            t = v.index_select(0, idx)
            ex[k] = t.cpu().numpy().view(np.uint32) if t.dtype == torch.int32 else _bits(t)
    remap = np.full(w.E, -1, np.int64)
    remap[used] = np.arange(len(used))
    sh = None if data["shared"] is None else {k: _bits(data["shared"][k])
                                              for k in ("gate", "up", "down")}
    return dict(xb=xb, wr=wr, off=off, bias=bias, ex=ex, sh=sh, remap=remap)


def oracle_step(w, h):
    """One timed oracle pass over the sampled tokens (router linear -> gate -> dispatch ->
    dense per-token layer), exactly as the oracle stands."""
    import oracle
    lg = oracle.router_logits(h["xb"], h["wr"], h["off"])
    inds, scores = oracle.route(lg, h["bias"], w.top_k, w.n_group, w.topk_group,
                                w.norm_topk_prob, w.routed_scaling_factor)
    E_used = int(h["remap"].max()) + 1
    loc = h["remap"][inds].astype(np.int32)
    oracle.permute(loc, E_used)
    return oracle.moe_layer(h["xb"], loc, scores, h["ex"], h["sh"])


def cpu_baseline(w, data, target_s=10.0):
    import oracle
    n = max(4, oracle.num_threads())
    rows = np.arange(min(w.T, n))
    h = oracle_inputs(w, data, rows)
    t0 = time.perf_counter()
    oracle_step(w, h)
    dt = time.perf_counter() - t0
    reps = max(1, min(int(target_s / max(dt, 1e-3)), 20))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_step(w, h)
    dt = time.perf_counter() - t0
    return {"value": round(len(rows) * reps / dt, 3), "unit": "tokens/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{len(rows)} tokens of {w.name} x {reps} passes (router linear, gate, "
                      f"dispatch, dense per-token expert loop incl. shared expert), "
                      f"{dt:.1f} s"}


# ---------------------------------------------------------------------------------------

def workload_data(name, dev, base=None):
    """Inputs of a layer workload; with `base`, its weights are reused (same shapes and
    width) and only the tokens, the bias and the logit offsets are drawn for `name`."""
    w = inputs.WORKLOADS[name]
    if base is None:
        return w, inputs.gen_layer(w, dev, seed=0)
    data = dict(base)
    data["x"] = inputs.gen_tokens(w, dev, seed=0)
    data["bias"] = inputs.gen_bias(w, dev, seed=0)
    data["logit_offset"] = inputs.zipf_offsets(w.E, dev, 0) if w.zipf else None
    return w, data


def run_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    src = kernel_source_hash()

    w, data = workload_data(args.workload, dev)
    do_pre = bool(args.prefill) and w.d == inputs.WORKLOADS[args.prefill].d and \
        w.E == inputs.WORKLOADS[args.prefill].E and w.bits == inputs.WORKLOADS[args.prefill].bits
    if do_pre:
        wp, dp = workload_data(args.prefill, dev, base=data)
    sampler = ClockSampler(dev)
    with sampler:  # clocks sampled across both timed loops
        t = time_layer(w, data, args.steps, args.warmup, dev, flush_l2=args.l2_flush)
        if do_pre:
            tp = time_layer(wp, dp, args.steps, args.warmup, dev, flush_l2=args.l2_flush)
    clocks = sampler.summary()
    e2e = time_e2e(w, data, args.steps, args.warmup, dev)
    alg = algorithmic(w, t["counts"])

    base_cpu = rank == 0 and ws == 1 and not args.no_cpu_baseline

    def summary(wx, tx, dx=None):
        """One workload's line.  Besides the nested roofline objects it carries their
        figures as plain numbers (a parser that keeps scalars only still sees them), the
        near-tie count of its routing, and, on rank 0 of a single-GPU run, the CPU oracle
        timed on a bounded sample of the same workload."""
        algx = algorithmic(wx, tx["counts"])
        kr = kernel_roofline(wx, tx, algx, peaks, src)
        lr = layer_roofline(algx, tx["ms"], peaks)
        out = {"workload": wx.name, "T": wx.T, "expert_bits": wx.bits,
               "value": round(wx.T / (tx["ms"] / 1e3), 1),
               "unit": "tokens/s", "ms_per_step": round(tx["ms"], 4),
               "experts_hit": algx["experts_hit"], "max_expert_load": int(tx["counts"].max()),
               "near_ties": tx["near_ties"],
               "roofline_bound": kr["bound"], "roofline_achieved": kr["achieved"],
               "roofline_peak": kr["peak"], "roofline_unit": kr["unit"],
               "roofline_frac": kr["frac"], "roofline_traffic": kr["traffic"],
               "gate_up_ms": kr["ms"], "ms_per_step_kernels_timed": round(tx["phased_ms"], 4),
               "layer_roofline_frac": lr["frac"],
               "layer_roofline_achieved": lr["achieved"], "layer_roofline_unit": lr["unit"],
               "phases_ms": {k: round(v, 4) for k, v in tx["phases"].items()},
               "roofline": kr, "layer_roofline": lr}
        if dx is not None and base_cpu:
            cb = cpu_baseline(wx, dx, target_s=4.0)
            out["cpu_baseline"] = cb
            out["cpu_baseline_tokens_per_s"] = cb["value"]
        return out

    pre = None
    if do_pre:
        pre = summary(wp, tp, dp)
        del dp
    # the same decode layer under near-uniform routing (bias at standard deviation 0.05):
    # the expert stream a uniform router touches
    uni = None
    if args.uniform and w.name == "dsv3_T128":
        wu, du = workload_data("dsv3_T128_uniform", dev, base=data)
        tu = time_layer(wu, du, args.steps, args.warmup, dev, flush_l2=args.l2_flush)
        uni = summary(wu, tu)
        del du
    # the affine 4-bit expert workloads (decode T=32, prefill T=4096 with Zipf routing)
    q4 = {}
    if args.q4 and w.d == 7168 and w.E == 256:
        wq, dq = workload_data("dsv3_q4_T32", dev)
        tq = time_layer(wq, dq, args.steps, args.warmup, dev, flush_l2=args.l2_flush)
        q4["q4_decode"] = summary(wq, tq, dq)
        if args.uniform:
            wqu, dqu = workload_data("dsv3_q4_T32_uniform", dev, base=dq)
            tqu = time_layer(wqu, dqu, args.steps, args.warmup, dev, flush_l2=args.l2_flush)
            q4["q4_decode_uniform"] = summary(wqu, tqu)
            del dqu
        wq2, dq2 = workload_data("dsv3_q4_T4096_zipf", dev, base=dq)
        tq2 = time_layer(wq2, dq2, args.steps, args.warmup, dev, flush_l2=args.l2_flush)
        q4["q4_prefill"] = summary(wq2, tq2, dq2)
        del dq, dq2
        torch.cuda.empty_cache()
    if args.q8 and w.d == 7168 and w.E == 256:
        wq, dq = workload_data("dsv3_q8_T32", dev)
        tq = time_layer(wq, dq, args.steps, args.warmup, dev, flush_l2=args.l2_flush)
        q4["q8_decode"] = summary(wq, tq, dq)
        wq2, dq2 = workload_data("dsv3_q8_T4096_zipf", dev, base=dq)
        tq2 = time_layer(wq2, dq2, args.steps, args.warmup, dev, flush_l2=args.l2_flush)
        q4["q8_prefill"] = summary(wq2, tq2, dq2)
        del dq, dq2
        torch.cuda.empty_cache()

    routing = time_routing(dev) if w.E == inputs.ROUTING["E"] else None
    indexer = time_indexer(dev) if args.indexer else None

    # aggregate over ranks: tokens of all ranks / max time
    total_ms, e2e_ms = max_over_ranks([t["total_ms"], e2e["ms"]], dev)
    value = replica_throughput(ws, args.steps, w.T, total_ms)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1/fan_in) random-init weights, N(0,1) tokens",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "I": w.I,
                   "top_k": w.top_k, "n_group": w.n_group, "topk_group": w.topk_group,
                   "shared_experts": 1 if w.shared else 0, "expert_bits": w.bits,
                   "parallelism": f"replicas x{ws}",
                   "l2": ("L2 flushed (256 MB write) before every timed step" if args.l2_flush
                          else "no flush: the expert weights streamed per step (4.6 GB "
                               "gate/up + 2.3 GB down at decode) exceed the 129 MB L2")},
        "roofline": kernel_roofline(w, t, alg, peaks, src),
        "layer_roofline": layer_roofline(alg, t["ms"], peaks),
        "peaks_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
        "phases_ms": {k: round(v, 4) for k, v in t["phases"].items()},
        "ms_per_step_kernels_timed": round(t["phased_ms"], 4),
        "experts_hit": alg["experts_hit"],
        "near_ties": t["near_ties"],
        "clocks": clocks,
        "e2e": {"value": round(ws * args.steps * w.T / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"]},
        "gpu_launches": t["launches"],
        "kernel_src": src,
    }
    if pre is not None:
        line["prefill"] = pre
    if uni is not None:
        line["decode_uniform"] = uni
    line.update(q4)
    if routing is not None:
        line["routing"] = routing
    if indexer is not None:
        line["indexer_topk"] = indexer
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, data)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    dev = torch.device(f"cuda:{local}") if torch.cuda.is_available() else torch.device("cpu")
    w, data = workload_data(args.workload, dev)
    n = max(4, oracle.num_threads())
    rows = np.arange(min(w.T, n))
    h = oracle_inputs(w, data, rows)
    for _ in range(args.warmup):
        oracle_step(w, h)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, h)
    dt = time.perf_counter() - t0
    v = len(rows) * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64",
        "data": "synthetic: seeded N(0,1/fan_in) random-init weights, N(0,1) tokens",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "I": w.I,
                   "top_k": w.top_k, "n_group": w.n_group, "topk_group": w.topk_group,
                   "shared_experts": 1 if w.shared else 0, "expert_bits": w.bits},
        "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "kind": "oracle",
                         "cores": oracle.num_threads(),
                         "sample": f"each step: {len(rows)} tokens of {w.name} through the "
                                   f"CPU oracle (router linear, gate, dispatch, dense "
                                   f"per-token experts + shared)"},
        "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dsv3_T128", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--prefill", default="dsv3_T8192_zipf")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2-flush", action="store_true",
                    help="write a 256 MB buffer before every timed layer step")
    ap.add_argument("--no-q8", dest="q8", action="store_false",
                    help="skip the affine 8-bit expert workloads")
    ap.add_argument("--no-indexer", dest="indexer", action="store_false",
                    help="skip the DSA indexer selection workloads")
    ap.add_argument("--no-q4", dest="q4", action="store_false",
                    help="skip the affine 4-bit expert workloads")
    ap.add_argument("--no-uniform", dest="uniform", action="store_false",
                    help="skip the near-uniform-routing decode workloads")
    args = ap.parse_args()
    if args.prefill in ("", "none"):
        args.prefill = None
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
