"""Test-side helpers: comparison rules of the parity tests and the near-tie detector.

Near ties: two candidates whose biased scores (or group scores) differ by less than 1e-6
can legitimately be ordered differently by two fp32 sigmoid implementations (CUDA expf
and the host libm agree to a few ulp only), so rows whose K-th and (K+1)-th biased scores,
or whose topk_group-th and next group scores, differ by a nonzero amount under 1e-6 are
counted, reported and left out of the bit-exactness verdict.  Exact ties (gap 0) stay in:
both sides see identical values there and break the tie by the lower index.
"""
import numpy as np
import torch

NEAR_TIE = 1e-6


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16/fp16 tensor, on the host."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def near_tie_rows(logits, bias, top_k, n_group, topk_group):
    lg = np.asarray(logits, np.float32).astype(np.float64)
    s = 1.0 / (1.0 + np.exp(-lg))
    b = s + np.asarray(bias, np.float32).astype(np.float64)[None, :]
    rows, E = b.shape
    flag = np.zeros(rows, bool)
    if n_group > 1 and n_group - topk_group > 0:
        eg = E // n_group
        g = np.sort(b.reshape(rows, n_group, eg), axis=2)
        gs = g[:, :, -1] + g[:, :, -2]
        order = np.sort(gs, axis=1)[:, ::-1]
        gap = order[:, topk_group - 1] - order[:, topk_group]
        flag |= (gap > 0) & (gap < NEAR_TIE)
        # mask the dropped groups as the gate does (stable order, ties to lower index)
        rank = np.argsort(-gs, axis=1, kind="stable")
        keep = np.zeros_like(gs, bool)
        np.put_along_axis(keep, rank[:, :topk_group], True, axis=1)
        b = np.where(np.repeat(keep, eg, axis=1), b, 0.0)
    if top_k < E:
        srt = np.sort(b, axis=1)[:, ::-1]
        gap = srt[:, top_k - 1] - srt[:, top_k]
        flag |= (gap > 0) & (gap < NEAR_TIE)
    return flag


def check_route(gpu_inds, gpu_scores, ref_inds, ref_scores, ties):
    """Indices bit-exact and weights within 1e-6 relative on every non-near-tie row."""
    gi, gs = np.asarray(gpu_inds), np.asarray(gpu_scores)
    ri, rs = np.asarray(ref_inds), np.asarray(ref_scores)
    ok = ~np.asarray(ties, bool)
    mism = np.where(ok & np.any(gi != ri, axis=1))[0]
    assert mism.size == 0, f"{mism.size} non-tie rows route differently, first {mism[:5]}"
    rel = np.abs(gs[ok] - rs[ok]) / np.maximum(np.abs(rs[ok]), 1e-30)
    assert rel.size == 0 or rel.max() <= 1e-6, f"weight rel err {rel.max():.3e}"
    return int((~ok).sum())


def check_layer(got, ref, max_tol=1e-2, mean_tol=5e-3):
    """max|d| <= max_tol * max|ref| and mean|d| / mean|ref| <= mean_tol."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got)), "non-finite output"
    d = np.abs(got - ref)
    mx = d.max() / np.abs(ref).max()
    mean = d.mean() / np.abs(ref).mean()
    assert mx <= max_tol and mean <= mean_tol, f"max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def oracle_experts(data_experts, uniq=None):
    """Host copies (bit patterns) of the stacked expert weights, optionally only the
    experts in `uniq` (index tensor), in the oracle's input format."""
    ex = data_experts
    sel = (lambda t: t) if uniq is None else (lambda t: t.index_select(0, uniq))
    if ex["bits"] == 16:
        return {"bits": 16, **{k: bits(sel(ex[k])) for k in ("gate", "up", "down")}}
    o = {"bits": ex["bits"], "group": ex.get("group", 64)}
    for k in ("gate", "up", "down"):
        o[k] = sel(ex[k]).cpu().numpy().view(np.uint32)
        o[k + "_s"] = bits(sel(ex[k + "_s"]))
        o[k + "_b"] = bits(sel(ex[k + "_b"]))
    return o


def oracle_shared(shared):
    return None if shared is None else {k: bits(shared[k]) for k in ("gate", "up", "down")}
