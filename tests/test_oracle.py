"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests re-types the oracle's own formulas: the routing selection is checked
by brute-force enumeration of subsets under the dominance order, the dispatch by a library
sort, the FFN by float64 matrix evaluation in numpy, the scalar conversions by numpy /
torch over every bit pattern, and the gate against the invariants the gate's PR states
("feat(engine): E1 DeepSeek-style MoE gate (sigmoid, group top-k, bias) (#108)", sections
"Algorithm", "Tests", and the review's "What looks solid" / "Non-issues").
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------------------------
# scalar conversions
# ------------------------------------------------------------------------------------

def test_bf16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.int64).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([oracle.bf16_to_f32(int(b)) for b in bits[::7]], np.float32)
    r = ref[::7]
    nan = np.isnan(r)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), r[~nan].view(np.uint32))


def test_f16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.int64).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ------------------------------------------------------------------------------------
# the gate
# ------------------------------------------------------------------------------------

def _sig(logits):
    """The oracle's fp32 sigmoid values, read through a pass-through configuration
    (n_group=1, top_k=E, no renorm, scale 1: the weights are the sigmoid values)."""
    lg = np.asarray(logits, np.float32).reshape(-1, np.shape(logits)[-1])
    E = lg.shape[1]
    inds, sc = oracle.route(lg, np.zeros(E, np.float32), E, 1, 1, False, 1.0)
    out = np.zeros_like(lg)
    np.put_along_axis(out, inds.astype(np.int64), sc, axis=1)
    return out.reshape(np.shape(logits))


def test_sigmoid_within_two_ulp_of_exact():
    x = np.linspace(-30, 30, 20001).astype(np.float32)
    got = _sig(x[None, :])[0]
    exact = 1.0 / (1.0 + np.exp(-x.astype(np.float64)))
    ulp = np.spacing(exact.astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(got.astype(np.float64) - exact) <= 2 * ulp)


def _dominates(va, ia, vb, ib):
    """a strictly precedes b: larger value, NaN lowest, equal values -> lower index."""
    if math.isnan(va) or math.isnan(vb):
        if math.isnan(va) and math.isnan(vb):
            return ia < ib
        return math.isnan(vb)
    return va > vb or (va == vb and ia < ib)


def _best_subset(values, k):
    """The unique k-subset every member of which precedes every non-member (brute force
    over all subsets)."""
    n = len(values)
    hits = []
    for S in itertools.combinations(range(n), k):
        Ss = set(S)
        if all(_dominates(values[a], a, values[b], b)
               for a in S for b in range(n) if b not in Ss):
            hits.append(S)
    assert len(hits) == 1
    return hits[0]


def brute_route(logits, bias, top_k, n_group, topk_group, norm, scale):
    s = _sig(logits[None, :])[0]
    E = len(s)
    biased = (s + np.asarray(bias, np.float32)).astype(np.float32)
    if n_group > 1 and n_group - topk_group > 0:
        eg = E // n_group
        gs = []
        for g in range(n_group):
            vals = biased[g * eg:(g + 1) * eg]
            # the largest sum over pairs of distinct members equals top1 + top2
            gs.append(max(np.float32(vals[i]) + np.float32(vals[j])
                          for i in range(eg) for j in range(eg) if i != j))
        kept = _best_subset([float(v) for v in gs], topk_group)
        for g in range(n_group):
            if g not in kept:
                biased[g * eg:(g + 1) * eg] = np.float32(0.0)
    sel = _best_subset([float(v) for v in biased], top_k)
    sel = sorted(sel, key=lambda e: (-float(biased[e]), e))
    w = np.array([s[e] for e in sel], np.float32)
    if top_k > 1 and norm:
        tot = np.float32(0.0)
        for v in w:
            tot = np.float32(tot + v)
        w = (w / tot).astype(np.float32)
    w = (w * np.float32(scale)).astype(np.float32)
    return np.array(sel, np.int32), w


def _case_params(E):
    out = []
    for G in [g for g in (1, 2, 3, 4) if E % g == 0 and (g == 1 or E // g >= 2)]:
        for tg in range(1, G + 1):
            for K in (1, 2, 3, 4):
                if K <= E:
                    out.append((K, G, tg))
    return out


@pytest.mark.parametrize("E", [4, 6, 8, 12])
def test_route_matches_brute_force_with_ties(E):
    rng = np.random.RandomState(E)
    for trial in range(6):
        # small-integer logits and quarter-integer bias force exact ties of all kinds
        logits = rng.randint(-2, 3, size=E).astype(np.float32)
        bias = (rng.randint(-2, 3, size=E) / 4.0).astype(np.float32)
        if trial == 0:
            bias[:] = 0.0
        for (K, G, tg) in _case_params(E):
            for norm in (False, True):
                bi, bw = brute_route(logits, bias, K, G, tg, norm, 2.5)
                oi, ow = oracle.route(logits[None], bias, K, G, tg, norm, 2.5)
                assert np.array_equal(oi[0], bi), (logits, bias, K, G, tg)
                assert np.array_equal(ow[0].view(np.uint32), bw.view(np.uint32))


def test_route_matches_brute_force_continuous():
    rng = np.random.RandomState(7)
    for _ in range(40):
        E = 12
        logits = rng.randn(E).astype(np.float32)
        bias = (0.3 * rng.randn(E)).astype(np.float32)
        for (K, G, tg) in [(4, 4, 2), (3, 3, 1), (2, 2, 2), (4, 1, 1), (1, 6, 3)]:
            bi, bw = brute_route(logits, bias, K, G, tg, True, 1.5)
            oi, ow = oracle.route(logits[None], bias, K, G, tg, True, 1.5)
            assert np.array_equal(oi[0], bi)
            assert np.array_equal(ow[0].view(np.uint32), bw.view(np.uint32))


def _case_b():
    vals = [float(l) for l in open(os.path.join(GOLDEN, "case_b_inputs.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(vals) == 32
    return np.array(vals[:16], np.float32), np.array(vals[16:], np.float32)


def test_case_b_inputs_regenerate():
    g, b = _case_b()
    rs = np.random.RandomState(42)
    assert np.array_equal(g, rs.randn(16).astype(np.float32))
    assert np.array_equal(b, (0.5 * rs.randn(16)).astype(np.float32))


@pytest.mark.parametrize("K,tg", [(k, t) for k in (1, 2, 4, 6, 8) for t in (1, 2, 3, 4)])
def test_case_b_n_group_4_brute_force(K, tg):
    g, b = _case_b()
    bi, bw = brute_route(g, b, K, 4, tg, True, 2.5)
    oi, ow = oracle.route(g[None], b, K, 4, tg, True, 2.5)
    assert np.array_equal(oi[0], bi)
    assert np.array_equal(ow[0].view(np.uint32), bw.view(np.uint32))


def test_bias_changes_selection_but_not_values():
    # "scores + bias ... selection only"; weights come from the pre-bias sigmoid
    logits = np.array([2.0, 1.9, 0.0, -1.0, 0.5, 0.4, -2.0, 1.0], np.float32)
    nob = np.zeros(8, np.float32)
    bias = np.array([0, 0, 3.0, 0, 0, 0, 3.0, 0], np.float32)
    i0, w0 = oracle.route(logits[None], nob, 2, 1, 1, False, 1.0)
    i1, w1 = oracle.route(logits[None], bias, 2, 1, 1, False, 1.0)
    assert list(i0[0]) == [0, 1] and list(i1[0]) == [2, 6]
    s = 1.0 / (1.0 + np.exp(-logits.astype(np.float64)))
    assert np.allclose(w1[0], s[[2, 6]], rtol=1e-6)
    # and with renormalisation the weights are the unbiased ones, renormalised
    i2, w2 = oracle.route(logits[None], bias, 2, 1, 1, True, 1.0)
    assert np.allclose(w2[0], s[[2, 6]] / s[[2, 6]].sum(), rtol=1e-6)


def test_top_k_1_norm_is_noop():
    rng = np.random.RandomState(3)
    for _ in range(20):
        logits = rng.randn(16).astype(np.float32)
        bias = (0.2 * rng.randn(16)).astype(np.float32)
        ia, wa = oracle.route(logits[None], bias, 1, 4, 2, True, 2.5)
        ib, wb = oracle.route(logits[None], bias, 1, 4, 2, False, 2.5)
        assert np.array_equal(ia, ib) and np.array_equal(wa, wb)
        e = ia[0, 0]
        assert abs(wa[0, 0] - 2.5 / (1 + math.exp(-float(logits[e])))) <= 1e-6 * 2.5


def test_group_wins_on_top2_sum_not_max():
    # group 0 holds the single largest expert; group 1 has the larger top-2 sum
    logits = np.array([6.0, -6.0, -6.0, -6.0, 2.0, 2.0, -6.0, -6.0], np.float32)
    bias = np.zeros(8, np.float32)
    inds, _ = oracle.route(logits[None], bias, 2, 2, 1, False, 1.0)
    assert sorted(inds[0].tolist()) == [4, 5]
    # with max-pooling the winner would have been group 0
    s = 1 / (1 + np.exp(-logits.astype(np.float64)))
    assert s[0] > s[4] and s[0] + s[1] < s[4] + s[5]


def test_k_drop_zero_equals_no_grouping():
    rng = np.random.RandomState(11)
    for _ in range(30):
        logits = rng.randn(3, 32).astype(np.float32)
        bias = (0.1 * rng.randn(32)).astype(np.float32)
        for G in (2, 4, 8):
            a = oracle.route(logits, bias, 6, G, G, True, 2.5)
            b = oracle.route(logits, bias, 6, 1, 1, True, 2.5)
            assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_masked_experts_hold_zero_and_stay_selectable():
    # dropped group is set to exactly 0.0, which beats a kept expert whose biased score
    # is negative (the review's "Non-issues": identical to the upstream gate).
    logits = np.array([-8.0, -8.0, -8.0, -8.0, 0.0, 0.0, -8.0, -8.0], np.float32)
    bias = np.array([-1.0, -1.0, -1.0, -1.0, -1.0, -0.2, -1.0, -1.0], np.float32)
    # group sums: g0 ~ -2.0, g1 = (0.5-1) + (0.5-0.2) = -0.2 -> keep g1, drop g0
    inds, w = oracle.route(logits[None], bias, 3, 2, 1, False, 1.0)
    # kept: e5 (0.3), e4 (-0.5), e6/e7 (~-1.0); dropped group 0 experts are 0.0 > -0.5
    assert inds[0].tolist() == [5, 0, 1]
    s = 1 / (1 + np.exp(-logits.astype(np.float64)))
    assert np.allclose(w[0], s[[5, 0, 1]], rtol=1e-6)


def test_closed_form_single_group_single_expert():
    rng = np.random.RandomState(5)
    logits = rng.randn(50, 10).astype(np.float32)
    bias = (0.5 * rng.randn(10)).astype(np.float32)
    inds, w = oracle.route(logits, bias, 1, 1, 1, False, 3.0)
    s = 1 / (1 + np.exp(-logits.astype(np.float64)))
    assert np.array_equal(inds[:, 0], np.argmax(s + bias, axis=1))
    assert np.allclose(w[:, 0], 3.0 * s[np.arange(50), inds[:, 0]], rtol=1e-6)


def test_norm_sums_to_scale():
    rng = np.random.RandomState(8)
    logits = rng.randn(100, 64).astype(np.float32)
    bias = (0.1 * rng.randn(64)).astype(np.float32)
    _, w = oracle.route(logits, bias, 8, 8, 4, True, 2.5)
    assert np.allclose(w.astype(np.float64).sum(1), 2.5, rtol=1e-6)


def test_zero_sum_has_no_guard():
    # all selected sigmoid weights underflow to 0 -> 0/0 = NaN, matching the upstream
    # gate, which has no zero-sum guard (review issue 1, kept for parity)
    logits = np.full((1, 4), -200.0, np.float32)
    _, w = oracle.route(logits, np.zeros(4, np.float32), 2, 1, 1, True, 1.0)
    assert np.all(np.isnan(w))


def test_route_rejects_invalid_parameters():
    lg = np.zeros((1, 8), np.float32)
    b = np.zeros(8, np.float32)
    for (K, G, tg) in [(0, 1, 1), (9, 1, 1), (2, 3, 1), (2, 2, 0), (2, 2, 3), (2, 8, 1),
                       (2, 1, 2)]:
        with pytest.raises(ValueError):
            oracle.route(lg, b, K, G, tg, True, 1.0)


# ------------------------------------------------------------------------------------
# dispatch
# ------------------------------------------------------------------------------------

@pytest.mark.parametrize("T,K,E", [(1, 1, 1), (7, 3, 5), (64, 4, 16), (300, 8, 32)])
def test_permute_is_stable_sort(T, K, E):
    rng = np.random.RandomState(T + K)
    inds = rng.randint(0, E, size=(T, K)).astype(np.int32)
    counts, offsets, perm, inv = oracle.permute(inds, E)
    flat = inds.reshape(-1)
    ref = sorted(range(T * K), key=lambda p: (flat[p], p))
    assert perm.tolist() == ref
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    assert np.array_equal(inv[perm], np.arange(T * K))
    assert np.array_equal(inv, np.argsort(perm))


# ------------------------------------------------------------------------------------
# router linear, 4-bit dequantisation, FFN and the layer
# ------------------------------------------------------------------------------------

def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _f64(t):
    return t.to(torch.float64).numpy()


def test_router_logits_match_numpy():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(17, 96, generator=g).to(torch.bfloat16)
    w = (torch.randn(12, 96, generator=g) * 0.1).to(torch.bfloat16)
    off = torch.randn(12, generator=g)
    got = oracle.router_logits(_bits(x), _bits(w), off.numpy())
    ref = _f64(x) @ _f64(w).T + off.double().numpy()
    assert np.allclose(got, ref, rtol=1e-6, atol=1e-6)


def _unpack_q4(words, cols):
    """Independent unpacker on Python integers: element j sits in word j // 8 at bit
    offset 4 * (j % 8) (low nibble first)."""
    words = np.asarray(words, np.uint32)
    rows = words.shape[0]
    out = np.zeros((rows, cols), np.int64)
    for r in range(rows):
        for j in range(cols):
            out[r, j] = (int(words[r, j // 8]) >> (4 * (j % 8))) & 15
    return out


def test_q4_nibble_order_low_first():
    q = np.array([[0x76543210, 0xFEDCBA98]], np.uint32)
    one = np.array([[np.float16(1.0).view(np.uint16)]], np.uint16)
    zero = np.array([[np.float16(0.0).view(np.uint16)]], np.uint16)
    out = oracle.dequant_q4(q, one, zero, cols=16, group=16)
    assert out[0].tolist() == list(range(16))


def test_q4_dequant_affine_per_group():
    rng = np.random.RandomState(2)
    rows, cols, group = 3, 192, 64
    q = rng.randint(0, 2**32, size=(rows, cols // 8), dtype=np.uint64).astype(np.uint32)
    s = rng.uniform(0.005, 0.02, size=(rows, cols // group)).astype(np.float16)
    b = (0.1 * rng.randn(rows, cols // group)).astype(np.float16)
    got = oracle.dequant_q4(q, s.view(np.uint16), b.view(np.uint16), cols, group)
    codes = _unpack_q4(q, cols)
    sf = np.repeat(s.astype(np.float32), group, axis=1)
    bf = np.repeat(b.astype(np.float32), group, axis=1)
    ref = sf.astype(np.float64) * codes + bf
    assert np.allclose(got, ref, rtol=1e-6, atol=1e-7)
    # scale 1, bias 0: exactly the integer codes
    one = np.full((rows, cols // group), np.float16(1)).view(np.uint16)
    zero = np.zeros((rows, cols // group), np.uint16)
    assert np.array_equal(oracle.dequant_q4(q, one, zero, cols, group), codes.astype(np.float32))


def _rand_layer(T, d, I, E, K, seed, bits=16):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    ex = {"bits": bits}
    if bits == 16:
        for k, shp, fan in (("gate", (E, I, d), d), ("up", (E, I, d), d), ("down", (E, d, I), I)):
            ex[k] = (torch.randn(*shp, generator=g) / math.sqrt(fan)).to(torch.bfloat16)
    else:
        for k, (r, c) in (("gate", (I, d)), ("up", (I, d)), ("down", (d, I))):
            ex[k] = torch.randint(-2**31, 2**31, (E, r, c // 8), generator=g,
                                  dtype=torch.int64).to(torch.int32)
            ex[k + "_s"] = (torch.rand(E, r, c // 64, generator=g) * 0.015 + 0.005).half()
            ex[k + "_b"] = (torch.randn(E, r, c // 64, generator=g) * 0.1).half()
    sh = {k: (torch.randn(*shp, generator=g) / math.sqrt(fan)).to(torch.bfloat16)
          for k, shp, fan in (("gate", (I, d), d), ("up", (I, d), d), ("down", (d, I), I))}
    inds = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)]).int()
    scores = torch.rand(T, K, generator=g)
    return x, ex, sh, inds.numpy(), scores.numpy()


def _np_expert_weights(ex, e):
    if ex["bits"] == 16:
        return [_f64(ex[k][e]) for k in ("gate", "up", "down")]
    out = []
    for k in ("gate", "up", "down"):
        q = ex[k][e].numpy().view(np.uint32)
        cols = q.shape[1] * 8
        codes = _unpack_q4(q, cols)
        s = np.repeat(ex[k + "_s"][e].float().numpy().astype(np.float64), 64, axis=1)
        b = np.repeat(ex[k + "_b"][e].float().numpy().astype(np.float64), 64, axis=1)
        out.append(((s * codes).astype(np.float32) + b).astype(np.float32).astype(np.float64))
    return out


def _np_ffn(xv, wg, wu, wd):
    a = xv @ wg.T
    return (a / (1.0 + np.exp(-a)) * (xv @ wu.T)) @ wd.T


def _to_oracle_experts(ex):
    if ex["bits"] == 16:
        return {"bits": 16, **{k: _bits(ex[k]) for k in ("gate", "up", "down")}}
    o = {"bits": 4}
    for k in ("gate", "up", "down"):
        o[k] = ex[k].numpy().view(np.uint32)
        o[k + "_s"] = ex[k + "_s"].numpy().view(np.uint16)
        o[k + "_b"] = ex[k + "_b"].numpy().view(np.uint16)
    return o


@pytest.mark.parametrize("bits", [16, 4])
def test_layer_matches_numpy_float64(bits):
    T, d, I, E, K = 5, 128, 64, 6, 3
    x, ex, sh, inds, scores = _rand_layer(T, d, I, E, K, seed=bits, bits=bits)
    got = oracle.moe_layer(_bits(x), inds, scores, _to_oracle_experts(ex),
                           {k: _bits(v) for k, v in sh.items()})
    xs = _f64(x)
    ref = np.zeros((T, d))
    for t in range(T):
        for k in range(K):
            ref[t] += scores[t, k] * _np_ffn(xs[t], *_np_expert_weights(ex, inds[t, k]))
        ref[t] += _np_ffn(xs[t], _f64(sh["gate"]), _f64(sh["up"]), _f64(sh["down"]))
    err = np.abs(got - ref).max() / np.abs(ref).max()
    assert err < 1e-6, err


def test_layer_expert_major_equals_token_major():
    """The same layer computed expert by expert over the oracle's own dispatch."""
    T, d, I, E, K = 9, 64, 64, 5, 2
    x, ex, sh, inds, scores = _rand_layer(T, d, I, E, K, seed=3)
    got = oracle.moe_layer(_bits(x), inds, scores, _to_oracle_experts(ex), None)
    counts, offsets, perm, inv = oracle.permute(inds, E)
    xs = _f64(x)
    acc = np.zeros((T, d))
    for e in range(E):
        slots = perm[offsets[e]:offsets[e + 1]]
        if len(slots) == 0:
            continue
        toks = slots // K
        a = xs[toks] @ _f64(ex["gate"][e]).T
        h = a / (1 + np.exp(-a)) * (xs[toks] @ _f64(ex["up"][e]).T)
        o = h @ _f64(ex["down"][e]).T
        for j, p in enumerate(slots):
            acc[p // K] += scores.reshape(-1)[p] * o[j]
    assert np.abs(got - acc).max() <= 1e-6 * np.abs(acc).max()


def test_layer_all_experts_reduces_to_sigmoid_mixture():
    """K = E, no group drop, no renorm, scale 1: y = sum_e sigmoid(logit_e) FFN_e + shared."""
    T, d, I, E = 4, 64, 64, 4
    x, ex, sh, _, _ = _rand_layer(T, d, I, E, 1, seed=4)
    g = torch.Generator().manual_seed(9)
    wr = (torch.randn(E, d, generator=g) / 8).to(torch.bfloat16)
    logits = oracle.router_logits(_bits(x), _bits(wr))
    inds, w = oracle.route(logits, np.zeros(E, np.float32), E, 2, 2, False, 1.0)
    got = oracle.moe_layer(_bits(x), inds, w, _to_oracle_experts(ex),
                           {k: _bits(v) for k, v in sh.items()})
    xs = _f64(x)
    lg = xs @ _f64(wr).T
    ref = np.zeros((T, d))
    for t in range(T):
        for e in range(E):
            ref[t] += 1 / (1 + np.exp(-lg[t, e])) * _np_ffn(xs[t], *_np_expert_weights(ex, e))
        ref[t] += _np_ffn(xs[t], _f64(sh["gate"]), _f64(sh["up"]), _f64(sh["down"]))
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max()


def test_silu_sign_and_gate_up_roles():
    """One expert, d = I = 1-like shapes: gate pre-activation a, up value u ->
    out = w_down * silu(a) * u with silu(a) = a / (1 + e^-a)."""
    d = I = 8
    x = torch.zeros(1, d); x[0, 0] = 1.0
    for a, u in ((2.0, 1.0), (-2.0, 1.0), (1.0, -3.0)):
        wg = torch.zeros(1, I, d); wg[0, 0, 0] = a
        wu = torch.zeros(1, I, d); wu[0, 0, 0] = u
        wd = torch.zeros(1, d, I); wd[0, 3, 0] = 0.5
        ex = {"bits": 16, "gate": _bits(wg.to(torch.bfloat16)), "up": _bits(wu.to(torch.bfloat16)),
              "down": _bits(wd.to(torch.bfloat16))}
        y = oracle.moe_layer(_bits(x.to(torch.bfloat16)), np.zeros((1, 1), np.int32),
                             np.ones((1, 1), np.float32), ex, None)
        assert abs(y[0, 3] - 0.5 * a / (1 + math.exp(-a)) * u) < 1e-6
        assert np.count_nonzero(y) == 1


# ------------------------------------------------------------------------------------
# softmax route and gated shared expert
# ------------------------------------------------------------------------------------

def test_softmax_route_matches_numpy_float64():
    rng = np.random.RandomState(21)
    for E, K in ((8, 1), (16, 4), (64, 6), (256, 8)):
        lg = (rng.randn(40, E) * 2).astype(np.float32)
        inds, w = oracle.route_softmax(lg, K)
        l64 = lg.astype(np.float64)
        p = np.exp(l64 - l64.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        ref_i = np.argsort(-p, axis=1, kind="stable")[:, :K]
        assert np.array_equal(inds, ref_i)
        ps = np.take_along_axis(p, ref_i, axis=1)
        assert np.allclose(w, ps / ps.sum(1, keepdims=True), rtol=1e-6, atol=0)


def test_softmax_route_ties_brute_force():
    rng = np.random.RandomState(22)
    for _ in range(30):
        lg = rng.randint(-2, 3, size=10).astype(np.float32)
        for K in (1, 2, 3, 5):
            sel = _best_subset([float(v) for v in lg], K)
            sel = sorted(sel, key=lambda e: (-float(lg[e]), e))
            inds, w = oracle.route_softmax(lg[None], K)
            assert inds[0].tolist() == sel
            assert abs(float(w[0].astype(np.float64).sum()) - 1.0) < 1e-6


def test_softmax_route_shift_invariant_and_k1():
    rng = np.random.RandomState(23)
    lg = rng.randn(20, 32).astype(np.float32)
    i0, w0 = oracle.route_softmax(lg, 4)
    i1, w1 = oracle.route_softmax(lg + np.float32(3.0), 4)
    assert np.array_equal(i0, i1) and np.allclose(w0, w1, rtol=1e-5)
    _, wk1 = oracle.route_softmax(lg, 1)
    assert np.all(wk1 == 1.0)


def test_gated_shared_expert_matches_numpy():
    T, d, I, E, K = 4, 64, 64, 5, 2
    x, ex, sh, inds, scores = _rand_layer(T, d, I, E, K, seed=31)
    g = torch.Generator().manual_seed(32)
    wsg = (torch.randn(d, generator=g) / 8).to(torch.bfloat16)
    got = oracle.moe_layer(_bits(x), inds, scores, _to_oracle_experts(ex),
                           {k: _bits(v) for k, v in sh.items()}, shared_gate=_bits(wsg))
    xs = _f64(x)
    ref = np.zeros((T, d))
    for t in range(T):
        for k in range(K):
            ref[t] += scores[t, k] * _np_ffn(xs[t], *_np_expert_weights(ex, inds[t, k]))
        gate = 1 / (1 + np.exp(-(xs[t] @ _f64(wsg))))
        ref[t] += gate * _np_ffn(xs[t], _f64(sh["gate"]), _f64(sh["up"]), _f64(sh["down"]))
    assert np.abs(got - ref).max() <= 1e-6 * np.abs(ref).max()


def test_zero_shared_gate_halves_the_shared_expert():
    T, d, I, E, K = 3, 64, 64, 4, 2
    x, ex, sh, inds, scores = _rand_layer(T, d, I, E, K, seed=33)
    oe = _to_oracle_experts(ex)
    osh = {k: _bits(v) for k, v in sh.items()}
    none = oracle.moe_layer(_bits(x), inds, scores, oe, None).astype(np.float64)
    full = oracle.moe_layer(_bits(x), inds, scores, oe, osh).astype(np.float64)
    half = oracle.moe_layer(_bits(x), inds, scores, oe, osh,
                            shared_gate=np.zeros(d, np.uint16)).astype(np.float64)
    assert np.allclose(half, none + 0.5 * (full - none), rtol=1e-5, atol=1e-6)


# ------------------------------------------------------------------------------------
# DSA indexer top-k selection ("SwiftLM issue #139", "What needs building" items 1 and 3,
# and the inertness remark of "The test that makes this verifiable without real weights")
# ------------------------------------------------------------------------------------

def _np_topk_positions(row, k):
    """Independent statement: numpy's lexicographic sort on (position, -score) with NaN
    moved below every number."""
    v = np.where(np.isnan(row), -np.inf, row.astype(np.float64))
    nan_last = np.isnan(row).astype(np.int8)
    order = np.lexsort((np.arange(len(row)), -v, nan_last))
    return np.sort(order[:k])


def test_indexer_topk_matches_numpy_sort_with_ties():
    rng = np.random.RandomState(41)
    for n, k in ((1, 1), (7, 3), (64, 8), (300, 64), (1000, 257)):
        # integer scores: many exact ties at the threshold, broken by the lower position
        sc = rng.randint(-3, 4, size=(9, n)).astype(np.float32)
        got = oracle.indexer_topk(sc, k)
        for r in range(sc.shape[0]):
            ref = _np_topk_positions(sc[r], min(k, n))
            assert got[r, :len(ref)].tolist() == ref.tolist()
            assert np.all(got[r, len(ref):] == -1)


def test_indexer_topk_is_argpartition_set_for_distinct_scores():
    rng = np.random.RandomState(42)
    sc = rng.randn(12, 5000).astype(np.float32)
    k = 2048
    got = oracle.indexer_topk(sc, k)
    part = np.argpartition(sc, -k, axis=1)[:, -k:]  # the pages' primitive, kth = -k
    for r in range(sc.shape[0]):
        assert set(got[r].tolist()) == set(part[r].tolist())
        assert np.all(np.diff(got[r]) > 0)  # ascending positions


def test_indexer_topk_inert_at_or_below_k():
    rng = np.random.RandomState(43)
    for n in (1, 5, 2048):
        sc = rng.randn(3, n).astype(np.float32)
        got = oracle.indexer_topk(sc, 2048)
        assert np.array_equal(got[:, :n], np.tile(np.arange(n, dtype=np.int32), (3, 1)))
        assert np.all(got[:, n:] == -1)


def test_indexer_topk_causal_lengths_and_mask():
    rng = np.random.RandomState(44)
    L, k = 40, 8
    sc = rng.randn(L, L).astype(np.float32)
    lengths = np.arange(1, L + 1, dtype=np.int32)  # query r sees positions 0..r
    inds, mask = oracle.indexer_topk(sc, k, lengths=lengths, want_mask=True)
    for r in range(L):
        m = min(k, r + 1)
        ref = _np_topk_positions(sc[r, :r + 1], m)
        assert inds[r, :m].tolist() == ref.tolist() and np.all(inds[r, m:] == -1)
        want = np.zeros(L, np.uint8)
        want[ref] = 1
        assert np.array_equal(mask[r], want)  # selection AND causal: nothing beyond r


def test_indexer_topk_order_invariant_nan_and_signed_zero():
    rng = np.random.RandomState(45)
    sc = rng.randn(6, 200).astype(np.float32)
    sc[0, ::3] = np.nan
    sc[1, :] = 0.0
    sc[1, ::2] = -0.0  # -0 and +0 tie: the lowest positions win
    sc[2, :150] = np.nan  # fewer numbers than k: NaN positions fill the rest, lowest first
    k = 64
    got = oracle.indexer_topk(sc, k)
    assert got[1].tolist() == list(range(k))
    assert got[2].tolist() == sorted(list(range(150, 200)) + list(range(14)))
    for r in range(sc.shape[0]):
        sel = set(got[r].tolist())
        num = lambda j: -np.inf if np.isnan(sc[r, j]) else float(sc[r, j])
        lo_sel = min(num(j) for j in sel)
        hi_rest = max((num(j) for j in range(200) if j not in sel), default=-np.inf)
        assert lo_sel >= hi_rest  # every selected score >= every unselected one
    # k = 1 is the argmax, first occurrence on ties
    sc4 = rng.randint(0, 5, size=(50, 30)).astype(np.float32)
    assert np.array_equal(oracle.indexer_topk(sc4, 1)[:, 0], np.argmax(sc4, axis=1))


# ------------------------------------------------------------------------------------
# other quantisation widths and groups: 8-bit codes, groups of 32 / 64 / 128 inputs
# ------------------------------------------------------------------------------------

def _unpack_bytes(words, cols, bits):
    """Independent unpacker through numpy's little-endian memory view: for 8 bits the
    codes are the row's bytes in order; for 4 bits each byte holds two codes, low first."""
    raw = np.ascontiguousarray(np.asarray(words, np.uint32).astype("<u4")).view(np.uint8)
    raw = raw.reshape(raw.shape[0], -1)
    if bits == 8:
        return raw[:, :cols].astype(np.int64)
    out = np.empty((raw.shape[0], 2 * raw.shape[1]), np.int64)
    out[:, 0::2] = raw & 15
    out[:, 1::2] = raw >> 4
    return out[:, :cols]


def test_q8_byte_order_low_first():
    q = np.array([[0x03020100, 0x07060504, 0xFFFEFDFC, 0x80807F7F]], np.uint32)
    one = np.array([[np.float16(1.0).view(np.uint16)]], np.uint16)
    zero = np.array([[np.float16(0.0).view(np.uint16)]], np.uint16)
    out = oracle.dequant(q, one, zero, cols=16, bits=8, group=16)
    assert out[0].tolist() == [0, 1, 2, 3, 4, 5, 6, 7, 252, 253, 254, 255, 127, 127, 128, 128]


@pytest.mark.parametrize("bits,group", [(8, 32), (8, 64), (8, 128), (4, 32), (4, 128)])
def test_dequant_affine_widths_and_groups(bits, group):
    rng = np.random.RandomState(bits * 1000 + group)
    rows, cols = 3, 384
    q = rng.randint(0, 2**32, size=(rows, cols * bits // 32), dtype=np.uint64).astype(np.uint32)
    s = rng.uniform(0.005, 0.02, size=(rows, cols // group)).astype(np.float16)
    b = (0.1 * rng.randn(rows, cols // group)).astype(np.float16)
    got = oracle.dequant(q, s.view(np.uint16), b.view(np.uint16), cols, bits, group)
    codes = _unpack_bytes(q, cols, bits)
    sf = np.repeat(s.astype(np.float64), group, axis=1)
    bf = np.repeat(b.astype(np.float64), group, axis=1)
    assert np.allclose(got, sf * codes + bf, rtol=1e-6, atol=1e-7)
    # the neighbouring group's scale would show: groups differ
    wrong = np.repeat(np.roll(s, 1, axis=1).astype(np.float64), group, axis=1) * codes
    assert not np.allclose(got, wrong + bf, rtol=1e-3)
    one = np.full((rows, cols // group), np.float16(1)).view(np.uint16)
    zero = np.zeros((rows, cols // group), np.uint16)
    assert np.array_equal(oracle.dequant(q, one, zero, cols, bits, group), codes.astype(np.float32))
    if bits == 4:  # the 4-bit entry point agrees with the general one
        assert np.array_equal(oracle.dequant_q4(q, s.view(np.uint16), b.view(np.uint16), cols,
                                                group), got)


@pytest.mark.parametrize("bits,group", [(8, 64), (8, 32), (4, 128)])
def test_layer_quant_widths_match_numpy_float64(bits, group):
    T, d, I, E, K = 4, 256, 128, 5, 2
    g = torch.Generator().manual_seed(bits + group)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    ex, ref_w = {"bits": bits, "group": group}, {}
    for k, (r, c) in (("gate", (I, d)), ("up", (I, d)), ("down", (d, I))):
        q = torch.randint(-2**31, 2**31, (E, r, c * bits // 32), generator=g,
                          dtype=torch.int64).to(torch.int32).numpy().view(np.uint32)
        sc = (torch.rand(E, r, c // group, generator=g) * 0.01 + 0.002).half().numpy()
        bi = (torch.randn(E, r, c // group, generator=g) * 0.05).half().numpy()
        ex[k], ex[k + "_s"], ex[k + "_b"] = q, sc.view(np.uint16), bi.view(np.uint16)
        ref_w[k] = [(np.repeat(sc[e].astype(np.float64), group, 1) *
                     _unpack_bytes(q[e], c, bits)).astype(np.float32).astype(np.float64) +
                    np.repeat(bi[e].astype(np.float64), group, 1) for e in range(E)]
    inds = np.stack([np.random.RandomState(t).permutation(E)[:K] for t in range(T)]).astype(np.int32)
    scores = np.random.RandomState(9).rand(T, K).astype(np.float32)
    got = oracle.moe_layer(_bits(x), inds, scores, ex, None)
    xs = _f64(x)
    ref = np.zeros((T, d))
    for t in range(T):
        for kk in range(K):
            e = inds[t, kk]
            ref[t] += scores[t, kk] * _np_ffn(xs[t], ref_w["gate"][e], ref_w["up"][e],
                                             ref_w["down"][e])
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max()
