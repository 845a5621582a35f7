"""GPU parity of the gate (moe_route_deepseek) and the dispatch (moe_permute) against the
oracle: indices and permutation bit-exact, weights within 1e-6 relative."""
import os

import numpy as np
import pytest
import torch

import oracle
from deepseek_moe_layer_gb300 import binding, inputs

from support import check_route, near_tie_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(logits, bias, K, G, tg, norm, scale):
    gi, gs = binding.route_deepseek(logits, bias, K, G, tg, norm, scale)
    torch.cuda.synchronize()
    lg = logits.float().cpu().numpy()
    b = bias.cpu().numpy()
    ri, rs = oracle.route(lg, b, K, G, tg, norm, scale)
    ties = near_tie_rows(lg.reshape(-1, lg.shape[-1]), b, K, G, tg)
    n = check_route(gi.cpu().numpy().reshape(-1, K), gs.cpu().numpy().reshape(-1, K),
                    ri.reshape(-1, K), rs.reshape(-1, K), ties)
    return n


@pytest.mark.parametrize("p", inputs.ROUTING["passes"], ids=["grouped", "flat"])
def test_routing_workload_16384x256(p):
    logits, bias = inputs.gen_routing(device=DEV, seed=0)
    n = _run(logits, bias, K=p["top_k"], G=p["n_group"],
             tg=p["topk_group"], norm=p["norm_topk_prob"], scale=p["routed_scaling_factor"])
    print(f"near-tie rows: {n} of {logits.shape[0]}")
    assert n < logits.shape[0] // 100


@pytest.mark.parametrize("E,G,tg,K", [
    (16, 4, 2, 4), (16, 1, 1, 16), (8, 4, 1, 1), (32, 8, 3, 6), (64, 8, 4, 8),
    (96, 4, 2, 8), (96, 12, 5, 7), (160, 8, 4, 8), (48, 16, 5, 3), (256, 8, 4, 8),
    (256, 1, 1, 32), (512, 32, 8, 16), (1024, 16, 4, 32), (1024, 1, 1, 1), (20, 10, 3, 5),
    (128, 4, 2, 8), (128, 2, 1, 5), (256, 4, 3, 7), (64, 1, 1, 8), (256, 8, 8, 8), (64, 2, 1, 1),
])
@pytest.mark.parametrize("norm", [True, False])
def test_route_shapes(E, G, tg, K, norm):
    g = torch.Generator(device=DEV).manual_seed(E * 131 + K)
    logits = torch.randn(777, E, generator=g, device=DEV) * 2
    bias = torch.randn(E, generator=g, device=DEV) * 0.3
    _run(logits, bias, K, G, tg, norm, 2.5)


@pytest.mark.parametrize("E,G,tg,K", [(16, 4, 2, 4), (12, 3, 1, 5), (64, 8, 2, 12), (96, 12, 5, 7),
                                     (64, 8, 2, 8), (128, 4, 2, 8), (256, 8, 4, 8), (256, 2, 1, 6)])
def test_route_exact_ties(E, G, tg, K):
    # integer logits and quarter-integer biases: many exact ties between experts and groups
    g = torch.Generator(device=DEV).manual_seed(E + 7 * K)
    logits = torch.randint(-2, 3, (500, E), generator=g, device=DEV).float()
    bias = torch.randint(-2, 3, (E,), generator=g, device=DEV).float() / 4
    n = _run(logits, bias, K, G, tg, True, 1.0)
    # sigma(a) + sigma(-a) = 1 exactly in real arithmetic, so group sums such as
    # sigma(2) + sigma(-2) and sigma(1) + sigma(-1) tie mathematically but round apart:
    # those rows are near ties (excluded above); every other row matched bit for bit
    assert n <= logits.shape[0] // 20
    # all-equal logits: selection is the K lowest indices of the kept groups
    _run(torch.zeros(3, E, device=DEV), torch.zeros(E, device=DEV), K, G, tg, True, 1.0)


@pytest.mark.parametrize("E,G,tg,K", [(256, 8, 4, 8), (256, 1, 1, 8), (128, 4, 2, 8),
                                     (64, 8, 4, 16), (256, 8, 4, 5), (256, 4, 3, 7)])
def test_route_winners_crowded_into_one_run(E, G, tg, K):
    """Rows whose largest scores crowd into 3, 4 or 8 neighbouring experts of one aligned run
    of eight (a lane of the gate holds such a run, and a lane giving more than three winners
    takes the exact re-scanning rounds), and the same rows with every kept score negative
    (bias - 2), where the dropped groups' zeros lead in index order."""
    g = torch.Generator(device=DEV).manual_seed(E * 7 + K)
    rows = 600
    logits = torch.randn(rows, E, generator=g, device=DEV)
    start = torch.randint(0, E // 8, (rows,), generator=g, device=DEV) * 8
    cnt = torch.tensor([3, 4, 8], device=DEV)[torch.arange(rows, device=DEV) % 3]
    off = torch.arange(8, device=DEV)
    cols = start[:, None] + off[None, :]
    vals = 6 + torch.rand(rows, 8, generator=g, device=DEV)
    logits.scatter_(1, cols, torch.where(off[None, :] < cnt[:, None], vals, logits.gather(1, cols)))
    bias = torch.randn(E, generator=g, device=DEV) * 0.1
    assert _run(logits, bias, K, G, tg, True, 2.5) <= rows // 50
    assert _run(logits, bias - 2.0, K, G, tg, True, 2.5) <= rows // 50


def test_route_nan_and_signed_zero():
    """NaN logits rank below every number (their experts and all-NaN groups are the last
    choices) and -0 == +0 (sigma(-0) and sigma(+0) tie, the lower expert index first), on
    both sides (the reading of the gate's comparisons for values the pages leave open)."""
    g = torch.Generator(device=DEV).manual_seed(12)
    E = 256
    logits = torch.randn(300, E, generator=g, device=DEV) * 2
    logits[::3, ::7] = float("nan")        # scattered NaNs
    logits[1::3, 32:64] = float("nan")     # a whole group of NaNs
    logits[2::3, 5] = -0.0
    logits[2::3, 6] = 0.0
    logits[2::3, 7:40] = -30.0             # the +-0 pair among the top scores of its rows
    bias = torch.zeros(E, device=DEV)
    _run(logits, bias, 8, 8, 4, True, 2.5)
    _run(logits, bias, 8, 1, 1, False, 1.0)
    gi, _ = _softmax_check(logits, 8)
    assert not torch.isnan(logits.gather(1, gi.long())).any()


def test_route_bf16_logits_and_leading_dims():
    g = torch.Generator(device=DEV).manual_seed(3)
    logits = torch.randn(4, 33, 256, generator=g, device=DEV).to(torch.bfloat16)
    bias = torch.randn(256, generator=g, device=DEV) * 0.05
    _run(logits, bias, 8, 8, 4, True, 2.5)


def test_route_case_b():
    path = os.path.join(os.path.dirname(__file__), "golden", "case_b_inputs.txt")
    vals = [float(l) for l in open(path)
            if l.strip() and not l.startswith("#")]
    lg = torch.tensor(vals[:16], dtype=torch.float32, device=DEV)[None]
    b = torch.tensor(vals[16:], dtype=torch.float32, device=DEV)
    for K in (1, 2, 4, 8):
        for tg in (1, 2, 3, 4):
            assert _run(lg, b, K, 4, tg, True, 2.5) == 0


def test_route_empty_rows():
    inds = torch.full((0, 4), -5, dtype=torch.int32, device=DEV)
    binding.route_deepseek(torch.zeros(0, 16, device=DEV), torch.zeros(16, device=DEV), 4, 4, 2,
                           True, 1.0, inds=inds)
    torch.cuda.synchronize()


def test_route_rejection_leaves_outputs_untouched():
    inds = torch.full((5, 3), -7, dtype=torch.int32, device=DEV)
    scores = torch.full((5, 3), -7.0, device=DEV)
    with pytest.raises(binding.MoeError):
        binding.route_deepseek(torch.zeros(5, 16, device=DEV), torch.zeros(16, device=DEV), 3, 4,
                               5, True, 1.0, inds=inds, scores=scores)
    torch.cuda.synchronize()
    assert torch.all(inds == -7) and torch.all(scores == -7)


# ------------------------------------------------------------------------------------
# softmax route: top-K by logit, weights renormalised over the selection
# ------------------------------------------------------------------------------------

def _softmax_check(logits, K):
    gi, gs = binding.route_softmax(logits, K)
    torch.cuda.synchronize()
    ri, rs = oracle.route_softmax(logits.float().cpu().numpy(), K)
    assert np.array_equal(gi.cpu().numpy(), ri)
    # both sides take exp in fp32; the library exponentials differ by a few ulp
    np.testing.assert_allclose(gs.cpu().numpy(), rs, rtol=2e-6, atol=1e-12)
    s = gs.cpu().numpy().sum(-1)
    assert np.all(np.abs(s - 1) < 1e-5)
    return gi, gs


@pytest.mark.parametrize("E,K", [(8, 1), (16, 4), (60, 6), (64, 8), (128, 8), (256, 8),
                                 (1024, 32), (5, 5)])
def test_softmax_route_shapes(E, K):
    g = torch.Generator(device=DEV).manual_seed(E * 17 + K)
    _softmax_check(torch.randn(555, E, generator=g, device=DEV) * 3, K)


def test_softmax_route_ties_and_bf16():
    g = torch.Generator(device=DEV).manual_seed(9)
    # integer logits: exact ties resolved to the lower expert index on both sides
    gi, _ = _softmax_check(torch.randint(-2, 3, (300, 24), generator=g, device=DEV).float(), 5)
    # all-equal logits: experts 0..K-1, each weight 1/K
    gi, gs = _softmax_check(torch.zeros(4, 12, device=DEV), 3)
    assert np.array_equal(gi.cpu().numpy(), np.tile(np.arange(3, dtype=np.int32), (4, 1)))
    # bf16 logits with leading dimensions
    _softmax_check((torch.randn(7, 9, 64, generator=g, device=DEV) * 2).to(torch.bfloat16), 4)


def test_softmax_route_empty_and_rejection():
    binding.route_softmax(torch.zeros(0, 16, device=DEV), 4)
    inds = torch.full((5, 17), -7, dtype=torch.int32, device=DEV)
    with pytest.raises(binding.MoeError):
        binding.route_softmax(torch.zeros(5, 16, device=DEV), 17, inds=inds)
    torch.cuda.synchronize()
    assert torch.all(inds == -7)


# ------------------------------------------------------------------------------------
# dispatch
# ------------------------------------------------------------------------------------

def _perm_check(inds_t, E):
    c, o, p, v = binding.permute(inds_t, E)
    torch.cuda.synchronize()
    rc, ro, rp, rv = oracle.permute(inds_t.cpu().numpy(), E)
    assert np.array_equal(c.cpu().numpy(), rc)
    assert np.array_equal(o.cpu().numpy(), ro)
    assert np.array_equal(p.cpu().numpy(), rp)
    assert np.array_equal(v.cpu().numpy(), rv)


@pytest.mark.parametrize("T,K,E", [(1, 1, 1), (3, 2, 5), (64, 4, 16), (128, 8, 256),
                                   (1000, 6, 33), (8192, 8, 256), (16384, 8, 256), (50, 8, 1024)])
def test_permute_uniform(T, K, E):
    g = torch.Generator(device=DEV).manual_seed(T + K + E)
    _perm_check(torch.randint(0, E, (T, K), generator=g, device=DEV, dtype=torch.int32), E)


def test_permute_skewed_and_single_expert():
    g = torch.Generator(device=DEV).manual_seed(1)
    z = torch.distributions.Categorical(probs=1.0 / torch.arange(1, 257).float() ** 1.1)
    inds = z.sample((8192, 8)).int().to(DEV)
    _perm_check(inds, 256)
    _perm_check(torch.full((5000, 4), 7, dtype=torch.int32, device=DEV), 16)


def test_permute_empty():
    c, o, p, v = binding.permute(torch.zeros(0, 8, dtype=torch.int32, device=DEV), 16)
    torch.cuda.synchronize()
    assert int(c.sum()) == 0 and int(o[-1]) == 0


def test_permute_out_of_range_ids_are_not_dispatched():
    g = torch.Generator(device=DEV).manual_seed(5)
    inds = torch.randint(0, 16, (300, 4), generator=g, device=DEV, dtype=torch.int32)
    inds[3, 1] = -1
    inds[100, 0] = 16
    inds[299, 3] = 1 << 20
    c, o, p, v = binding.permute(inds, 16)
    torch.cuda.synchronize()
    flat = inds.cpu().numpy().reshape(-1)
    valid = (flat >= 0) & (flat < 16)
    ref = sorted(np.where(valid)[0].tolist(), key=lambda q: (flat[q], q))
    assert int(o[-1]) == valid.sum()
    assert p.cpu().numpy()[: valid.sum()].tolist() == ref
    vv = v.cpu().numpy()
    assert np.all(vv[~valid] == -1)
    assert np.array_equal(vv[ref], np.arange(len(ref)))
