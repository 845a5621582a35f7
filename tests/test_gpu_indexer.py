"""GPU parity of the DSA indexer selection (moe_indexer_topk) against the oracle: selected
positions and masks bit-exact ("SwiftLM issue #139", "What needs building" items 1 and 3).

Sizes cover every launch shape of the kernel: one CTA per row with the keys in shared
memory, clusters of 2..8 CTAs per row, rows too long to cache (keys re-read per pass), the
inert regime (n_r <= k), ragged causal lengths, strided rows, bf16 scores, exact ties,
NaN and signed zeros."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_moe_layer_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check(scores, k, lengths=None):
    gi, gm = binding.indexer_topk(scores, k, lengths=lengths, want_mask=True)
    torch.cuda.synchronize()
    sc = scores.float().cpu().numpy()
    ln = None if lengths is None else lengths.cpu().numpy()
    ri, rm = oracle.indexer_topk(sc, k, lengths=ln, want_mask=True)
    gi, gm = gi.cpu().numpy(), gm.cpu().numpy()
    bad = np.nonzero((gi != ri).any(1))[0]
    assert bad.size == 0, f"rows {bad[:5]} differ: {gi[bad[0]][:8]} vs {ri[bad[0]][:8]}"
    assert np.array_equal(gm, rm)
    return gi


@pytest.mark.parametrize("rows,n,k", [
    (5, 100, 8), (37, 5000, 256), (3, 16384, 2048), (4, 16385, 2048), (3, 40000, 2048),
    (2, 131072, 2048), (2, 140000, 2048), (3, 1000, 1000), (3, 999, 1000), (6, 777, 1),
    (2, 70000, 30000),
])
def test_indexer_topk_shapes(rows, n, k):
    g = torch.Generator(device=DEV).manual_seed(rows * 7 + n)
    _check(torch.randn(rows, n, generator=g, device=DEV), k)


def test_indexer_topk_rows_too_long_to_cache():
    # rows longer than 8 x 16384 keys: the keys stay in global memory (L2), sparse rows take
    # the sampled window, dense ones the full radix select
    g = torch.Generator(device=DEV).manual_seed(11)
    _check(torch.randn(3, 200000, generator=g, device=DEV), 2048)
    _check((torch.randn(3, 150000, generator=g, device=DEV) * 2).to(torch.bfloat16), 1024)
    big = torch.randn(2, 160003, generator=g, device=DEV)
    _check(big[:, 3:], 700)  # misaligned rows: scalar loads
    ties = torch.randint(-3, 4, (3, 140000), generator=g, device=DEV).float()
    _check(ties, 2048)
    _check(torch.randn(2, 140000, generator=g, device=DEV), 40000)  # dense: no window
    # a window wider than one CTA's candidate buffer: each CTA keeps its own candidates
    _check(torch.randn(2, 1 << 20, generator=g, device=DEV), 2048)


def test_indexer_topk_workload_scores_small():
    w = inputs.INDEXER_WORKLOADS["dsa_small_R37_N5000"]
    _check(inputs.gen_indexer_scores(w, DEV, seed=1), w.k)


def test_indexer_topk_exact_ties_and_bf16():
    g = torch.Generator(device=DEV).manual_seed(3)
    # integer scores: thousands of positions tie with the threshold, lowest positions win,
    # across the segments of a cluster
    _check(torch.randint(-4, 5, (4, 50000), generator=g, device=DEV).float(), 2048)
    _check(torch.randint(0, 3, (3, 3000), generator=g, device=DEV).float(), 700)
    # bf16 scores (8 mantissa bits: heavy ties), 16-byte vectors of 8 elements
    _check((torch.randn(5, 20000, generator=g, device=DEV) * 3).to(torch.bfloat16), 2048)
    _check((torch.randn(3, 1001, generator=g, device=DEV)).to(torch.bfloat16), 100)
    # all equal: the first k positions
    gi = _check(torch.zeros(2, 9000, device=DEV), 512)
    assert np.array_equal(gi[0], np.arange(512))


def test_indexer_topk_nan_and_signed_zero():
    g = torch.Generator(device=DEV).manual_seed(4)
    sc = torch.randn(4, 6000, generator=g, device=DEV)
    sc[0, ::3] = float("nan")
    sc[1] = 0.0
    sc[1, ::2] = -0.0
    sc[2, :5000] = float("nan")
    sc[3, ::7] = float("inf")
    sc[3, 1::7] = float("-inf")
    _check(sc, 1200)


def test_indexer_topk_causal_lengths_and_strided_rows():
    g = torch.Generator(device=DEV).manual_seed(5)
    rows, n, k = 300, 3000, 256
    big = torch.randn(rows, n + 13, generator=g, device=DEV)
    sc = big[:, :n]  # row stride n + 13: scalar loads
    lengths = (n - rows + torch.arange(rows, device=DEV) + 1).to(torch.int32)
    _check(sc, k, lengths)
    ragged = torch.randint(-5, n + 50, (rows,), generator=g, device=DEV).to(torch.int32)
    ragged[:3] = torch.tensor([0, k, k + 1], dtype=torch.int32)
    _check(sc, k, ragged)
    # lengths that leave whole cluster segments empty
    long_sc = torch.randn(4, 100000, generator=g, device=DEV)
    _check(long_sc, 2048, torch.tensor([100000, 30000, 2049, 17000], dtype=torch.int32,
                                       device=DEV))


def test_indexer_topk_full_decode_workload():
    w = inputs.INDEXER_WORKLOADS["dsa_decode_B64_N131072"]
    _check(inputs.gen_indexer_scores(w, DEV, seed=0), w.k)


def test_indexer_topk_full_prefill_workload_sampled_rows():
    w = inputs.INDEXER_WORKLOADS["dsa_prefill_L8192"]
    sc = inputs.gen_indexer_scores(w, DEV, seed=0)
    ln = inputs.indexer_lengths(w, DEV)
    gi, gm = binding.indexer_topk(sc, w.k, lengths=ln, want_mask=True)
    torch.cuda.synchronize()
    rows = np.r_[0:4, 2040:2056, np.random.RandomState(0).randint(0, w.rows, 40), w.rows - 3:w.rows]
    ri, rm = oracle.indexer_topk(sc[rows].cpu().numpy(), w.k, lengths=ln[rows].cpu().numpy(),
                                 want_mask=True)
    assert np.array_equal(gi[rows].cpu().numpy(), ri)
    assert np.array_equal(gm[rows].cpu().numpy(), rm)
    # every row: the selection count is min(k, n_r) and the mask agrees with the indices
    cnt = (gi >= 0).sum(1).cpu()
    assert torch.equal(cnt, torch.clamp(ln.cpu().long(), max=w.k))
    assert torch.equal(gm.sum(1).cpu().long(), cnt.long())


def test_indexer_topk_empty_and_rejection():
    binding.indexer_topk(torch.zeros(0, 16, device=DEV), 4)
    gi = binding.indexer_topk(torch.zeros(3, 0, device=DEV), 4)
    torch.cuda.synchronize()
    assert torch.all(gi == -1)
    inds = torch.full((2, 3), -7, dtype=torch.int32, device=DEV)
    with pytest.raises(binding.MoeError):
        binding.indexer_topk(torch.zeros(2, 16, device=DEV), 0, inds=inds)
    torch.cuda.synchronize()
    assert torch.all(inds == -7)
