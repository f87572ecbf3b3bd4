"""Pins for the oracle's content-based block selection.

* block means: within the pairwise-summation error bound of the exact fp64
  mean (numpy), and exact when the block's values are all equal;
* block scores: within the error bound of the exact fp64 dot product of the
  pooled vectors; the stated order (two fused multiply-add chains) replayed
  exactly in rational arithmetic with one rounding per step;
* selection: equal to numpy's lexsort over (score desc, index asc) on the same
  scores (library routine); planted clusters whose answer is known by
  construction; all-equal scores pick the smallest indices (tie rule); the
  diagonal is always present; every selected non-diagonal score >= every
  unselected score.

Selection rule: "the model predicts importance scores and picks top-k" ("How
Do Sparse Attention Kernels Work in GPU Clusters?", section "What Exactly Is
a Sparse Attention Kernel?"), on mean-pooled routing features ("The Only
Guide You Need for Sparse Attention Kernels", section "Flash-MSA"), plus the
diagonal block.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

import bsa_inputs
import oracle

U = 2.0 ** -24


def rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("bs", [16, 64, 128])
def test_block_means_error_bound(bs):
    BH, N, D = 3, bs * 6, 64
    x = rand_bf16((BH, N, D), 1, 3.0)
    got = oracle.block_means(bsa_inputs.bf16_bits(x), bs)
    xd = x.double().numpy().reshape(BH, N // bs, bs, D)
    exact = xd.mean(2)
    bound = np.ceil(np.log2(bs)) * U * np.abs(xd).sum(2) / bs * 1.01 + 1e-30
    assert np.all(np.abs(got - exact) <= bound)
    c = torch.full((1, bs * 2, D), 1.5, dtype=torch.bfloat16)
    np.testing.assert_array_equal(oracle.block_means(bsa_inputs.bf16_bits(c), bs), 1.5)


def test_block_scores_error_bound_and_order():
    rng = np.random.default_rng(3)
    BH, nb, D = 2, 9, 128
    qb = rng.standard_normal((BH, nb, D)).astype(np.float32)
    kb = rng.standard_normal((BH, nb, D)).astype(np.float32)
    got = oracle.block_scores(qb, kb)
    exact = np.einsum("bid,bjd->bij", qb.astype(np.float64), kb.astype(np.float64))
    mag = np.einsum("bid,bjd->bij", np.abs(qb).astype(np.float64), np.abs(kb).astype(np.float64))
    assert np.all(np.abs(got - exact) <= (D // 2 + 2) * U * mag * 1.01)
    # the stated order replayed in exact rational arithmetic with one
    # round-to-nearest-even to fp32 per fused multiply-add: a_c over d = c
    # (mod 2), then a0 + a1
    for (bh, i, j) in [(b, i, (5 * i + 3 * b + 1) % nb) for b in range(BH) for i in range(0, nb, 2)]:
        a = [Fraction(0), Fraction(0)]
        for d in range(D):
            a[d % 2] = Fraction(float(f32_round(Fraction(float(qb[bh, i, d])) * Fraction(float(kb[bh, j, d])) + a[d % 2])))
        want = f32_round(a[0] + a[1])
        assert got[bh, i, j] == want, (bh, i, j)


def f32_round(x: Fraction) -> np.float32:
    """x rounded once to the nearest fp32 (ties to even); normal range."""
    if x == 0:
        return np.float32(0.0)
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    m = x / Fraction(2) ** (e - 23)  # in [2^23, 2^24)
    mi = m.numerator // m.denominator
    rem = m - mi
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and mi % 2 == 1):
        mi += 1
    return np.float32(sign * float(Fraction(mi) * Fraction(2) ** (e - 23)))


def test_f32_round_reference():
    # the helper above against cases with a known answer
    assert f32_round(Fraction(1)) == np.float32(1.0)
    one_ulp = Fraction(1, 2 ** 23)
    assert f32_round(1 + one_ulp / 2) == np.float32(1.0)              # tie, even stays
    assert f32_round(1 + one_ulp * 3 / 2) == np.float32(1 + 2 * 2.0 ** -23)  # tie, odd rounds up
    assert f32_round(Fraction(-3, 10)) == np.float32(-0.3)
    rng = np.random.default_rng(0)
    for x in rng.standard_normal(200):
        assert f32_round(Fraction(float(x))) == np.float32(x)        # numpy's cast rounds once from fp64


def lexsort_select(scores, topk, include_diag):
    BH, nb, _ = scores.shape
    rows = []
    for bh in range(BH):
        for i in range(nb):
            order = np.lexsort((np.arange(nb), -scores[bh, i].astype(np.float64)))
            sel = set(order[:topk].tolist())
            if include_diag:
                sel.add(i)
            rows.append(sorted(sel))
    return rows


@pytest.mark.parametrize("topk,diag", [(4, True), (1, True), (6, False), (12, True)])
def test_selection_matches_lexsort(topk, diag):
    rng = np.random.default_rng(topk)
    BH, nb = 3, 12
    s = rng.standard_normal((BH, nb, nb)).astype(np.float32)
    s[0, 2, :] = 0.5                       # a row of ties
    s[1, 3, 5] = s[1, 3, 6] = s[1, 3].max() + 1  # a tie at the top
    rp, ci = oracle.topk_csr_from_scores(s, topk, diag)
    got = [ci[rp[r]:rp[r + 1]].tolist() for r in range(BH * nb)]
    assert got == lexsort_select(s, topk, diag)


def test_planted_clusters():
    """Key block j carries centroid j % 4 (a scaled basis vector), query block
    i centroid i % 4, no noise: row i's top-8 are exactly the 8 key blocks of
    its own centroid."""
    B, H, nb, bs, D, topk = 1, 2, 32, 16, 64, 8
    N = nb * bs
    q = torch.zeros((B, H, N, D))
    k = torch.zeros((B, H, N, D))
    for blk in range(nb):
        q[:, :, blk * bs:(blk + 1) * bs, blk % 4] = 8.0
        k[:, :, blk * bs:(blk + 1) * bs, blk % 4] = 8.0
    rp, ci, scores = oracle.topk_csr(bsa_inputs.bf16_bits(q.to(torch.bfloat16)),
                                     bsa_inputs.bf16_bits(k.to(torch.bfloat16)), bs, topk, True)
    assert np.all(np.isin(scores, [0.0, 64.0]))
    for r in range(B * H * nb):
        i = r % nb
        assert ci[rp[r]:rp[r + 1]].tolist() == [j for j in range(nb) if j % 4 == i % 4]


def test_all_ties_pick_smallest_indices_plus_diagonal():
    BH, nb, topk = 2, 20, 5
    s = np.zeros((BH, nb, nb), np.float32)
    rp, ci = oracle.topk_csr_from_scores(s, topk, True)
    for r in range(BH * nb):
        i = r % nb
        want = sorted(set(range(topk)) | {i})
        assert ci[rp[r]:rp[r + 1]].tolist() == want


def test_selection_invariants_on_clustered_inputs():
    w = bsa_inputs.small_workload(bsa_inputs.workload("content_topk"), B=1, H=2, N=64 * 48)
    d = bsa_inputs.make_qkv(w)
    rp, ci, s = oracle.topk_csr(bsa_inputs.bf16_bits(d["q"]), bsa_inputs.bf16_bits(d["k"]),
                                w.block, w.topk, True)
    nb = w.n_blocks
    for r in range(w.B * w.H * nb):
        bh, i = divmod(r, nb)
        row = ci[rp[r]:rp[r + 1]]
        assert w.topk <= len(row) <= w.topk + 1
        assert i in row and np.all(np.diff(row) > 0)
        non_diag = [j for j in row if j != i] if len(row) == w.topk + 1 else list(row)
        unsel = np.setdiff1d(np.arange(nb), row)
        if len(unsel):
            assert s[bh, i, non_diag].min() >= s[bh, i, unsel].max()
