"""Pins for the oracle's pattern -> block-mask CSR (orc_pattern_csr).

Pinned against: hand-written golden rows and closed-form counts
(tests/golden/pattern_masks.json); the token-level sliding window of
"Flash MSA Sparse Attention vs Full Attention" (section "The Mechanics",
Mask[i][j] = 1 if |i - j| <= W, causal form j >= i - W and j <= i), which a
block size of 1 must reproduce exactly; and the covering rule (a block window
of w blocks is exactly the set of key blocks that a token window of w*bs
tokens touches), brute-forced.
"""

import json
import os

import numpy as np
import pytest

import bsa_inputs
import oracle
from oracle import brute

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pattern_masks.json")))
PATTERN_WORKLOADS = [w for w in bsa_inputs.WORKLOADS if not w.is_topk]


def rows_of(rp, ci):
    return [ci[rp[i]:rp[i + 1]].tolist() for i in range(len(rp) - 1)]


def test_tiny_rows_golden():
    w = bsa_inputs.workload("tiny_window_global")
    rp, ci = oracle.Pattern.from_workload(w).csr()
    assert rows_of(rp, ci) == GOLDEN["tiny_window_global"]["rows"]


@pytest.mark.parametrize("w", PATTERN_WORKLOADS, ids=lambda w: w.name)
def test_nnz_and_row_lengths_closed_form(w):
    g = GOLDEN[w.name]
    rp, ci = oracle.Pattern.from_workload(w).csr()
    lens = np.diff(rp)
    assert int(rp[-1]) == g["nnz_per_head"]
    assert int(lens.min()) == g["row_len_min"]
    assert int(lens.max()) == g["row_len_max"]
    # rows ascending, distinct, in range
    for i in range(w.n_blocks):
        row = ci[rp[i]:rp[i + 1]]
        assert np.all(np.diff(row) > 0)
        assert row.min() >= 0 and row.max() < w.n_blocks


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("W", [0, 1, 3, 7])
def test_block_size_one_is_token_window(causal, W):
    N = 40
    p = oracle.Pattern(N, window_left=W, window_right=W, causal=causal)
    rp, ci = p.csr()
    bm = brute.block_mask_from_csr(rp, ci, N)
    np.testing.assert_array_equal(bm, brute.token_window_mask(N, W, causal))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("w_blocks,bs", [(1, 4), (2, 8), (4, 4)])
def test_covering_rule(causal, w_blocks, bs):
    nb = 12
    N = nb * bs
    tok = brute.token_window_mask(N, w_blocks * bs, causal)
    touched = tok.reshape(nb, bs, nb, bs).any(axis=(1, 3))
    p = oracle.Pattern(nb, window_left=w_blocks, window_right=w_blocks, causal=causal)
    rp, ci = p.csr()
    np.testing.assert_array_equal(brute.block_mask_from_csr(rp, ci, nb), touched)


def test_global_blocks_and_rows():
    nb = 20
    G = (0, 7)
    p = oracle.Pattern(nb, window_left=1, window_right=1, causal=False, global_blocks=G,
                       global_rows_attend_all=True)
    bm = brute.block_mask_from_csr(*p.csr(), nb)
    for g in G:
        assert bm[:, g].all()          # attended by everything
        assert bm[g, :].all()          # attends to everything
    # a non-global row holds its window plus the globals only
    assert sorted(np.nonzero(bm[12])[0].tolist()) == [0, 7, 11, 12, 13]
    pc = oracle.Pattern(nb, window_left=1, window_right=1, causal=True, global_blocks=G,
                        global_rows_attend_all=True)
    bmc = brute.block_mask_from_csr(*pc.csr(), nb)
    assert not np.triu(bmc, 1).any()   # causal: no key block after the query block
    assert bmc[7, :8].all() and not bmc[7, 8:].any()
