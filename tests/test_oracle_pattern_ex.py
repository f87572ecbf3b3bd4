"""Pins for the oracle's dilated-window / strided patterns
(orc_pattern_ex_allows, orc_pattern_ex_csr) and its per-head CSR assembly.

Pinned against: rows written out by hand (tests/golden/pattern_ex_masks.json,
from "Flash MSA Sparse Attention vs Full Attention", section "Sparse Patterns
Beyond Sliding Windows", items "Strided Patterns" and "Dilated Sliding
Window"); closed-form row lengths of a lone stride and a lone dilated window;
the plain pattern (already pinned to its own golden rows and to the token
window) as the special case of one window of dilation 1; and, at block size
1, the page's example of three windows covering every token, every 2nd and
every 4th, built here from explicit offset sets.
"""

import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pattern_ex_masks.json")))
CASES = [k for k in GOLDEN if not k.startswith("_")]


def rows_of(rp, ci):
    return [ci[rp[i]:rp[i + 1]].tolist() for i in range(len(rp) - 1)]


def from_spec(spec):
    return oracle.PatternEx(spec["n_blocks"], [tuple(w) for w in spec["windows"]], spec["stride"],
                            spec["causal"], spec["global_blocks"], spec["global_rows_attend_all"])


@pytest.mark.parametrize("name", CASES)
def test_golden_rows(name):
    g = GOLDEN[name]
    rp, ci = from_spec(g["pattern"]).csr()
    assert int(rp[-1]) == g["nnz"]
    assert rows_of(rp, ci) == g["rows"]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nb,s", [(17, 1), (17, 3), (30, 4), (9, 9), (9, 12)])
def test_lone_stride_row_lengths(nb, s, causal):
    rp, ci = oracle.PatternEx(nb, stride=s, causal=causal).csr()
    for i in range(nb):
        # blocks j = i (mod s) in [0, nb) (or [0, i] when causal)
        want = (i // s + 1) if causal else ((nb - 1 - (i % s)) // s + 1)
        assert rp[i + 1] - rp[i] == want, (i, s)
        row = ci[rp[i]:rp[i + 1]]
        assert np.all((row - i) % s == 0) and i in row


@pytest.mark.parametrize("l,r,d", [(0, 0, 1), (2, 3, 1), (3, 1, 2), (2, 2, 5), (4, 0, 3)])
def test_lone_dilated_window_row_lengths(l, r, d):
    nb = 29
    rp, ci = oracle.PatternEx(nb, windows=[(l, r, d)]).csr()
    for i in range(nb):
        want = min(l, i // d) + min(r, (nb - 1 - i) // d) + 1
        assert rp[i + 1] - rp[i] == want, (i, l, r, d)


def test_one_plain_window_is_the_plain_pattern():
    rng = np.random.default_rng(5)
    for _ in range(40):
        nb = int(rng.integers(1, 40))
        wl, wr = int(rng.integers(0, 6)), int(rng.integers(0, 6))
        causal = bool(rng.integers(0, 2))
        gra = bool(rng.integers(0, 2))
        globals_ = sorted(set(int(x) for x in rng.integers(0, nb, size=int(rng.integers(0, 4)))))
        a = oracle.Pattern(nb, wl, wr, causal, globals_, gra).csr()
        b = oracle.PatternEx(nb, [(wl, wr, 1)], 0, causal, globals_, gra).csr()
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


def test_page_example_three_dilations_at_block_size_one():
    # windows of every token, every 2nd, every 4th, each W steps back and ahead
    N, W = 50, 3
    offsets = set()
    for d in (1, 2, 4):
        offsets |= {d * t for t in range(-W, W + 1)}
    want = np.zeros((N, N), dtype=bool)
    for i in range(N):
        for o in offsets:
            if 0 <= i + o < N:
                want[i, i + o] = True
    rp, ci = oracle.PatternEx(N, [(W, W, 1), (W, W, 2), (W, W, 4)]).csr()
    got = np.zeros((N, N), dtype=bool)
    for i in range(N):
        got[i, ci[rp[i]:rp[i + 1]]] = True
    np.testing.assert_array_equal(got, want)


def test_heads_csr_layout():
    a = oracle.PatternEx(8, windows=[(1, 2, 3)])
    b = oracle.PatternEx(8, stride=2)
    rp, ci = oracle.heads_csr([a, b], B=2, H=3, head_pattern=[1, 1, 0])
    ra, ca = a.csr()
    rb, cb = b.csr()
    per_b = [(rb, cb), (rb, cb), (ra, ca)]
    for bi in range(2):
        for h in range(3):
            rpp, cpp = per_b[h]
            for i in range(8):
                r = (bi * 3 + h) * 8 + i
                assert ci[rp[r]:rp[r + 1]].tolist() == cpp[rpp[i]:rpp[i + 1]].tolist()
    assert int(rp[-1]) == 2 * (2 * len(cb) + len(ca))
