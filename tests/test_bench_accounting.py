"""The benchmark's FLOP accounting (its metric: TFLOP/s on active block pairs,
4 * Bq * Bk * D FLOPs per active (query block, key block) pair per head).

The active-pair count of each workload's CSR (built by the oracle) is checked
against closed forms of the pattern, and the counting rule itself against
hand-made CSRs: entries out of range and, when causal, key blocks after the
query block are not computed and not counted.
"""

import os
import sys

import numpy as np
import pytest

import bsa_inputs
import oracle

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

W = {w.name: w for w in bsa_inputs.WORKLOADS}


def _csr(w):
    rp1, ci1 = oracle.Pattern.from_workload(w).csr()
    return oracle.replicate_csr(rp1, ci1, w.B * w.H)


def test_pair_flops():
    assert bench.pair_flops(W["window_16k"]) == 4 * 128 * 128 * 128
    assert bench.pair_flops(W["tiny_window_global"]) == 4 * 64 * 64 * 64


def test_window_16k_pairs_closed_form():
    # causal window i-4..i: rows 0..3 hold 1..4 blocks, the other 124 hold 5
    w = W["window_16k"]
    rp, ci = _csr(w)
    assert bench.active_pairs(rp, ci, w.n_blocks, w.causal) == w.B * w.H * (1 + 2 + 3 + 4 + 124 * 5)


def test_window_global_64k_pairs_closed_form():
    # causal window i-63..i plus global key blocks 0 and 1 (global rows 0, 1
    # attend every block up to themselves): row i holds min(i, 63) + 1 window
    # blocks, plus the globals below i - 63
    w = W["window_global_64k"]
    nb = w.n_blocks
    per_head = sum(min(i, 63) + 1 + sum(1 for g in (0, 1) if g < i - 63) for i in range(nb))
    rp, ci = _csr(w)
    assert bench.active_pairs(rp, ci, nb, w.causal) == w.B * w.H * per_head


def test_dense_pairs_closed_form():
    w = W["window_16k"]
    rp, ci = bench.dense_csr(w)
    nb = w.n_blocks
    assert bench.active_pairs(rp, ci, nb, True) == w.B * w.H * nb * (nb + 1) // 2
    lens = np.diff(rp)
    assert np.array_equal(lens[:nb], np.arange(1, nb + 1))


@pytest.mark.parametrize("causal", [False, True])
def test_counting_rule_on_hand_made_csr(causal):
    nb = 4
    # two heads; rows list in-range, out-of-range and future blocks
    rows = [[0], [0, 1, 3], [5, 2, -1], [], [3, 2, 1, 0], [1], [2, 0], [0, 4]]
    rp = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    ci = np.array([j for r in rows for j in r], dtype=np.int32)
    want = 0
    for r, lst in enumerate(rows):
        i = r % nb
        want += sum(1 for j in lst if 0 <= j < nb and (not causal or j <= i))
    assert bench.active_pairs(rp, ci, nb, causal) == want
