"""Pins for the oracle functions added for global query rows without the
causal cut, sharded key ranges, the merge of partial results and per-block
FP8 scales.  Each is checked against something other than itself:

* non-causal global rows (orc_pattern_allows with global_rows_noncausal):
  hand-written golden rows and flags (tests/golden/pattern_masks.json,
  "reading_b_small"), the closed-form count of the 128K workload with its
  sink row attending to everything, and the attention of such a row against
  torch's fp64 scaled_dot_product_attention over every key (a library
  routine) while the other rows match the literal -inf-masked form;
* attention_blocks_f64 (fp64 inputs, key range apart from the query range):
  equals the pinned C oracle on bf16-valued inputs (random unsorted CSRs,
  causal or not, with row flags), and a query shard with its offset equals
  the same rows of the unsharded problem;
* merge_partials: attention over a key set split into disjoint parts, each
  computed separately and merged, equals attention over the whole set
  (the identity log sum exp of a union of disjoint sets);
* quantize_e4m3_blocks: the largest magnitude of every block lands exactly on
  +-448, all-zero blocks give zero codes, and every block's codes equal the
  per-tensor codec (pinned in test_oracle_fp8.py) at that block's scale.
"""

import json
import os

import numpy as np
import pytest
import torch

import bsa_inputs
import oracle
from oracle import brute

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pattern_masks.json")))


def rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def bits(t):
    return bsa_inputs.bf16_bits(t)


def f64(t):
    return t.double().numpy()


# ------------------------------------------------------------------ non-causal global rows
def test_reading_b_golden_rows_and_flags():
    g = GOLDEN["reading_b_small"]
    p = oracle.Pattern(**g["pattern"])
    rp, ci = p.csr()
    assert int(rp[-1]) == g["nnz_per_head"]
    assert [ci[rp[i]:rp[i + 1]].tolist() for i in range(len(rp) - 1)] == g["rows"]
    assert p.row_flags().tolist() == g["row_flags"]


def test_long_window_128k_global_row_closed_form():
    g = GOLDEN["long_window_128k_global_row"]
    w = bsa_inputs.workload("long_window_128k").with_(global_rows_noncausal=True)
    rp, ci = oracle.Pattern.from_workload(w).csr()
    lens = np.diff(rp)
    assert int(rp[-1]) == g["nnz_per_head"]
    assert int(lens.min()) == g["row_len_min"] and int(lens.max()) == g["row_len_max"]
    assert ci[:1024].tolist() == list(range(1024))       # the sink row sees every block
    rpa, cia = oracle.Pattern.from_workload(bsa_inputs.workload("long_window_128k")).csr()
    np.testing.assert_array_equal(np.diff(rp)[1:], np.diff(rpa)[1:])   # other rows unchanged
    np.testing.assert_array_equal(ci[1024:], cia[1:])


def test_noncausal_global_row_attention():
    nb, bs, D = 10, 8, 32
    N = nb * bs
    p = oracle.Pattern(nb, window_left=2, window_right=0, causal=True, global_blocks=(0, 4),
                       global_rows_attend_all=True, global_rows_noncausal=True)
    rp, ci = p.csr()
    flags = p.row_flags()
    q, k, v = (rand_bf16((1, 1, N, D), s) for s in (11, 12, 13))
    scale = 1.0 / np.sqrt(D)
    O, L = oracle.attention_rows(bits(q), bits(k), bits(v), rp, ci, bs, scale, True, row_flags=flags)
    # flagged rows: plain attention over every key (library routine)
    qd, kd, vd = (x.double() for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, scale=scale, is_causal=False)[0, 0]
    lse_ref = torch.logsumexp((qd[0, 0] @ kd[0, 0].T) * scale, dim=-1)
    for i in (0, 4):
        sl = slice(i * bs, (i + 1) * bs)
        np.testing.assert_allclose(O[sl], ref[sl].numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(L[sl], lse_ref[sl].numpy(), rtol=0, atol=1e-12)
    # every row: the literal -inf form with the causal cut lifted on flagged rows
    bm = brute.block_mask_from_csr(rp, ci, nb)
    allowed = brute.expand_block_mask(bm, bs, True, noncausal_rows=[0, 4])
    Ob, Lb = brute.masked_attention(f64(q[0, 0]), f64(k[0, 0]), f64(v[0, 0]), allowed, scale)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lb, rtol=0, atol=1e-12)
    # without the flags the same CSR is cut causally: row 0 then sees block 0's past only
    O0, L0 = oracle.attention_rows(bits(q), bits(k), bits(v), rp, ci, bs, scale, True)
    assert np.abs(O0[:bs] - O[:bs]).max() > 1e-3


# ------------------------------------------------------------------ fp64 inputs, general geometry
def random_csr(BH, nbq, nbk, rng, max_len):
    rp, ci = [0], []
    for _ in range(BH * nbq):
        n = int(rng.integers(0, max_len + 1))
        ci += [int(x) for x in rng.choice(nbk, size=min(n, nbk), replace=False)]
        rp.append(len(ci))
    return np.array(rp, np.int32), np.array(ci, np.int32)


@pytest.mark.parametrize("causal", [False, True])
def test_blocks_f64_equals_c_oracle(causal):
    rng = np.random.default_rng(5 + causal)
    BH, nb, bs, D = 3, 9, 16, 32
    N = nb * bs
    q, k, v = (rand_bf16((BH, N, D), s) for s in (21, 22, 23))
    rp, ci = random_csr(BH, nb, nb, rng, 6)
    flags = (rng.random(BH * nb) < 0.3).astype(np.uint8)
    scale = 0.17
    Oc, Lc = oracle.attention_rows(bits(q), bits(k), bits(v), rp, ci, bs, scale, causal, row_flags=flags)
    O, L = oracle.attention_blocks_f64(f64(q), f64(k), f64(v), rp, ci, bs, scale, causal, row_flags=flags)
    np.testing.assert_allclose(O, Oc, rtol=0, atol=1e-12)
    both = np.isneginf(L) & np.isneginf(Lc)
    np.testing.assert_allclose(np.where(both, 0, L), np.where(both, 0, Lc), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_query_shard_with_offset_equals_unsharded_rows(causal):
    rng = np.random.default_rng(40 + causal)
    BH, nb, bs, D = 2, 12, 8, 16
    N = nb * bs
    q, k, v = (rand_bf16((BH, N, D), s) for s in (31, 32, 33))
    rp, ci = random_csr(BH, nb, nb, rng, 7)
    scale = 0.3
    O, L = oracle.attention_blocks_f64(f64(q), f64(k), f64(v), rp, ci, bs, scale, causal)
    s0, s1 = 5, 9                                      # the shard's query blocks
    q_sh = f64(q)[:, s0 * bs:s1 * bs]
    rows_sh = []
    for bh in range(BH):
        for i in range(s0, s1):
            r = bh * nb + i
            rows_sh.append(ci[rp[r]:rp[r + 1]])
    rp_sh = np.concatenate([[0], np.cumsum([len(x) for x in rows_sh])]).astype(np.int32)
    ci_sh = np.concatenate(rows_sh).astype(np.int32)
    Os, Ls = oracle.attention_blocks_f64(q_sh, f64(k), f64(v), rp_sh, ci_sh, bs, scale, causal,
                                         q_block_offset=s0)
    want = np.concatenate([np.arange(bh * N + s0 * bs, bh * N + s1 * bs) for bh in range(BH)])
    np.testing.assert_allclose(Os, O[want], rtol=0, atol=1e-12)
    both = np.isneginf(Ls) & np.isneginf(L[want])
    np.testing.assert_allclose(np.where(both, 0, Ls), np.where(both, 0, L[want]), rtol=0, atol=1e-12)


# ------------------------------------------------------------------ merge
@pytest.mark.parametrize("n_parts", [1, 2, 3])
def test_merge_of_disjoint_parts_equals_whole(n_parts):
    rng = np.random.default_rng(70 + n_parts)
    BH, nb, bs, D = 2, 10, 8, 16
    N = nb * bs
    q, k, v = (rand_bf16((BH, N, D), s) for s in (41, 42, 43))
    rp, ci = random_csr(BH, nb, nb, rng, 8)
    scale = 0.25
    for causal in (False, True):
        O, L = oracle.attention_rows(bits(q), bits(k), bits(v), rp, ci, bs, scale, causal)
        # split every row's entries at random into n_parts disjoint parts
        parts = [([0], []) for _ in range(n_parts)]
        for r in range(len(rp) - 1):
            lab = rng.integers(0, n_parts, size=rp[r + 1] - rp[r])
            for p_ in range(n_parts):
                parts[p_][1].extend(int(x) for x in ci[rp[r]:rp[r + 1]][lab == p_])
                parts[p_][0].append(len(parts[p_][1]))
        outs, lses = [], []
        for prp, pci in parts:
            Op, Lp = oracle.attention_rows(bits(q), bits(k), bits(v), np.array(prp, np.int32),
                                           np.array(pci, np.int32), bs, scale, causal)
            outs.append(Op)
            lses.append(Lp)
        Om, Lm = oracle.merge_partials(outs, lses)
        np.testing.assert_allclose(Om, O, rtol=0, atol=1e-12)
        both = np.isneginf(Lm) & np.isneginf(L)
        assert np.array_equal(np.isneginf(Lm), np.isneginf(L))
        np.testing.assert_allclose(np.where(both, 0, Lm), np.where(both, 0, L), rtol=0, atol=1e-12)


def test_merge_empty_parts():
    O = np.ones((3, 4))
    L = np.array([-np.inf, 0.5, -np.inf])
    Om, Lm = oracle.merge_partials([O, 2 * O], [L, np.full(3, -np.inf)])
    assert np.isneginf(Lm[0]) and np.isneginf(Lm[2]) and Lm[1] == 0.5
    assert np.all(Om[0] == 0) and np.all(Om[2] == 0) and np.all(Om[1] == 1)


# ------------------------------------------------------------------ per-block e4m3
def test_block_quantization_pins():
    BH, nb, bs, D = 2, 6, 16, 32
    x = rand_bf16((BH, nb * bs, D), 51, scale=3.0)
    x[0, 2 * bs:3 * bs] = 0                          # an all-zero block
    x[1, 4 * bs:5 * bs] *= 1000                      # a peaked block
    xb = bits(x)
    codes, desc = oracle.quantize_e4m3_blocks(xb, bs)
    xf = x.float().numpy().reshape(BH, nb, bs, D)
    for bh in range(BH):
        for b in range(nb):
            cb = codes[bh, b * bs:(b + 1) * bs]
            amax = np.float32(np.abs(xf[bh, b]).max())
            if amax == 0:
                assert not cb.any() and desc[bh, b] == 1.0
                continue
            # the block's largest magnitude lands on +-448 exactly
            vals = oracle.e4m3_decode(cb)
            assert np.abs(vals).max() == 448.0
            # the per-tensor codec at this block's scale gives the same codes
            inv = np.float32(448.0) / amax
            np.testing.assert_array_equal(cb, oracle.quantize_e4m3(xb[bh, b * bs:(b + 1) * bs], float(inv)))
            assert desc[bh, b] == np.float32(amax / np.float32(448.0))
