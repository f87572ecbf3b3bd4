"""Pins for the oracle's exact masked attention (orc_attention_rows).

Each test pins the C oracle to something other than itself:

* dense mask == torch's fp64 scaled_dot_product_attention and logsumexp
  (library routines; the Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V
  formula of "Flash MSA Sparse Attention vs Full Attention", "The Mechanics");
* any block mask == the literal full-row -inf-masked numpy form (the naive
  masked attention of "Sparse Attention Kernels vs Full Attention
  Performance", "How Sparse Attention Kernels Actually Speed Up Inference");
* closed forms: Q = 0 gives the plain mean of the allowed V rows and
  LSE = ln(#allowed keys), with the count taken from the hand-written golden
  rows; constant V gives that constant; causal row 0 gives V_0 and
  LSE = scale * q0.k0;
* invariants: with V = identity the output rows are the attention weights
  (non-negative, zero off the mask, summing to 1); outputs are convex
  combinations of the allowed V rows; permuting a CSR row changes nothing.
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


def bits(t):
    return bsa_inputs.bf16_bits(t)


def rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def dense_csr(BH, nb, causal):
    rows = [[j for j in range(nb) if (not causal or j <= i)] for i in range(nb)]
    rp = [0]
    ci = []
    for _ in range(BH):
        for r in rows:
            ci += r
            rp.append(len(ci))
    return np.array(rp, np.int32), np.array(ci, np.int32)


@pytest.mark.parametrize("causal", [False, True])
def test_dense_mask_equals_sdpa(causal):
    B, H, N, D, bs = 1, 2, 96, 32, 16
    q, k, v = (rand_bf16((B, H, N, D), s) for s in (1, 2, 3))
    rp, ci = dense_csr(B * H, N // bs, causal)
    scale = 1.0 / np.sqrt(D)
    O, L = oracle.attention_rows(bits(q), bits(k), bits(v), rp, ci, bs, scale, causal)
    qd, kd, vd = (t.to(torch.float64) for t in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, is_causal=causal, scale=scale)
    np.testing.assert_allclose(O.reshape(B, H, N, D), ref.numpy(), rtol=0, atol=1e-12)
    s = (qd @ kd.transpose(-1, -2)) * scale
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
    np.testing.assert_allclose(L.reshape(B, H, N), torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


PATTERNS = [
    dict(window_left=1, window_right=1, global_blocks=(0,), global_rows_attend_all=True, causal=False),
    dict(window_left=2, window_right=2, causal=True),
    dict(window_left=3, window_right=0, global_blocks=(0, 1), global_rows_attend_all=True, causal=True),
    dict(window_left=0, window_right=0, causal=False),
]


@pytest.mark.parametrize("pat", PATTERNS)
def test_matches_literal_full_row_form(pat):
    B, H, N, D, bs = 1, 3, 128, 16, 16
    nb = N // bs
    q, k, v = (rand_bf16((B, H, N, D), s, 2.0) for s in (11, 12, 13))
    p = oracle.Pattern(nb, **pat)
    rp1, ci1 = p.csr()
    rp, ci = oracle.replicate_csr(rp1, ci1, B * H)
    scale = 1.0 / np.sqrt(D)
    O, L = oracle.attention_rows(bits(q), bits(k), bits(v), rp, ci, bs, scale, pat["causal"])
    O = O.reshape(B * H, N, D)
    L = L.reshape(B * H, N)
    allowed = brute.expand_block_mask(brute.block_mask_from_csr(rp1, ci1, nb), bs, pat["causal"])
    for bh in range(B * H):
        qd = brute.bf16_to_f64(bits(q).reshape(B * H, N, D)[bh])
        kd = brute.bf16_to_f64(bits(k).reshape(B * H, N, D)[bh])
        vd = brute.bf16_to_f64(bits(v).reshape(B * H, N, D)[bh])
        o_ref, l_ref = brute.masked_attention(qd, kd, vd, allowed, scale)
        np.testing.assert_allclose(O[bh], o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(L[bh], l_ref, rtol=0, atol=1e-12)


def test_zero_q_gives_mean_of_allowed_rows_and_log_count():
    """Q = 0: every allowed key has logit 0, so O = mean of allowed V rows and
    LSE = ln(count).  Counts come from the hand-written golden rows."""
    w = bsa_inputs.workload("tiny_window_global")
    rows = GOLDEN["tiny_window_global"]["rows"]
    B, H, N, D, bs = w.B, w.H, w.N, w.D, w.block
    q = torch.zeros((B, H, N, D), dtype=torch.bfloat16)
    k = rand_bf16((B, H, N, D), 5)
    v = rand_bf16((B, H, N, D), 6)
    rp1, ci1 = oracle.Pattern.from_workload(w).csr()
    rp, ci = oracle.replicate_csr(rp1, ci1, B * H)
    O, L = oracle.attention_rows(bits(q), bits(k), bits(v), rp, ci, bs, w.scale, False)
    vd = v.to(torch.float64).reshape(B * H, N, D).numpy()
    O = O.reshape(B * H, N, D)
    L = L.reshape(B * H, N)
    for bh in range(B * H):
        for t in range(0, N, 37):
            keys = np.concatenate([np.arange(j * bs, (j + 1) * bs) for j in rows[t // bs]])
            np.testing.assert_allclose(O[bh, t], vd[bh, keys].mean(0), rtol=0, atol=1e-13)
            assert abs(L[bh, t] - np.log(len(keys))) < 1e-13


def test_constant_v_and_causal_row_zero():
    B, H, N, D, bs = 1, 2, 64, 16, 16
    q = rand_bf16((B, H, N, D), 21, 3.0)
    k = rand_bf16((B, H, N, D), 22, 3.0)
    c = torch.linspace(-2, 2, D).to(torch.bfloat16)
    v = c.expand(B, H, N, D).contiguous()
    p = oracle.Pattern(N // bs, window_left=1, window_right=0, causal=True)
    rp, ci = oracle.replicate_csr(*p.csr(), B * H)
    scale = 1.0 / np.sqrt(D)
    O, L = oracle.attention_rows(bits(q), bits(k), bits(v), rp, ci, bs, scale, True)
    np.testing.assert_allclose(O, np.broadcast_to(c.double().numpy(), O.shape), rtol=0, atol=1e-13)
    # causal row 0 of each head sees only key 0
    v2 = rand_bf16((B, H, N, D), 23)
    O2, L2 = oracle.attention_rows(bits(q), bits(k), bits(v2), rp, ci, bs, scale, True)
    O2 = O2.reshape(B * H, N, D)
    L2 = L2.reshape(B * H, N)
    qd, kd, vd = (t.double().reshape(B * H, N, D).numpy() for t in (q, k, v2))
    for bh in range(B * H):
        np.testing.assert_array_equal(O2[bh, 0], vd[bh, 0])
        assert abs(L2[bh, 0] - scale * float(qd[bh, 0] @ kd[bh, 0])) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_identity_v_gives_weights(causal):
    """With N == D and V = I, O[q, :] are the softmax weights of row q."""
    B, H, N, D, bs = 1, 1, 64, 64, 8
    nb = N // bs
    q = rand_bf16((B, H, N, D), 31, 2.0)
    k = rand_bf16((B, H, N, D), 32, 2.0)
    v = torch.eye(N, dtype=torch.bfloat16).reshape(B, H, N, D)
    p = oracle.Pattern(nb, window_left=2, window_right=1, causal=causal, global_blocks=(5,),
                       global_rows_attend_all=False)
    rp1, ci1 = p.csr()
    O, L = oracle.attention_rows(bits(q), bits(k), bits(v), rp1, ci1, bs, 1.0 / np.sqrt(D), causal)
    allowed = brute.expand_block_mask(brute.block_mask_from_csr(rp1, ci1, nb), bs, causal)
    assert np.all(O >= 0)
    assert np.all(O[~allowed] == 0)
    np.testing.assert_allclose(O.sum(1), 1.0, rtol=0, atol=1e-14)
    s = (q.double()[0, 0].numpy() @ k.double()[0, 0].numpy().T) / np.sqrt(D)
    w_ref = np.where(allowed, np.exp(s - L[:, None]), 0.0)
    np.testing.assert_allclose(O, w_ref, rtol=0, atol=1e-13)


def test_convex_combination_and_permutation_invariance():
    B, H, N, D, bs = 2, 2, 128, 32, 16
    nb = N // bs
    q, k, v = (rand_bf16((B, H, N, D), s, 1.5) for s in (41, 42, 43))
    p = oracle.Pattern(nb, window_left=2, window_right=2, causal=False, global_blocks=(3,),
                       global_rows_attend_all=True)
    rp1, ci1 = p.csr()
    rp, ci = oracle.replicate_csr(rp1, ci1, B * H)
    scale = 1.0 / np.sqrt(D)
    O, L = oracle.attention_rows(bits(q), bits(k), bits(v), rp, ci, bs, scale, False)
    vd = v.double().reshape(B * H, N, D).numpy()
    O3 = O.reshape(B * H, N, D)
    bm = brute.block_mask_from_csr(rp1, ci1, nb)
    for bh in range(B * H):
        for t in range(N):
            keys = np.concatenate([np.arange(j * bs, (j + 1) * bs) for j in np.nonzero(bm[t // bs])[0]])
            lo, hi = vd[bh, keys].min(0), vd[bh, keys].max(0)
            assert np.all(O3[bh, t] >= lo - 1e-12) and np.all(O3[bh, t] <= hi + 1e-12)
    rng = np.random.default_rng(0)
    ci_perm = ci.copy()
    for r in range(len(rp) - 1):
        seg = ci_perm[rp[r]:rp[r + 1]]
        ci_perm[rp[r]:rp[r + 1]] = rng.permutation(seg)
    assert not np.array_equal(ci_perm, ci)
    O2, L2 = oracle.attention_rows(bits(q), bits(k), bits(v), rp, ci_perm, bs, scale, False)
    np.testing.assert_array_equal(O2, O)
    np.testing.assert_array_equal(L2, L)


def test_empty_row_and_row_subset():
    B, H, N, D, bs = 1, 1, 64, 16, 16
    q, k, v = (rand_bf16((B, H, N, D), s) for s in (51, 52, 53))
    # row 1 empty, others dense
    rp = np.array([0, 4, 4, 8, 12], np.int32)
    ci = np.array([0, 1, 2, 3] * 3, np.int32)
    O, L = oracle.attention_rows(bits(q), bits(k), bits(v), rp, ci, bs, 0.25, False)
    assert np.all(O[16:32] == 0) and np.all(np.isneginf(L[16:32]))
    rows = np.array([3, 40, 63, 17], np.int64)
    Os, Ls = oracle.attention_rows(bits(q), bits(k), bits(v), rp, ci, bs, 0.25, False, rows=rows)
    np.testing.assert_array_equal(Os, O[rows])
    np.testing.assert_array_equal(Ls, L[rows])
