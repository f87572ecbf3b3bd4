"""Pins for the oracle's backward (orc_attention_backward): gradients of
L = sum(dO * O) with respect to Q, K and V for the masked attention.

Training needs gradients through the sparse mask ("How Do Sparse Attention
Kernels Work in GPU Clusters?", FAQ on training versus inference).  Pinned
against:
* torch fp64 autograd through the dense masked form (a library routine);
* central finite differences of the independent numpy forward
  (oracle/brute.py) on tiny shapes;
* closed forms: V constant over the keys gives O independent of Q and K, so
  dQ = dK = 0; Q = 0 gives uniform weights, so dV_k = sum over the query rows
  that see key k of dO_q / (number of keys row q sees).
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import brute


def csr_random(nb, rng, causal, max_len):
    """Random block rows (each holds its diagonal, so no row is empty)."""
    rp, ci = [0], []
    for i in range(nb):
        cand = np.arange(0, i + 1) if causal else np.arange(nb)
        n = int(rng.integers(1, min(max_len, len(cand)) + 1))
        row = set(int(x) for x in rng.choice(cand, size=n, replace=False)) | {i}
        row = list(row)
        rng.shuffle(row)
        ci += row
        rp.append(len(ci))
    return np.array(rp, np.int32), np.array(ci, np.int32)


def dense_mask(rp, ci, nb, block, causal):
    return brute.expand_block_mask(brute.block_mask_from_csr(rp, ci, nb), block, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_autograd(causal):
    rng = np.random.default_rng(7 + causal)
    nb, block, D = 6, 8, 16
    N = nb * block
    rp, ci = csr_random(nb, rng, causal, 4)
    q, k, v, do = (rng.standard_normal((1, N, D)) for _ in range(4))
    scale = 0.3
    dq, dk, dv = oracle.attention_backward(q, k, v, do, rp, ci, block, scale, causal)
    allowed = torch.as_tensor(dense_mask(rp, ci, nb, block, causal))
    tq, tk, tv = (torch.tensor(a[0], dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    s = (tq @ tk.T) * scale
    s = s.masked_fill(~allowed, float("-inf"))
    o = torch.softmax(s, dim=1) @ tv
    (o * torch.tensor(do[0])).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_row_flags_match_torch_autograd():
    """Causal model whose flagged query blocks (bit 0) take no causal cut: the
    flagged rows list later key blocks too and see every key of them; the
    dense mask of brute.expand_block_mask with those rows exempt from the cut
    goes through torch autograd.  A flag on a row lifts only that row's cut,
    so a mistake in which row it applies to fails here."""
    rng = np.random.default_rng(31)
    nb, block, D = 6, 8, 16
    N = nb * block
    rp, ci = csr_random(nb, rng, True, 4)
    # rows 1 and 4 list every block (later ones included) and are flagged
    rows = [list(ci[rp[i]:rp[i + 1]]) for i in range(nb)]
    for i in (1, 4):
        rows[i] = list(range(nb))
    rp = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    ci = np.array([j for r in rows for j in r], np.int32)
    flags = np.zeros(nb, np.uint8)
    flags[[1, 4]] = 1
    q, k, v, do = (rng.standard_normal((1, N, D)) for _ in range(4))
    scale = 0.3
    dq, dk, dv = oracle.attention_backward(q, k, v, do, rp, ci, block, scale, True, row_flags=flags)
    allowed = torch.as_tensor(brute.expand_block_mask(brute.block_mask_from_csr(rp, ci, nb), block, True,
                                                      noncausal_rows=[1, 4]))
    tq, tk, tv = (torch.tensor(a[0], dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    s = ((tq @ tk.T) * scale).masked_fill(~allowed, float("-inf"))
    o = torch.softmax(s, dim=1) @ tv
    (o * torch.tensor(do[0])).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)
    # without the flags the same CSR gives the causal gradients (different)
    dq0, _, _ = oracle.attention_backward(q, k, v, do, rp, ci, block, scale, True)
    assert np.abs(dq0 - dq).max() > 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_central_differences(causal):
    rng = np.random.default_rng(11 + causal)
    nb, block, D = 4, 3, 3
    N = nb * block
    rp, ci = csr_random(nb, rng, causal, 3)
    allowed = dense_mask(rp, ci, nb, block, causal)
    q, k, v, do = (rng.standard_normal((1, N, D)) for _ in range(4))
    scale = 0.7

    def loss(qq, kk, vv):
        o, _ = brute.masked_attention(qq[0], kk[0], vv[0], allowed, scale)
        return float((o * do[0]).sum())

    dq, dk, dv = oracle.attention_backward(q, k, v, do, rp, ci, block, scale, causal)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(g)
        for t in range(N):
            for d in range(D):
                xp, xm = x.copy(), x.copy()
                xp[0, t, d] += h
                xm[0, t, d] -= h
                args_p = [q, k, v]
                args_m = [q, k, v]
                idx = "qkv".index(name)
                args_p[idx], args_m[idx] = xp, xm
                num[t, d] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8, err_msg=name)


def test_constant_v_and_zero_q_closed_forms():
    rng = np.random.default_rng(3)
    nb, block, D = 5, 4, 8
    N = nb * block
    rp, ci = csr_random(nb, rng, True, 3)
    q, k, do = (rng.standard_normal((1, N, D)) for _ in range(3))
    c = rng.standard_normal(D)
    v = np.broadcast_to(c, (1, N, D)).copy()
    dq, dk, dv = oracle.attention_backward(q, k, v, do, rp, ci, block, 0.5, True)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    # Q = 0: every allowed key of row q has weight 1 / n_q
    v = rng.standard_normal((1, N, D))
    _, _, dv = oracle.attention_backward(np.zeros_like(q), k, v, do, rp, ci, block, 0.5, True)
    allowed = dense_mask(rp, ci, nb, block, True)
    n_q = allowed.sum(1)
    want = (allowed / n_q[:, None]).T @ do[0]
    np.testing.assert_allclose(dv, want, rtol=1e-12, atol=1e-12)
