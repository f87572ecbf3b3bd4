"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded bf16 inputs.

* pattern CSRs and top-k selections: bit-exact, at full size;
* forward: every row at sizes the oracle finishes in seconds (several tiles,
  every pattern recipe, all four (block, head-dim) instances), and sampled
  rows (every head; query blocks 0, 1, 2, nb-1 and seeded random ones) at the
  full sizes the benchmark runs;
* closed forms and edge cases on the GPU: Q = 0 (uniform weights, so a
  dropped or extra key shows up in O and in LSE = ln(count)), permuted and
  unsorted CSR rows, empty rows, causal lists holding future blocks,
  out-of-range entries (skipped and flagged), dense masks.
"""

import numpy as np
import pytest
import torch

import bsa_inputs
import oracle
from parity import (TOL_LSE, assert_close, bits, compare, ex_pair, gpu_csr, oracle_csr, random_ex_specs,
                    run_forward_case)

pytestmark = pytest.mark.gpu

W = {w.name: w for w in bsa_inputs.WORKLOADS}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_flashattention_bsa_gb300 import build
    build.build()
    import block_sparse_flashattention_bsa_gb300 as bsa
    bsa.device_error()  # clear


# ------------------------------------------------------------------ CSR
@pytest.mark.parametrize("name", ["tiny_window_global", "window_16k", "window_global_64k", "long_window_128k"])
def test_mask_csr_bit_exact_full_size(name):
    import block_sparse_flashattention_bsa_gb300 as bsa
    w = W[name]
    rp_ref, ci_ref = oracle_csr(w)
    dev = torch.device("cuda")
    rp, ci = gpu_csr(w, torch.empty(1, device=dev), None)
    np.testing.assert_array_equal(rp.cpu().numpy(), rp_ref)
    np.testing.assert_array_equal(ci.cpu().numpy(), ci_ref)
    assert bsa.validate_csr((w.B, w.H, w.N, w.D), w.block, rp, ci) == 0


@pytest.mark.parametrize("kw", [dict(B=1, H=2, N=64 * 96), dict(B=2, H=16, N=32768)], ids=["small", "full"])
def test_topk_bit_exact(kw):
    w = bsa_inputs.small_workload(W["content_topk"], **kw)
    d = bsa_inputs.make_qkv(w)
    rp_ref, ci_ref = oracle_csr(w, d["q"], d["k"])
    rp, ci = gpu_csr(w, d["q"].cuda(), d["k"].cuda())
    np.testing.assert_array_equal(rp.cpu().numpy(), rp_ref)
    np.testing.assert_array_equal(ci.cpu().numpy(), ci_ref)


@pytest.mark.parametrize("topk,diag,block,D", [(4, True, 32, 64), (1, False, 128, 128), (32, True, 16, 128)])
def test_topk_other_shapes(topk, diag, block, D):
    w = bsa_inputs.Workload("t", 1, 3, block * 40, D, block, topk=topk, include_diag=diag, n_centroids=8,
                            centroid_gain=1.0, seed=77)
    d = bsa_inputs.make_qkv(w)
    rp_ref, ci_ref = oracle_csr(w, d["q"], d["k"])
    rp, ci = gpu_csr(w, d["q"].cuda(), d["k"].cuda())
    np.testing.assert_array_equal(rp.cpu().numpy(), rp_ref)
    np.testing.assert_array_equal(ci.cpu().numpy(), ci_ref)


def _topk_shape(case):
    """(q, k, block, topk, include_diag) for the selection edge cases."""
    g = torch.Generator().manual_seed(4242)
    if case == "zero_q":
        # every score is +-0: all tie, so the smallest block indices win
        B, H, N, D, block, topk, diag = 1, 2, 64 * 100, 128, 64, 16, True
        k = torch.randn(B, H, N, D, generator=g).to(torch.bfloat16)
        return torch.zeros_like(k), k, block, topk, diag
    if case == "block_signs":
        # each block's tokens repeat one +-1 vector: pooled vectors are +-1
        # exactly and the scores are even integers with many ties
        B, H, nb, D, block, topk, diag = 1, 2, 300, 64, 16, 12, True

        def signs():
            x = torch.randint(0, 2, (B, H, nb, 1, D), generator=g) * 2 - 1
            return x.expand(B, H, nb, block, D).reshape(B, H, nb * block, D).to(torch.bfloat16)

        q = signs()
        return q, signs(), block, topk, diag
    if case == "nb2000":
        # more than 1024 key blocks
        B, H, N, D, block, topk, diag = 1, 1, 16 * 2000, 64, 16, 8, False
    elif case == "many_heads":
        # 1024 key blocks in 72 heads: 288 MB of scores, over the split path's
        # budget, so the fused kernel runs at this size too
        B, H, N, D, block, topk, diag = 1, 72, 16 * 1024, 64, 16, 8, True
    else:
        # fewer than 32 key blocks, every block chosen
        B, H, N, D, block, topk, diag = 1, 2, 64 * 20, 64, 64, 20, True
    q = torch.randn(B, H, N, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, H, N, D, generator=g).to(torch.bfloat16)
    return q, k, block, topk, diag


@pytest.mark.parametrize("case", ["zero_q", "block_signs", "nb2000", "many_heads", "nb20_all"])
def test_topk_ties_and_sizes(case):
    import block_sparse_flashattention_bsa_gb300 as bsa
    q, k, block, topk, diag = _topk_shape(case)
    rp_ref, ci_ref, _ = oracle.topk_csr(bits(q), bits(k), block, topk, diag)
    rp, ci = bsa.topk_blocks(q.cuda(), k.cuda(), block, topk, diag)
    np.testing.assert_array_equal(rp.cpu().numpy(), rp_ref)
    np.testing.assert_array_equal(ci[: int(rp[-1].item())].cpu().numpy(), ci_ref)
    if case == "zero_q":
        first = ci_ref[: rp_ref[1]]
        assert list(first) == list(range(topk)), first


# ------------------------------------------------------------------ per-head patterns
def _spec(nb, windows=(), stride=0, causal=False, globals_=(), gra=False):
    return dict(n_blocks=nb, windows=[list(w) for w in windows], stride=stride, causal=causal,
                global_blocks=list(globals_), global_rows_attend_all=gra)


HEAD_SETS = {
    # four head types of a causal long-context model, 16 heads, 512 blocks
    "causal_mixed": (2, 16, None, [
        _spec(512, [(8, 0, 1), (8, 0, 2), (8, 0, 4), (8, 0, 8)], causal=True),
        _spec(512, [(4, 0, 1)], stride=16, causal=True),
        _spec(512, [(16, 0, 1)], causal=True, globals_=(0, 1), gra=True),
        _spec(512, [(63, 0, 1)], causal=True)]),
    # non-causal heads with an explicit head map
    "bidirectional_map": (1, 6, [2, 0, 1, 1, 0, 2], [
        _spec(256, [(2, 2, 1), (2, 2, 3)]),
        _spec(256, [(1, 1, 1)], stride=5),
        _spec(256, [(0, 0, 1)], globals_=(0, 100, 255), gra=True)]),
}


def _heads_csrs(B, H, hp, specs):
    import block_sparse_flashattention_bsa_gb300 as bsa
    pairs = [ex_pair(s) for s in specs]
    rp_ref, ci_ref = oracle.heads_csr([o for _, o in pairs], B, H, hp)
    rp, ci = bsa.build_mask_csr_heads([p for p, _ in pairs], B, H, hp)
    return (rp, ci), (rp_ref, ci_ref)


@pytest.mark.parametrize("name", list(HEAD_SETS))
def test_mask_heads_bit_exact(name):
    import block_sparse_flashattention_bsa_gb300 as bsa
    B, H, hp, specs = HEAD_SETS[name]
    (rp, ci), (rp_ref, ci_ref) = _heads_csrs(B, H, hp, specs)
    np.testing.assert_array_equal(rp.cpu().numpy(), rp_ref)
    np.testing.assert_array_equal(ci.cpu().numpy(), ci_ref)
    nb = specs[0]["n_blocks"]
    assert bsa.validate_csr((B, H, nb * 64, 64), 64, rp, ci) == 0


def test_mask_heads_random_sets():
    rng = np.random.default_rng(2027)
    for trial in range(25):
        nb = int(rng.integers(1, 200))
        specs = random_ex_specs(rng, nb, int(rng.integers(1, 9)))
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 20))
        hp = [int(x) for x in rng.integers(0, len(specs), size=H)] if trial % 2 else None
        (rp, ci), (rp_ref, ci_ref) = _heads_csrs(B, H, hp, specs)
        np.testing.assert_array_equal(rp.cpu().numpy(), rp_ref, err_msg=str((trial, specs)))
        np.testing.assert_array_equal(ci.cpu().numpy(), ci_ref, err_msg=str((trial, specs)))


@pytest.mark.parametrize("block,D,causal", [(128, 128, True), (64, 64, False)])
def test_forward_on_per_head_masks(block, D, causal):
    nb = 40
    specs = [_spec(nb, [(3, 0 if causal else 3, 1), (3, 0 if causal else 3, 4)], causal=causal),
             _spec(nb, [(1, 0 if causal else 1, 1)], stride=6, causal=causal),
             _spec(nb, [(2, 0 if causal else 2, 1)], causal=causal, globals_=(0, 17), gra=True)]
    w = bsa_inputs.Workload("heads", 1, 4, block * nb, D, block, causal=causal, seed=31)
    (rp, ci), (rp_ref, ci_ref) = _heads_csrs(w.B, w.H, [0, 1, 2, 1], specs)
    np.testing.assert_array_equal(rp.cpu().numpy(), rp_ref)
    np.testing.assert_array_equal(ci.cpu().numpy(), ci_ref)
    stats, err = run_forward_case(w, csr=(rp_ref, ci_ref), causal=causal)
    assert err == 0
    assert_close(stats, "per-head masks")


# ------------------------------------------------------------------ forward, all rows
SMALL = [
    ("tiny_window_global", {}),
    ("window_16k", dict(H=2, N=128 * 24)),
    ("window_global_64k", dict(H=2, N=128 * 80)),
    ("long_window_128k", dict(H=2, N=128 * 48)),
    ("content_topk", dict(B=1, H=2, N=64 * 40)),
]


@pytest.mark.parametrize("name,kw", SMALL, ids=[s[0] for s in SMALL])
def test_forward_all_rows_small(name, kw):
    w = bsa_inputs.small_workload(W[name], **kw)
    stats, err = run_forward_case(w)
    assert err == 0
    assert_close(stats, name)


@pytest.mark.parametrize("block,D,causal", [(128, 64, True), (128, 64, False), (64, 128, True), (64, 64, True),
                                            (128, 128, False)])
def test_forward_instances(block, D, causal):
    w = bsa_inputs.Workload("inst", 2, 3, block * 20, D, block, window_left=3, window_right=2, causal=causal,
                            global_blocks=(0, 7), global_rows_attend_all=True, seed=5)
    stats, err = run_forward_case(w)
    assert err == 0
    assert_close(stats, "instance %d/%d" % (block, D))


# ------------------------------------------------------------------ forward, full size, sampled rows
@pytest.mark.parametrize("name,nrand", [("window_16k", 12), ("window_global_64k", 6), ("long_window_128k", 4),
                                        ("content_topk", 8)])
def test_forward_full_size_sampled(name, nrand):
    w = W[name]
    rows = bsa_inputs.sample_rows(w, n_random_blocks=nrand).numpy()
    stats, err = run_forward_case(w, rows=rows)
    assert err == 0
    assert_close(stats, name)


# ------------------------------------------------------------------ closed forms, edge cases
def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def test_zero_q_reveals_key_counts():
    """Q = 0: O = mean of the allowed V rows and LSE = ln(#allowed keys)."""
    import block_sparse_flashattention_bsa_gb300 as bsa
    for name, kw in SMALL[:4]:
        w = bsa_inputs.small_workload(W[name], **kw)
        d = bsa_inputs.make_qkv(w)
        d["q"] = torch.zeros_like(d["q"])
        stats, err = run_forward_case(w, data=d)
        assert err == 0
        assert_close(stats, name)
        # LSE must be exactly ln(count) up to fp32 rounding
        rp, ci = oracle_csr(w)
        rows = np.arange(w.B * w.H * w.N)
        _, L_ref, cnt = oracle.attention_rows(bits(d["q"]), bits(d["k"]), bits(d["v"]), rp, ci, w.block,
                                              w.scale, w.causal, rows=rows, return_counts=True)
        np.testing.assert_allclose(L_ref, np.log(cnt), rtol=0, atol=1e-12)


def _random_csr(BH, nb, rng, max_len, allow_empty=True, causal=False):
    rp = [0]
    ci = []
    for r in range(BH * nb):
        i = r % nb
        n = int(rng.integers(0 if allow_empty else 1, max_len + 1))
        row = rng.choice(nb, size=min(n, nb), replace=False)
        if not causal and not allow_empty and i not in row:
            row[0] = i
        ci += [int(x) for x in row]  # random order
        rp.append(len(ci))
    return np.array(rp, np.int32), np.array(ci, np.int32)


@pytest.mark.parametrize("block,D,causal", [(128, 128, False), (128, 128, True), (64, 128, False), (64, 64, True)])
def test_random_unsorted_rows_with_empty_rows(block, D, causal):
    rng = np.random.default_rng(block + D + causal)
    w = bsa_inputs.Workload("rand", 1, 3, block * 12, D, block, causal=causal, seed=9)
    rp, ci = _random_csr(w.B * w.H, w.n_blocks, rng, 7, allow_empty=True, causal=causal)
    stats, err = run_forward_case(w, csr=(rp, ci), causal=causal)
    assert err == 0
    assert_close(stats, "random csr")


@pytest.mark.parametrize("D,causal", [(128, True), (64, False), (128, False)])
def test_block64_pairs_singles_and_empty_rows(D, causal):
    """64-token blocks run two query blocks per tile: rows of at most 32
    entries are paired by key-set similarity, longer rows run alone; odd
    counts, empty rows, unsorted rows and (causal) future blocks included."""
    rng = np.random.default_rng(640 + D + causal)
    w = bsa_inputs.Workload("pairs", 1, 3, 64 * 45, D, 64, causal=causal, seed=12)
    rp, ci = _random_csr(w.B * w.H, w.n_blocks, rng, 45, allow_empty=True, causal=causal)
    stats, err = run_forward_case(w, csr=(rp, ci), causal=causal)
    assert err == 0
    assert_close(stats, "block-64 pairs")


def test_block64_identical_rows():
    """Every row of a head lists the same blocks: every pair's union is one list."""
    w = bsa_inputs.Workload("same", 1, 2, 64 * 24, 128, 64, seed=13)
    nb = w.n_blocks
    row = np.array([0, 3, 7, 11, 12, 20, 23], np.int32)
    rp = np.arange(0, (w.B * w.H * nb + 1) * len(row), len(row), dtype=np.int32)
    ci = np.tile(row, w.B * w.H * nb)
    stats, err = run_forward_case(w, csr=(rp, ci), causal=False)
    assert err == 0
    assert_close(stats, "identical rows")


def test_row_permutation_invariance():
    import block_sparse_flashattention_bsa_gb300 as bsa
    w = bsa_inputs.small_workload(W["window_global_64k"], H=2, N=128 * 72)
    rp, ci = oracle_csr(w)
    rng = np.random.default_rng(1)
    ci_p = ci.copy()
    for r in range(len(rp) - 1):
        ci_p[rp[r]:rp[r + 1]] = rng.permutation(ci_p[rp[r]:rp[r + 1]])
    d = bsa_inputs.make_qkv(w)
    s1, e1 = run_forward_case(w, data=d, csr=(rp, ci))
    s2, e2 = run_forward_case(w, data=d, csr=(rp, ci_p))
    assert e1 == 0 and e2 == 0
    assert_close(s1, "sorted")
    assert_close(s2, "permuted")


def test_out_of_range_entries_are_skipped_and_flagged():
    w = bsa_inputs.Workload("oob", 1, 2, 128 * 6, 128, 128, seed=3)
    nb = w.n_blocks
    rp_good, ci_good = oracle.replicate_csr(*oracle.Pattern(nb, 1, 1).csr(), w.B * w.H)
    # insert an out-of-range block id at the front of every row
    rp_bad, ci_bad = [0], []
    for r in range(len(rp_good) - 1):
        ci_bad += [nb + 3] + ci_good[rp_good[r]:rp_good[r + 1]].tolist()
        rp_bad.append(len(ci_bad))
    import block_sparse_flashattention_bsa_gb300 as bsa
    d = bsa_inputs.make_qkv(w)
    dev = torch.device("cuda")
    q, k, v = (d[x].to(dev) for x in "qkv")
    rp_t = torch.tensor(rp_bad, dtype=torch.int32, device=dev)
    ci_t = torch.tensor(ci_bad, dtype=torch.int32, device=dev)
    assert bsa.validate_csr(q.shape, w.block, rp_t, ci_t) & 2
    o, lse = bsa.forward(q, k, v, rp_t, ci_t, w.block, scale=w.scale, causal=False)
    assert bsa.device_error() & 2
    rows = np.arange(w.B * w.H * w.N)
    O_ref, L_ref = oracle.attention_rows(bits(d["q"]), bits(d["k"]), bits(d["v"]), rp_good, ci_good, w.block,
                                         w.scale, False, rows=rows)
    assert_close(compare(o, lse, O_ref, L_ref, rows, w.D), "oob")
    assert bsa.device_error() == 0


def test_dense_masks():
    for causal in (False, True):
        w = bsa_inputs.Workload("dense", 1, 2, 128 * 16, 128, 128, causal=causal, window_left=10 ** 6,
                                window_right=10 ** 6, seed=11)
        stats, err = run_forward_case(w)
        assert err == 0
        assert_close(stats, "dense causal=%s" % causal)


def test_constant_v_and_causal_first_row_exact():
    import block_sparse_flashattention_bsa_gb300 as bsa
    w = bsa_inputs.small_workload(W["window_16k"], H=2, N=128 * 8)
    d = bsa_inputs.make_qkv(w)
    c = torch.linspace(-3, 3, w.D).to(torch.bfloat16)
    d["v"] = c.expand_as(d["v"]).contiguous()
    stats, err = run_forward_case(w, data=d)
    assert err == 0 and stats[0] <= 1e-2
    # causal query row 0 of every head sees key 0 only: O = V_0 exactly
    d2 = bsa_inputs.make_qkv(w)
    dev = torch.device("cuda")
    q, k, v = (d2[x].to(dev) for x in "qkv")
    rp, ci = bsa.build_mask_csr(
        bsa.Pattern(w.n_blocks, w.window_left, w.window_right, True), w.B, w.H, device=dev)
    o, lse = bsa.forward(q, k, v, rp, ci, w.block, scale=w.scale, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o[:, :, 0, :], v[:, :, 0, :])
    l0 = (q[:, :, 0, :].double() * k[:, :, 0, :].double()).sum(-1) * w.scale
    assert float((lse[:, :, 0].double() - l0).abs().max()) <= TOL_LSE
