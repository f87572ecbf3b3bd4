"""GPU parity of the backward (bsa_backward through the C ABI) against the
fp64 oracle (orc_attention_backward) on the same seeded bf16 inputs.

The forward runs first on the GPU; its O and LSE feed the backward.  The
oracle rebuilds P exactly from Q and K, so the comparison covers the whole
chain.  Tolerance, per gradient tensor, relative to its largest reference
magnitude G: max |d| <= 2e-2 G and mean |d| <= 2e-3 G.  Derivation: P and dS
enter the tensor-core products rounded to bf16 (relative 2^-9 each), Dv uses
the forward's bf16 O (2^-9), and the outputs are rounded to bf16 (2^-9); fp32
accumulation adds ~2^-24 per term.  With independent roundings the error of
an entry is a few 2^-9 of the typical term; 2e-2 G leaves room for the
largest entries, and 2e-3 G bounds the average.
"""

import numpy as np
import pytest
import torch

import bsa_inputs
import oracle

pytestmark = pytest.mark.gpu

TOL_MAX = 2e-2
TOL_MEAN = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_flashattention_bsa_gb300 import build
    build.build()
    import block_sparse_flashattention_bsa_gb300 as bsa
    bsa.device_error()


def window_csr(BH, nb, wl, causal):
    rp, ci = [0], []
    for r in range(BH * nb):
        i = r % nb
        ci += [j for j in range(max(0, i - wl), min(nb, i + (0 if causal else wl) + 1))]
        rp.append(len(ci))
    return np.array(rp, np.int32), np.array(ci, np.int32)


def random_csr(BH, nb, rng, max_len):
    """Unsorted rows, some empty, some listing future blocks (skipped when causal)."""
    rp, ci = [0], []
    for _ in range(BH * nb):
        n = int(rng.integers(0, max_len + 1))
        ci += [int(x) for x in rng.choice(nb, size=min(n, nb), replace=False)]
        rp.append(len(ci))
    return np.array(rp, np.int32), np.array(ci, np.int32)


def run_backward(w, rp, ci, causal, qrows=None, krows=None):
    import block_sparse_flashattention_bsa_gb300 as bsa
    d = bsa_inputs.make_qkv(w)
    dout = bsa_inputs.make_grad_out(w)
    dev = torch.device("cuda")
    q, k, v, do = (x.to(dev) for x in (d["q"], d["k"], d["v"], dout))
    rpd = torch.as_tensor(rp, device=dev)
    cid = torch.as_tensor(ci if len(ci) else np.zeros(1, np.int32), device=dev)
    o, lse = bsa.forward(q, k, v, rpd, cid, w.block, scale=w.scale, causal=causal)
    dq, dk, dv = bsa.backward(q, k, v, o, do, lse, rpd, cid, w.block, scale=w.scale, causal=causal)
    torch.cuda.synchronize()
    err = bsa.device_error()
    BH, N, D = w.B * w.H, w.N, w.D
    f64 = lambda t: t.double().numpy().reshape(BH, N, D)
    ref = oracle.attention_backward(f64(d["q"]), f64(d["k"]), f64(d["v"]), f64(dout), rp, ci, w.block,
                                    w.scale, causal, qrows, krows)
    allr = np.arange(BH * N)
    qr = allr if qrows is None else qrows
    kr = allr if krows is None else krows
    got = (dq.reshape(-1, D)[torch.as_tensor(qr, device=dev)],
           dk.reshape(-1, D)[torch.as_tensor(kr, device=dev)],
           dv.reshape(-1, D)[torch.as_tensor(kr, device=dev)])
    out = {}
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        g = g.double().cpu().numpy()
        G = float(np.abs(r).max())
        dd = np.abs(g - r)
        out[name] = (float(dd.max()), float(dd.mean()), G)
    return out, err


def check(stats, what):
    for name, (mx, mean, G) in stats.items():
        assert mx <= TOL_MAX * G, "%s %s max|d| %.3g > %.3g (G %.3g)" % (what, name, mx, TOL_MAX * G, G)
        assert mean <= TOL_MEAN * G, "%s %s mean|d| %.3g > %.3g (G %.3g)" % (what, name, mean, TOL_MEAN * G, G)


@pytest.mark.parametrize("D,causal", [(128, True), (128, False), (64, True)])
def test_backward_window_all_rows(D, causal):
    w = bsa_inputs.Workload("bwd_window", 1, 2, 128 * 12, D, 128, causal=causal, seed=41)
    rp, ci = window_csr(w.B * w.H, w.n_blocks, 3, causal)
    stats, err = run_backward(w, rp, ci, causal)
    assert err == 0
    check(stats, "window")


@pytest.mark.parametrize("D,causal", [(128, True), (64, False)])
def test_backward_many_short_blocks_all_rows(D, causal):
    """640 key blocks of 1-3 steps each: every CTA takes several in turn, so
    the K/V tile slots alternate and a block's next S is issued ahead only
    inside the block."""
    w = bsa_inputs.Workload("bwd_many", 1, 8, 128 * 80, D, 128, causal=causal, seed=47)
    rp, ci = window_csr(w.B * w.H, w.n_blocks, 1, causal)
    stats, err = run_backward(w, rp, ci, causal)
    assert err == 0
    check(stats, "many short blocks")


@pytest.mark.parametrize("D,causal", [(128, False), (128, True), (64, False)])
def test_backward_random_rows_all_rows(D, causal):
    """Unsorted rows, empty rows, key blocks no row lists (dK = dV = 0)."""
    rng = np.random.default_rng(100 + D + causal)
    w = bsa_inputs.Workload("bwd_rand", 1, 2, 128 * 10, D, 128, causal=causal, seed=43)
    rp, ci = random_csr(w.B * w.H, w.n_blocks, rng, 5)
    stats, err = run_backward(w, rp, ci, causal)
    assert err == 0
    check(stats, "random")


@pytest.mark.parametrize("D,causal", [(128, True), (64, False)])
def test_backward_block64_paired(D, causal):
    """64-token blocks in the paired form: window rows (causal) and random
    unsorted rows (empty rows, key blocks no row lists, pairs whose union
    leaves quarters of a step unlisted)."""
    w = bsa_inputs.Workload("bwd_b64", 1, 2, 64 * 20, D, 64, causal=causal, seed=47)
    if causal:
        rp, ci = window_csr(w.B * w.H, w.n_blocks, 4, True)
    else:
        rp, ci = random_csr(w.B * w.H, w.n_blocks, np.random.default_rng(64 + D), 6)
    stats, err = run_backward(w, rp, ci, causal)
    assert err == 0
    check(stats, "block 64")


def test_backward_block64_topk_lists():
    """The content top-k selection's lists (block 64, top-8 + diagonal)."""
    import dataclasses
    w = dataclasses.replace(bsa_inputs.small_workload(bsa_inputs.workload("content_topk"), B=1, H=2, N=64 * 40),
                            topk=8)
    d = bsa_inputs.make_qkv(w)
    rp, ci, _ = oracle.topk_csr(bsa_inputs.bf16_bits(d["q"]), bsa_inputs.bf16_bits(d["k"]), w.block, w.topk,
                                w.include_diag)
    stats, err = run_backward(w, rp, ci, False)
    assert err == 0
    check(stats, "block 64 top-k")


@pytest.mark.parametrize("D", [128, 64])
def test_backward_block64_long_and_short_lists(D):
    """Block 64 with global key blocks every row lists (transposed lists longer
    than the pairing limit of 32: those key blocks run alone, two query blocks
    per step) beside short window lists (paired), causal."""
    w = bsa_inputs.Workload("bwd_b64_global", 1, 2, 64 * 48, D, 64, window_left=2, window_right=0, causal=True,
                            global_blocks=(0, 5), seed=53)
    p = oracle.Pattern.from_workload(w)
    rp1, ci1 = p.csr()
    rp, ci = oracle.replicate_csr(rp1, ci1, w.B * w.H)
    stats, err = run_backward(w, rp, ci, True)
    assert err == 0
    check(stats, "block 64 global + window")


def test_backward_block64_flags_too_small_capacity():
    """Block 64 (paired form) with col_capacity below the CSR's entries: bit 16
    of the device error word is set and every read of the transposed lists
    (pairing pass included) stays below the capacity."""
    import ctypes
    import block_sparse_flashattention_bsa_gb300 as bsa
    from block_sparse_flashattention_bsa_gb300._binding import _Shape
    w = bsa_inputs.Workload("bwd_cap64", 1, 2, 64 * 12, 128, 64, causal=True, seed=57)
    rp, ci = window_csr(w.B * w.H, w.n_blocks, 3, True)
    d = bsa_inputs.make_qkv(w)
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in (d["q"], d["k"], d["v"]))
    do = bsa_inputs.make_grad_out(w).to(dev)
    rpd, cid = torch.as_tensor(rp, device=dev), torch.as_tensor(ci, device=dev)
    o, lse = bsa.forward(q, k, v, rpd, cid, w.block, scale=w.scale, causal=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bsa.device_error()
    sh = _Shape(w.B, w.H, w.N, w.D, w.block)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    st = bsa.lib().bsa_backward(ctypes.byref(sh), P(q), P(k), P(v), P(o), P(do), P(lse), P(rpd), P(cid),
                                len(ci) - 7, P(dq), P(dk), P(dv), ctypes.c_float(w.scale), 1,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert bsa.device_error() & 16


def _head_csr(rp, ci, bh, nb):
    """The CSR rows of head slab bh alone (row_ptr rebased to 0)."""
    a, b = int(rp[bh * nb]), int(rp[(bh + 1) * nb])
    return (rp[bh * nb:(bh + 1) * nb + 1] - a).astype(np.int32), np.asarray(ci[a:b], np.int32)


def test_backward_full_size_content_topk_sampled():
    """content_topk at full size (B=2 H=16 N=32768, block 64, paired form), in
    the benchmark's launch configuration: top-k CSR on the device (checked
    bit-exactly against the oracle's), forward, backward over every head.
    The oracle then checks dQ, dK, dV on sampled rows of three seeded heads
    (query and key blocks {0, 1, 2, nb-1} plus six random ones per head), from
    that head's inputs and CSR rows alone (heads do not interact)."""
    import block_sparse_flashattention_bsa_gb300 as bsa
    from parity import gpu_csr, oracle_csr
    w = bsa_inputs.workload("content_topk")
    d = bsa_inputs.make_qkv(w)
    dout = bsa_inputs.make_grad_out(w)
    dev = torch.device("cuda")
    q, k, v, do = (x.to(dev) for x in (d["q"], d["k"], d["v"], dout))
    rp_ref, ci_ref = oracle_csr(w, d["q"], d["k"])
    rp, ci = gpu_csr(w, q, k)
    np.testing.assert_array_equal(rp.cpu().numpy(), rp_ref)
    np.testing.assert_array_equal(ci.cpu().numpy(), ci_ref)
    o, lse = bsa.forward(q, k, v, rp, ci, w.block, scale=w.scale, causal=w.causal)
    dq, dk, dv = bsa.backward(q, k, v, o, do, lse, rp, ci, w.block, scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    assert bsa.device_error() == 0
    BH, N, D, nb = w.B * w.H, w.N, w.D, w.n_blocks
    rng = np.random.default_rng(2027)
    heads = sorted(int(x) for x in rng.choice(BH, size=3, replace=False))
    one = bsa_inputs.Workload("one_head", 1, 1, N, D, w.block, causal=w.causal)
    f64 = lambda t, bh: t.reshape(BH, N, D)[bh:bh + 1].double().numpy()
    for bh in heads:
        rows = bsa_inputs.sample_rows(one, n_random_blocks=6, seed=bh).numpy()
        rph, cih = _head_csr(rp_ref, ci_ref, bh, nb)
        ref = oracle.attention_backward(f64(d["q"], bh), f64(d["k"], bh), f64(d["v"], bh), f64(dout, bh), rph, cih,
                                        w.block, w.scale, w.causal, rows, rows)
        sel = torch.as_tensor(bh * N + rows, device=dev)
        got = [t.reshape(-1, D)[sel].double().cpu().numpy() for t in (dq, dk, dv)]
        stats = {}
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            dd = np.abs(g - r)
            stats[name] = (float(dd.max()), float(dd.mean()), float(np.abs(r).max()))
        check(stats, "content_topk head %d" % bh)


@pytest.mark.parametrize("name", ["window_global_64k", "long_window_128k"])
def test_backward_full_size_long_windows_sampled(name):
    """The long-window workloads at full size (B=1 H=32, N 65536 / 131072),
    mask built on the device as the benchmark does, backward over every head.
    The oracle checks one seeded head: dQ on the rows of query blocks {0, 1,
    2, nb-1} plus four random ones, dK and dV on the rows of key blocks 2,
    nb-1 and one random block (not a global block, whose gradients gather
    every query row of the head: too slow for the fp64 oracle here; the
    global blocks are checked at small size), from that head's inputs and CSR
    rows alone (heads do not interact)."""
    import block_sparse_flashattention_bsa_gb300 as bsa
    from parity import gpu_csr, oracle_csr
    w = bsa_inputs.workload(name)
    d = bsa_inputs.make_qkv(w)
    dout = bsa_inputs.make_grad_out(w)
    dev = torch.device("cuda")
    q, k, v, do = (x.to(dev) for x in (d["q"], d["k"], d["v"], dout))
    rp_ref, ci_ref = oracle_csr(w)
    rp, ci = gpu_csr(w, q, k)
    np.testing.assert_array_equal(rp.cpu().numpy(), rp_ref)
    np.testing.assert_array_equal(ci.cpu().numpy(), ci_ref)
    o, lse = bsa.forward(q, k, v, rp, ci, w.block, scale=w.scale, causal=w.causal)
    dq, dk, dv = bsa.backward(q, k, v, o, do, lse, rp, ci, w.block, scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    assert bsa.device_error() == 0
    BH, N, D, nb = w.B * w.H, w.N, w.D, w.n_blocks
    rng = np.random.default_rng(2028)
    bh = int(rng.integers(0, BH))
    one = bsa_inputs.Workload("one_head", 1, 1, N, D, w.block, causal=w.causal)
    qrows = bsa_inputs.sample_rows(one, n_random_blocks=4, seed=bh).numpy()
    kblocks = [2, nb - 1, int(rng.integers(len(w.global_blocks) + 1, nb - 1))]
    assert not set(kblocks) & set(w.global_blocks)
    krows = np.concatenate([np.arange(j * w.block, (j + 1) * w.block) for j in kblocks]).astype(np.int64)
    f64 = lambda t: t.reshape(BH, N, D)[bh:bh + 1].double().numpy()
    rph, cih = _head_csr(rp_ref, ci_ref, bh, nb)
    ref = oracle.attention_backward(f64(d["q"]), f64(d["k"]), f64(d["v"]), f64(dout), rph, cih,
                                    w.block, w.scale, w.causal, qrows, krows)
    stats = {}
    for nm, t, rows, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), (qrows, krows, krows), ref):
        g = t.reshape(-1, D)[torch.as_tensor(bh * N + rows, device=dev)].double().cpu().numpy()
        dd = np.abs(g - r)
        stats[nm] = (float(dd.max()), float(dd.mean()), float(np.abs(r).max()))
    check(stats, "%s head %d" % (name, bh))


def test_backward_full_size_window_16k_sampled():
    w = bsa_inputs.workload("window_16k")
    rp, ci = window_csr(w.B * w.H, w.n_blocks, w.window_left, w.causal)
    rows = bsa_inputs.sample_rows(w, n_random_blocks=4).numpy()
    stats, err = run_backward(w, rp, ci, w.causal, qrows=rows, krows=rows)
    assert err == 0
    check(stats, "window_16k sampled")


def test_backward_global_rows_and_blocks():
    """Global key blocks every row sees and global query rows that see every
    block (long transposed lists for the global key blocks)."""
    import block_sparse_flashattention_bsa_gb300 as bsa
    w = bsa_inputs.Workload("bwd_global", 1, 2, 128 * 10, 128, 128, window_left=1, window_right=0, causal=True,
                            global_blocks=(0, 3), global_rows_attend_all=True, seed=49)
    p = oracle.Pattern.from_workload(w)
    rp1, ci1 = p.csr()
    rp, ci = oracle.replicate_csr(rp1, ci1, w.B * w.H)
    stats, err = run_backward(w, rp, ci, True)
    assert err == 0
    check(stats, "global rows and blocks")


def test_backward_flags_too_small_capacity():
    """col_capacity below the CSR's entries: the extra entries are dropped and
    bit 16 of the device error word is set; nothing is written out of bounds."""
    import ctypes
    import block_sparse_flashattention_bsa_gb300 as bsa
    from block_sparse_flashattention_bsa_gb300._binding import _Shape
    w = bsa_inputs.Workload("bwd_cap", 1, 1, 128 * 6, 64, 128, causal=True, seed=51)
    rp, ci = window_csr(w.B * w.H, w.n_blocks, 2, True)
    d = bsa_inputs.make_qkv(w)
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in (d["q"], d["k"], d["v"]))
    do = bsa_inputs.make_grad_out(w).to(dev)
    rpd, cid = torch.as_tensor(rp, device=dev), torch.as_tensor(ci, device=dev)
    o, lse = bsa.forward(q, k, v, rpd, cid, w.block, scale=w.scale, causal=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bsa.device_error()
    sh = _Shape(w.B, w.H, w.N, w.D, w.block)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    st = bsa.lib().bsa_backward(ctypes.byref(sh), P(q), P(k), P(v), P(o), P(do), P(lse), P(rpd), P(cid),
                                len(ci) - 3, P(dq), P(dk), P(dv), ctypes.c_float(w.scale), 1,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert bsa.device_error() & 16
