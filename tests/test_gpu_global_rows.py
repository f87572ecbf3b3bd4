"""GPU parity for global query rows that take no causal cut.

In a causal model a global query block may still "attend to everything"
("Flash MSA Sparse Attention vs Full Attention", "Sparse Patterns Beyond
Sliding Windows", "Global Tokens"); the 128K workload's "block 0 ... itself
attends to all blocks" read literally is such a row.  The pattern's
global_rows_noncausal lists every key block for those rows, bsa_pattern_row_flags
marks them, and bsa_forward_ex lifts the causal cut for the flagged rows only.

Checked against the fp64 oracle (orc_pattern_csr with the same field, and
orc_attention_rows with the same flags): CSR and flags bit-exact; the forward
element by element at the stated tolerances, on every row of small cases
(blocks 128 and 64, head dims 128 and 64, random unsorted CSRs with random
flags) and on every query block of two heads of the full-size 128K workload
with its sink row attending to everything.  The backward (bsa_backward_ex)
takes the same flags and is checked against the oracle's backward with them
on every row of small cases (blocks 128 and 64, random flags; the pattern's
global rows).
"""

import numpy as np
import pytest
import torch

import bsa_inputs
import oracle
from parity import assert_close, bits, compare

pytestmark = pytest.mark.gpu

W = {w.name: w for w in bsa_inputs.WORKLOADS}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_flashattention_bsa_gb300 import build
    build.build()
    import block_sparse_flashattention_bsa_gb300 as bsa
    bsa.device_error()


def _pattern_pair(w):
    import block_sparse_flashattention_bsa_gb300 as bsa
    args = (w.n_blocks, w.window_left, w.window_right, w.causal, w.global_blocks, w.global_rows_attend_all,
            w.global_rows_noncausal)
    return bsa.Pattern(*args), oracle.Pattern(*args)


def _run(w, rows=None, heads=None):
    import block_sparse_flashattention_bsa_gb300 as bsa
    d = bsa_inputs.make_qkv(w)
    dev = torch.device("cuda")
    q, k, v = (d[x].to(dev) for x in "qkv")
    pg, po = _pattern_pair(w)
    rp, ci = bsa.build_mask_csr(pg, w.B, w.H, device=dev)
    flags = bsa.pattern_row_flags(pg, w.B, w.H, device=dev)
    rp1, ci1 = po.csr()
    rp_ref, ci_ref = oracle.replicate_csr(rp1, ci1, w.B * w.H)
    fl_ref = np.tile(po.row_flags(), w.B * w.H)
    np.testing.assert_array_equal(rp.cpu().numpy(), rp_ref)
    np.testing.assert_array_equal(ci.cpu().numpy(), ci_ref)
    np.testing.assert_array_equal(flags.cpu().numpy(), fl_ref)
    o, lse = bsa.forward_ex(q, k, v, rp, ci, w.block, scale=w.scale, causal=w.causal, row_flags=flags)
    torch.cuda.synchronize()
    assert bsa.device_error() == 0
    if rows is None:
        rows = np.arange(w.B * w.H * w.N, dtype=np.int64)
    O_ref, L_ref = oracle.attention_rows(bits(d["q"]), bits(d["k"]), bits(d["v"]), rp_ref, ci_ref, w.block,
                                         w.scale, w.causal, rows=rows, row_flags=fl_ref)
    return compare(o, lse, O_ref, L_ref, rows, w.D)


@pytest.mark.parametrize("base,kw", [
    ("long_window_128k", dict(H=2, N=128 * 48)),
    ("window_global_64k", dict(H=2, N=128 * 80)),
    ("tiny_window_global", dict(H=3, causal=True)),              # block 64 (paired form), D 64
    ("window_global_64k", dict(H=2, N=128 * 40, D=64)),          # block 128, D 64
])
def test_global_rows_noncausal_all_rows(base, kw):
    w = bsa_inputs.small_workload(W[base], **kw).with_(global_rows_noncausal=True)
    assert_close(_run(w), "%s non-causal global rows" % base)


def test_long_window_128k_sink_row_attends_everything_full_size():
    """The full-size 128K workload with block 0 attending to every block:
    every query block of two heads, row 0 (1024 key blocks) included."""
    w = W["long_window_128k"].with_(global_rows_noncausal=True)
    rng = np.random.default_rng(128)
    heads = sorted(int(x) for x in rng.choice(w.B * w.H, size=2, replace=False))
    rows = np.concatenate([bsa_inputs.head_rows(w, bh).numpy() for bh in heads])
    assert_close(_run(w, rows=rows), "long_window_128k sink row")


@pytest.mark.parametrize("block,D", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_random_rows_with_random_flags(block, D):
    """Random unsorted CSRs (future blocks and empty rows included) with a
    random third of the rows flagged: the causal cut is lifted exactly there."""
    import block_sparse_flashattention_bsa_gb300 as bsa
    rng = np.random.default_rng(block * 3 + D)
    w = bsa_inputs.Workload("flags", 1, 3, block * 14, D, block, causal=True, seed=17)
    nb = w.n_blocks
    rp, ci = [0], []
    for _ in range(w.B * w.H * nb):
        n = int(rng.integers(0, 9))
        ci += [int(x) for x in rng.choice(nb, size=n, replace=False)]
        rp.append(len(ci))
    rp, ci = np.array(rp, np.int32), np.array(ci, np.int32)
    fl = (rng.random(w.B * w.H * nb) < 0.33).astype(np.uint8)
    d = bsa_inputs.make_qkv(w)
    dev = torch.device("cuda")
    q, k, v = (d[x].to(dev) for x in "qkv")
    o, lse = bsa.forward_ex(q, k, v, torch.as_tensor(rp, device=dev), torch.as_tensor(ci, device=dev), block,
                            scale=w.scale, causal=True, row_flags=torch.as_tensor(fl, device=dev))
    torch.cuda.synchronize()
    assert bsa.device_error() == 0
    rows = np.arange(w.B * w.H * w.N, dtype=np.int64)
    O_ref, L_ref = oracle.attention_rows(bits(d["q"]), bits(d["k"]), bits(d["v"]), rp, ci, block, w.scale, True,
                                         rows=rows, row_flags=fl)
    assert_close(compare(o, lse, O_ref, L_ref, rows, D), "random flags %d/%d" % (block, D))


# ------------------------------------------------------------------ backward
BWD_TOL_MAX, BWD_TOL_MEAN = 2e-2, 2e-3  # of the largest reference gradient, as in test_gpu_backward


def _bwd_check(w, rp, ci, fl, what):
    """Forward (bsa_forward_ex) then backward (bsa_backward_ex) with the same
    flags, every row, against the oracle's backward with those flags."""
    import block_sparse_flashattention_bsa_gb300 as bsa
    d = bsa_inputs.make_qkv(w)
    dout = bsa_inputs.make_grad_out(w)
    dev = torch.device("cuda")
    q, k, v, do = (x.to(dev) for x in (d["q"], d["k"], d["v"], dout))
    rpd = torch.as_tensor(rp, device=dev)
    cid = torch.as_tensor(ci if len(ci) else np.zeros(1, np.int32), device=dev)
    fld = torch.as_tensor(fl, device=dev)
    o, lse = bsa.forward_ex(q, k, v, rpd, cid, w.block, scale=w.scale, causal=True, row_flags=fld)
    dq, dk, dv = bsa.backward(q, k, v, o, do, lse, rpd, cid, w.block, scale=w.scale, causal=True, row_flags=fld)
    torch.cuda.synchronize()
    assert bsa.device_error() == 0
    BH, N, D = w.B * w.H, w.N, w.D
    f64 = lambda t: t.double().numpy().reshape(BH, N, D)
    ref = oracle.attention_backward(f64(d["q"]), f64(d["k"]), f64(d["v"]), f64(dout), rp, ci, w.block, w.scale,
                                    True, row_flags=fl)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        dd = np.abs(g.reshape(-1, D).double().cpu().numpy() - r)
        G = float(np.abs(r).max())
        assert dd.max() <= BWD_TOL_MAX * G, "%s %s max|d| %.3g (G %.3g)" % (what, name, dd.max(), G)
        assert dd.mean() <= BWD_TOL_MEAN * G, "%s %s mean|d| %.3g (G %.3g)" % (what, name, dd.mean(), G)


@pytest.mark.parametrize("block,D", [(128, 128), (64, 128), (64, 64)])
def test_backward_random_rows_with_random_flags(block, D):
    """The backward with per-row causal flags: random unsorted CSRs (future
    blocks and empty rows included), a random third of the rows flagged;
    block 64 runs the paired form."""
    rng = np.random.default_rng(block * 5 + D)
    w = bsa_inputs.Workload("flags_bwd", 1, 2, block * 12, D, block, causal=True, seed=19)
    nb = w.n_blocks
    rp, ci = [0], []
    for _ in range(w.B * w.H * nb):
        n = int(rng.integers(0, 8))
        ci += [int(x) for x in rng.choice(nb, size=n, replace=False)]
        rp.append(len(ci))
    rp, ci = np.array(rp, np.int32), np.array(ci, np.int32)
    fl = (rng.random(w.B * w.H * nb) < 0.33).astype(np.uint8)
    _bwd_check(w, rp, ci, fl, "random flags %d/%d" % (block, D))


def test_backward_pattern_global_rows_noncausal():
    """The pattern path: global query rows of a causal window + global pattern
    attending to every block (bsa_pattern_row_flags), forward and backward."""
    import block_sparse_flashattention_bsa_gb300 as bsa
    w = bsa_inputs.small_workload(W["window_global_64k"], H=2, N=128 * 24).with_(global_rows_noncausal=True)
    pg, po = _pattern_pair(w)
    rp1, ci1 = po.csr()
    rp, ci = oracle.replicate_csr(rp1, ci1, w.B * w.H)
    fl = np.tile(po.row_flags(), w.B * w.H)
    flags = bsa.pattern_row_flags(pg, w.B, w.H, device=torch.device("cuda"))
    np.testing.assert_array_equal(flags.cpu().numpy(), fl)
    _bwd_check(w, rp, ci, fl, "window + global, non-causal global rows")
