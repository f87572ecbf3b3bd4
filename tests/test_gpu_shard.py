"""GPU parity of the sequence-sharded forward's device work, on one GPU.

The collectives and the planners are checked on CPU ranks
(test_multiprocess_shard.py); what they deliver to a rank is fixed by the
plan.  Here every rank of a 2- and a 4-way split is run in turn on the one
GPU, its received blocks placed by bsa_copy_blocks straight from the full
tensors (the blocks the all-to-all would bring), and the device operations
checked against the unsharded fp64 oracle at the stated tolerances
(max |dO| <= 1e-2, mean |dO| <= 1e-3, max |dLSE| <= 1e-3):

* key/value exchange: bsa_forward_ex on the extended key range through the
  renumbered CSR, with q_block_offset = n_before;
* partial outputs: the local part (bsa_forward_ex on the shard), every peer's
  guest rows computed at the key owner (bsa_forward_ex, no causal cut), and
  the partial results merged by bsa_merge_partial_blocks;
* the merge kernel alone against the oracle's merge_partials (fp32 parts,
  fp32 arithmetic: 1e-5).  Partial results stay fp32 until the merge is
  done: a bf16 partial adds its own rounding (up to 2^-9 |O|) to the final
  one, which the clustered top-k rows (|O| up to 3.3) cannot afford.

No kernel here waits on another rank: the ranks run one after another.
"""

import numpy as np
import pytest
import torch

import bsa_inputs
import oracle
from parity import TOL_LSE, assert_close, bits, compare

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


def _rank_rows(w, rp, ci, flags, first, count):
    nb = w.n_blocks
    BH = w.B * w.H
    rows = [ci[rp[bh * nb + i]:rp[bh * nb + i + 1]] for bh in range(BH) for i in range(first, first + count)]
    lrp = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    lci = np.concatenate(rows).astype(np.int32)
    lfl = None if flags is None else np.concatenate([flags[bh * nb + first: bh * nb + first + count]
                                                     for bh in range(BH)])
    return lrp, lci, lfl


def _oracle_rows(w, d, rp, ci, flags, first, count):
    N = w.N
    rows = np.concatenate([np.arange(bh * N + first * w.block, bh * N + (first + count) * w.block)
                           for bh in range(w.B * w.H)])
    O, L = oracle.attention_rows(bits(d["q"]), bits(d["k"]), bits(d["v"]), rp, ci, w.block, w.scale, w.causal,
                                 rows=rows, row_flags=flags)
    return O, L


CASES = [
    ("window_global_64k", dict(H=2, N=128 * 64), False),
    ("long_window_128k", dict(H=2, N=128 * 96), True),     # sink row without the causal cut
    ("content_topk", dict(B=1, H=2, N=64 * 64), False),    # block 64 (paired form), per-head lists
]


def _csr_for(w, d):
    if w.is_topk:
        rp, ci, _ = oracle.topk_csr(bits(d["q"]), bits(d["k"]), w.block, w.topk, w.include_diag)
        return rp, ci, None
    po = oracle.Pattern.from_workload(w)
    rp, ci = oracle.replicate_csr(*po.csr(), w.B * w.H)
    return rp, ci, (np.tile(po.row_flags(), w.B * w.H) if w.global_rows_noncausal else None)


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("name,kw,grnc", CASES, ids=[c[0] for c in CASES])
def test_kv_exchange_forward(world, name, kw, grnc):
    from block_sparse_flashattention_bsa_gb300 import seqshard
    w = bsa_inputs.small_workload(W[name], **kw).with_(global_rows_noncausal=grnc)
    d = bsa_inputs.make_qkv(w)
    rp, ci, flags = _csr_for(w, d)
    ops = seqshard.DeviceOps()
    dev = torch.device("cuda")
    BH, N, D, bs, nb = w.B * w.H, w.N, w.D, w.block, w.n_blocks
    kf, vf = (d[x].to(dev).reshape(-1, D) for x in "kv")
    qf = d["q"].to(dev)
    for rank in range(world):
        first, count = seqshard.shard_range(world, rank, nb, BH)
        lrp, lci, lfl = _rank_rows(w, rp, ci, flags, first, count)
        plan = seqshard.plan_kv(world, rank, nb, BH, lrp, lci)
        Ne = plan.n_k_ext * bs
        k_ext = torch.zeros((w.B, w.H, Ne, D), dtype=torch.bfloat16, device=dev)
        v_ext = torch.zeros_like(k_ext)
        # the shard itself and the fetched blocks, as the exchange places them
        own_src = (np.arange(BH)[:, None] * N + (first + np.arange(count))[None, :] * bs).reshape(-1)
        own_dst = (np.arange(BH)[:, None] * Ne + (plan.n_before + np.arange(count))[None, :] * bs).reshape(-1)
        rem_src = plan.need_bh.astype(np.int64) * N + plan.need_j.astype(np.int64) * bs
        rem_dst = plan.need_bh.astype(np.int64) * Ne + plan.need_pos.astype(np.int64) * bs
        for full, ext in ((kf, k_ext), (vf, v_ext)):
            ops.copy_blocks(full, ext.reshape(-1, D), own_src, own_dst, bs)
            ops.copy_blocks(full, ext.reshape(-1, D), rem_src, rem_dst, bs)
        q_loc = qf[:, :, first * bs:(first + count) * bs].contiguous()
        o, lse = ops.forward_ex(q_loc, k_ext, v_ext, lrp, plan.col_idx_ext, bs, w.scale, w.causal, lfl,
                                plan.n_before)
        torch.cuda.synchronize()
        import block_sparse_flashattention_bsa_gb300 as bsa
        assert bsa.device_error() == 0
        O, L = _oracle_rows(w, d, rp, ci, flags, first, count)
        assert_close(compare(o, lse, O, L, np.arange(len(L)), D), "%s rank %d/%d" % (name, rank, world))


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("name,kw,grnc", CASES, ids=[c[0] for c in CASES])
def test_partial_outputs_merged(world, name, kw, grnc):
    import block_sparse_flashattention_bsa_gb300 as bsa
    from block_sparse_flashattention_bsa_gb300 import seqshard
    w = bsa_inputs.small_workload(W[name], **kw).with_(global_rows_noncausal=grnc)
    d = bsa_inputs.make_qkv(w)
    rp, ci, flags = _csr_for(w, d)
    ops = seqshard.DeviceOps()
    dev = torch.device("cuda")
    B, H, BH, N, D, bs, nb = w.B, w.H, w.B * w.H, w.N, w.D, w.block, w.n_blocks
    qf, kf, vf = (d[x].to(dev) for x in "qkv")
    shards = [seqshard.shard_range(world, g, nb, BH) for g in range(world)]
    rows_of = [_rank_rows(w, rp, ci, flags, f, c) for f, c in shards]
    plans = [seqshard.plan_partial(world, g, nb, BH, rows_of[g][0], rows_of[g][1], w.causal, rows_of[g][2])
             for g in range(world)]
    loc = lambda t, g: t[:, :, shards[g][0] * bs:(shards[g][0] + shards[g][1]) * bs].contiguous()  # noqa: E731
    for g in range(world):
        f, c = shards[g]
        Nl = c * bs
        pl = plans[g]
        o, lse = ops.forward_ex(loc(qf, g), loc(kf, g), loc(vf, g), pl.local_row_ptr, pl.local_col_idx, bs, w.scale,
                                w.causal, rows_of[g][2], 0, out_f32=True)
        off_rows, off_ents = 0, 0
        for p in range(world):
            n, ne = pl.guest_rows_by_rank[p], pl.guest_entries_by_rank[p]
            if n == 0:
                continue
            gq = pl.guest_q[off_rows:off_rows + n].astype(np.int64)
            gp = pl.guest_ptr[off_rows:off_rows + n + 1]
            ent = pl.guest_col[gp[0]:gp[-1]]
            hdr = np.stack([(gq // c).astype(np.int32), np.diff(gp).astype(np.int32)], 1)
            gmax, row_of, grp, gci = seqshard.guest_layout(hdr, ent, BH)
            qg = torch.zeros((B, H, gmax * bs, D), dtype=torch.bfloat16, device=dev)
            src = (gq // c) * Nl + (gq % c) * bs
            ops.copy_blocks(loc(qf, g).reshape(-1, D), qg.reshape(-1, D), src, row_of * bs, bs)
            og, lg = ops.forward_ex(qg, loc(kf, p), loc(vf, p), grp, gci, bs, w.scale, False, None, 0, out_f32=True)
            po = torch.empty((n * bs, D), dtype=torch.float32, device=dev)
            plse = torch.empty((n, bs), dtype=torch.float32, device=dev)
            ops.copy_blocks(og.reshape(-1, D), po, row_of * bs, np.arange(n, dtype=np.int64) * bs, bs)
            ops.copy_blocks(lg.reshape(-1, bs), plse, row_of, np.arange(n, dtype=np.int64), 1)
            ops.merge(o.reshape(-1, D), lse.reshape(-1), po, plse.reshape(-1), src, bs)
            off_rows += n
            off_ents += ne
        o = ops.to_bf16(o)
        torch.cuda.synchronize()
        assert bsa.device_error() == 0
        O, L = _oracle_rows(w, d, rp, ci, flags, f, c)
        assert_close(compare(o, lse, O, L, np.arange(len(L)), D), "%s rank %d/%d merged" % (name, g, world))


def test_merge_kernel_against_oracle():
    """bsa_merge_partial_blocks on random partial results (some parts empty,
    some accumulator rows empty) against the oracle's merge_partials."""
    from block_sparse_flashattention_bsa_gb300 import seqshard
    g = torch.Generator().manual_seed(99)
    rows_acc, bs, D, nblk = 64 * 10, 64, 128, 6
    o_acc = torch.randn(rows_acc, D, generator=g) * 0.5
    l_acc = torch.randn(rows_acc, generator=g) * 3
    l_acc[:64] = -float("inf")
    o_acc[:64] = 0
    o_part = torch.randn(nblk * bs, D, generator=g) * 0.5
    l_part = torch.randn(nblk * bs, generator=g) * 3
    l_part[bs:2 * bs:3] = -float("inf")
    dst = np.array([0, 2, 3, 5, 7, 9], np.int64) * bs
    dev = torch.device("cuda")
    oa, la = o_acc.to(dev), l_acc.to(dev)
    seqshard.DeviceOps().merge(oa, la, o_part.to(dev), l_part.to(dev), dst, bs)
    torch.cuda.synchronize()
    O_ref = o_acc.double().numpy().copy()
    L_ref = l_acc.double().numpy().copy()
    for n, d0 in enumerate(dst):
        sl, ps = slice(d0, d0 + bs), slice(n * bs, (n + 1) * bs)
        Om, Lm = oracle.merge_partials([o_acc[sl].double().numpy(), o_part[ps].double().numpy()],
                                       [l_acc[sl].double().numpy(), l_part[ps].double().numpy()])
        O_ref[sl], L_ref[sl] = Om, Lm
    dO = np.abs(oa.double().cpu().numpy() - O_ref)
    assert dO.max() <= 1e-5 and dO.mean() <= 1e-6   # fp32 arithmetic on fp32 parts
    lg = la.double().cpu().numpy()
    both = np.isneginf(lg) & np.isneginf(L_ref)
    assert np.array_equal(np.isneginf(lg), np.isneginf(L_ref))
    assert np.abs(np.where(both, 0, lg - L_ref)).max() <= TOL_LSE
