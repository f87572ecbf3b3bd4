"""The sequence-sharded forward's host logic on CPU ranks (gloo).

Two and three ranks each hold one contiguous shard of the query and key
blocks and the CSR rows of their own query blocks.  The planners
(bsa_shard_plan_kv, bsa_shard_plan_partial in libbsa.so, host code), the
all-to-all exchanges (torch.distributed over gloo, the same calls NCCL runs
on GPUs) and the bookkeeping of both strategies run exactly as on GPUs; the
three device operations (block copy, forward, merge) are replaced by CPU
stand-ins built from the fp64 oracle, so every rank's result must equal the
unsharded oracle's rows to rounding (1e-12).  Patterns: sliding window plus
global blocks (causal), the same with global query rows that take no causal
cut (their rows fetch blocks after the shard), and random unsorted CSRs with
empty rows, non-causal and causal.  The device operations themselves are
checked on the GPU in test_gpu_shard.py.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle

BH, NB, BS, D = 3, 13, 8, 16


class CpuOps:
    """CPU stand-ins for the three device operations (test infrastructure)."""

    def copy_blocks(self, src, dst, src_rows, dst_rows, rows_per_block):
        for s, d in zip(np.asarray(src_rows, np.int64), np.asarray(dst_rows, np.int64)):
            dst[d:d + rows_per_block] = src[s:s + rows_per_block]

    def forward_ex(self, q, k, v, row_ptr, col_idx, block, scale, causal, row_flags, q_block_offset,
                   out_f32=False):
        B, H, Nq, Dd = q.shape
        O, L = oracle.attention_blocks_f64(q.reshape(B * H, Nq, Dd).numpy(), k.reshape(B * H, -1, Dd).numpy(),
                                           v.reshape(B * H, -1, Dd).numpy(), np.asarray(row_ptr),
                                           np.asarray(col_idx), block, scale, causal, row_flags=row_flags,
                                           q_block_offset=q_block_offset)
        return torch.from_numpy(O).reshape(B, H, Nq, Dd), torch.from_numpy(L).reshape(B, H, Nq)

    def to_bf16(self, x):
        return x  # fp64 stays fp64: the comparison is to rounding

    def merge(self, o_acc, lse_acc, o_part, lse_part, dst_rows, rows_per_block):
        for n, d in enumerate(np.asarray(dst_rows, np.int64)):
            sl = slice(d, d + rows_per_block)
            ps = slice(n * rows_per_block, (n + 1) * rows_per_block)
            Om, Lm = oracle.merge_partials([o_acc[sl].numpy(), o_part[ps].numpy()],
                                           [lse_acc[sl].numpy(), lse_part[ps].numpy()])
            o_acc[sl] = torch.from_numpy(Om)
            lse_acc[sl] = torch.from_numpy(Lm)


def _case(kind):
    """Full problem: q, k, v fp64 [BH, N, D], CSR over BH*NB rows, causal, flags."""
    rng = np.random.default_rng(sum(map(ord, kind)))
    N = NB * BS
    q, k, v = (rng.standard_normal((BH, N, D)) for _ in range(3))
    flags = None
    if kind in ("window_global", "global_rows_noncausal"):
        grnc = kind == "global_rows_noncausal"
        p = oracle.Pattern(NB, 3, 0, True, (0, 6), True, grnc)
        rp, ci = oracle.replicate_csr(*p.csr(), BH)
        causal = True
        if grnc:
            flags = np.tile(p.row_flags(), BH)
    else:
        causal = kind == "random_causal"
        rp, ci = [0], []
        for _ in range(BH * NB):
            n = int(rng.integers(0, 7))
            ci += [int(x) for x in rng.choice(NB, size=n, replace=False)]
            rp.append(len(ci))
        rp, ci = np.array(rp, np.int32), np.array(ci, np.int32)
    return q, k, v, np.asarray(rp, np.int32), np.asarray(ci, np.int32), causal, flags


def _worker(rank, world, port, kind, strategy):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from block_sparse_flashattention_bsa_gb300 import seqshard
        q, k, v, rp, ci, causal, flags = _case(kind)
        scale = 0.31
        first, count = seqshard.shard_range(world, rank, NB, BH)
        sl = slice(first * BS, (first + count) * BS)
        # this rank's rows of the CSR (entries stay global ids) and flags
        rows = [ci[rp[bh * NB + i]:rp[bh * NB + i + 1]] for bh in range(BH) for i in range(first, first + count)]
        lrp = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
        lci = np.concatenate(rows).astype(np.int32) if rows else np.zeros(0, np.int32)
        lfl = None if flags is None else np.concatenate(
            [flags[bh * NB + first: bh * NB + first + count] for bh in range(BH)])
        ql, kl, vl = (torch.from_numpy(np.ascontiguousarray(x[:, sl])).reshape(1, BH, count * BS, D)
                      for x in (q, k, v))
        fn = seqshard.forward_kv_exchange if strategy == "kv" else seqshard.forward_partial_merge
        o, lse, plan = fn(ql, kl, vl, lrp, lci, BS, NB, scale=scale, causal=causal, row_flags=lfl, ops=CpuOps())
        # the unsharded oracle's rows of this shard
        want = np.concatenate([np.arange(bh * NB * BS + first * BS, bh * NB * BS + (first + count) * BS)
                               for bh in range(BH)])
        O, L = oracle.attention_blocks_f64(q, k, v, rp, ci, BS, scale, causal, rows=want, row_flags=flags)
        og = o.reshape(-1, D).numpy()
        lg = lse.reshape(-1).numpy()
        np.testing.assert_allclose(og, O, rtol=0, atol=1e-12)
        both = np.isneginf(lg) & np.isneginf(L)
        assert np.array_equal(np.isneginf(lg), np.isneginf(L))
        np.testing.assert_allclose(np.where(both, 0, lg), np.where(both, 0, L), rtol=0, atol=1e-12)
        if strategy == "kv" and kind == "global_rows_noncausal" and rank < world - 1:
            assert plan.n_after > 0  # global rows fetch blocks after the shard
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("strategy", ["kv", "merge"])
@pytest.mark.parametrize("kind", ["window_global", "global_rows_noncausal", "random", "random_causal"])
def test_sharded_forward_equals_unsharded(world, strategy, kind):
    from block_sparse_flashattention_bsa_gb300 import build
    build.build()
    oracle.build()
    mp.spawn(_worker, args=(world, _free_port(), kind, strategy), nprocs=world, join=True)


def test_plans_on_the_host():
    """Plan details against brute force: the renumbered entries map back to
    the same global blocks, every remote block is fetched exactly once from
    its owner, and the partial plan's parts partition each row."""
    from block_sparse_flashattention_bsa_gb300 import build, seqshard
    build.build()
    q, k, v, rp, ci, causal, flags = _case("global_rows_noncausal")
    world = 3
    for rank in range(world):
        first, count = seqshard.shard_range(world, rank, NB, BH)
        rows = [ci[rp[bh * NB + i]:rp[bh * NB + i + 1]] for bh in range(BH) for i in range(first, first + count)]
        lrp = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
        lci = np.concatenate(rows).astype(np.int32)
        plan = seqshard.plan_kv(world, rank, NB, BH, lrp, lci)
        owners = [seqshard.shard_range(world, p, NB, BH) for p in range(world)]
        fetched = {}
        for x, (bh, j, pos) in enumerate(zip(plan.need_bh, plan.need_j, plan.need_pos)):
            assert not (first <= j < first + count)
            fetched[(int(bh), int(pos))] = int(j)
        assert len(fetched) == len(plan.need_bh)
        for r in range(BH * count):
            bh = r // count
            for e in range(lrp[r], lrp[r + 1]):
                j, x = int(lci[e]), int(plan.col_idx_ext[e])
                if first <= j < first + count:
                    assert x == plan.n_before + j - first
                else:
                    assert fetched[(bh, x)] == j
        # the per-owner counts
        for p in range(world):
            f, c = owners[p]
            assert plan.need_count_by_rank[p] == sum(1 for j in plan.need_j if f <= j < f + c)
        # extended order = global order
        for bh in range(BH):
            m = {pos: j for (b, pos), j in fetched.items() if b == bh}
            m.update({plan.n_before + i: first + i for i in range(count)})
            ks = sorted(m)
            assert [m[x] for x in ks] == sorted(m.values())
        pp = seqshard.plan_partial(world, rank, NB, BH, lrp, lci, True,
                                   np.concatenate([flags[bh * NB + first: bh * NB + first + count]
                                                   for bh in range(BH)]))
        assert pp.local_row_ptr[-1] == sum(1 for j in lci if first <= j < first + count)
