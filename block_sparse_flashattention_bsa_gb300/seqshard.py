"""Sequence-sharded block-sparse forward over torch.distributed ranks.

"How Do Sparse Attention Kernels Work in GPU Clusters?", section
"Distributed Sparse Attention", gives two ways to run the forward on a
sequence split across GPUs; both are here:

* :func:`forward_kv_exchange` -- a sparse all-to-all of the key/value blocks
  each rank's rows need (indices first, then the blocks), into the rank's own
  memory, then the unchanged forward on the rank's query blocks against the
  extended key range (received blocks before the shard, the shard, received
  blocks after it) through a renumbered CSR;
* :func:`forward_partial_merge` -- local attention against the rank's own key
  blocks, the query blocks that need other ranks' keys shipped to those
  ranks and computed there, and the partial (O, LSE) pairs merged at home
  with the online-softmax rescale.

Shards are contiguous: rank g of W owns query and key blocks
[g*nb/W, (g+1)*nb/W) of every (batch, head); a rank holds q, k, v of its
blocks only ([B, H, count*block, D]) and the CSR rows of its own query blocks
(rows bh*count + i_local, entries GLOBAL key-block ids).  The plans come from
the C ABI's host planners (bsa_shard_plan_kv, bsa_shard_plan_partial) and are
reusable while the mask is unchanged.  Collectives are torch.distributed
all_to_all_single calls on int32 views (NCCL on GPUs); every block move, the
forward and the merge run in libbsa.so's kernels through :class:`DeviceOps`.
Each exchange lands in the receiving rank's own memory: no kernel reads
another GPU's memory.
"""

from __future__ import annotations

import ctypes
import dataclasses
from typing import List, Optional, Tuple

import numpy as np
import torch

from . import _binding as _b


class _Geom(ctypes.Structure):
    _fields_ = [("world", ctypes.c_int32), ("rank", ctypes.c_int32), ("n_blocks", ctypes.c_int32),
                ("BH", ctypes.c_int32)]


def _sigs():
    L = _b.lib()
    if getattr(L, "_shard_sigs", False):
        return L
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    PG = ctypes.POINTER(_Geom)
    L.bsa_shard_range.argtypes = [PG, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.bsa_shard_plan_kv.argtypes = [PG, P, P, P, P, P, P, i64, P, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.bsa_shard_plan_partial.argtypes = [PG, P, P, P, i32, P, P, P, P, P, i64, P, P]
    L.bsa_copy_blocks.argtypes = [P, P, P, P, i64, i32, i32, P]
    L.bsa_merge_partial_blocks.argtypes = [P, P, P, P, P, i64, i32, i32, P]
    L.bsa_convert_f32_bf16.argtypes = [P, P, i64, P]
    for f in ("bsa_shard_range", "bsa_shard_plan_kv", "bsa_shard_plan_partial", "bsa_copy_blocks",
              "bsa_merge_partial_blocks", "bsa_convert_f32_bf16"):
        getattr(L, f).restype = ctypes.c_int
    L._shard_sigs = True
    return L


def _np_ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def shard_range(world: int, rank: int, n_blocks: int, BH: int = 1) -> Tuple[int, int]:
    """(first block, block count) of `rank`'s shard."""
    g = _Geom(world, rank, n_blocks, BH)
    first, count = ctypes.c_int32(0), ctypes.c_int32(0)
    _b._check("bsa_shard_range", _sigs().bsa_shard_range(ctypes.byref(g), ctypes.byref(first), ctypes.byref(count)))
    return int(first.value), int(count.value)


# ---------------------------------------------------------------- device work
class DeviceOps:
    """The device work of the sharded forward, in libbsa.so's kernels."""

    def copy_blocks(self, src: torch.Tensor, dst: torch.Tensor, src_rows: np.ndarray, dst_rows: np.ndarray,
                    rows_per_block: int) -> None:
        """dst rows dst_rows[n] .. + rows_per_block = src rows src_rows[n] ..;
        src, dst are [rows, D] views of contiguous tensors."""
        n = len(src_rows)
        if n == 0:
            return
        dev = dst.device
        sr = torch.as_tensor(np.asarray(src_rows, np.int64), device=dev)
        dr = torch.as_tensor(np.asarray(dst_rows, np.int64), device=dev)
        row_bytes = dst.shape[-1] * dst.element_size()
        _b._check("bsa_copy_blocks", _sigs().bsa_copy_blocks(
            ctypes.c_void_p(src.data_ptr()), ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(sr.data_ptr()),
            ctypes.c_void_p(dr.data_ptr()), n, int(rows_per_block), int(row_bytes), _b._stream(None)))

    def forward_ex(self, q, k, v, row_ptr: np.ndarray, col_idx: np.ndarray, block: int, scale: float, causal: bool,
                   row_flags: Optional[np.ndarray], q_block_offset: int, out_f32: bool = False):
        dev = q.device
        rp = torch.as_tensor(np.asarray(row_ptr, np.int32), device=dev)
        ci = torch.as_tensor(np.asarray(col_idx if len(col_idx) else np.zeros(1), np.int32), device=dev)
        fl = None if row_flags is None else torch.as_tensor(np.asarray(row_flags, np.uint8), device=dev)
        return _b.forward_ex(q, k, v, rp, ci, block, scale=scale, causal=causal, row_flags=fl,
                             q_block_offset=q_block_offset,
                             out_dtype=torch.float32 if out_f32 else torch.bfloat16)

    def to_bf16(self, x: torch.Tensor) -> torch.Tensor:
        """fp32 -> bf16 (nearest even), same shape."""
        y = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
        _b._check("bsa_convert_f32_bf16", _sigs().bsa_convert_f32_bf16(
            ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), x.numel(), _b._stream(None)))
        return y

    def merge(self, o_acc: torch.Tensor, lse_acc: torch.Tensor, o_part: torch.Tensor, lse_part: torch.Tensor,
              dst_rows: np.ndarray, rows_per_block: int) -> None:
        """o_acc [rows, D] fp32, lse_acc [rows] updated with the compact fp32 parts."""
        n = len(dst_rows)
        if n == 0:
            return
        dr = torch.as_tensor(np.asarray(dst_rows, np.int64), device=o_acc.device)
        _b._check("bsa_merge_partial_blocks", _sigs().bsa_merge_partial_blocks(
            ctypes.c_void_p(o_acc.data_ptr()), ctypes.c_void_p(lse_acc.data_ptr()),
            ctypes.c_void_p(o_part.data_ptr()), ctypes.c_void_p(lse_part.data_ptr()),
            ctypes.c_void_p(dr.data_ptr()), n, int(rows_per_block), int(o_acc.shape[-1]), _b._stream(None)))


# ---------------------------------------------------------------- collectives
def _world(group):
    import torch.distributed as dist
    return dist.get_world_size(group), dist.get_rank(group)


def _a2a_counts(send: List[int], device, group) -> List[int]:
    """All-to-all of one int per peer."""
    import torch.distributed as dist
    s = torch.tensor(send, dtype=torch.int32, device=device)
    r = torch.empty_like(s)
    dist.all_to_all_single(r, s, group=group)
    return [int(x) for x in r.cpu()]


def _a2a(send: torch.Tensor, send_counts: List[int], recv_counts: List[int], unit: int, group) -> torch.Tensor:
    """All-to-all of a contiguous buffer of `unit`-int32 records (send is any
    dtype; it travels as int32 words and comes back in send's dtype)."""
    import torch.distributed as dist
    words = send.contiguous().view(torch.int32).reshape(-1)
    per = words.numel() // max(1, sum(send_counts)) if sum(send_counts) else unit
    assert sum(send_counts) == 0 or per == unit
    out = torch.empty(sum(recv_counts) * unit, dtype=torch.int32, device=send.device)
    dist.all_to_all_single(out, words, output_split_sizes=[c * unit for c in recv_counts],
                           input_split_sizes=[c * unit for c in send_counts], group=group)
    return out.view(send.dtype)


# ---------------------------------------------------------------- key/value exchange
@dataclasses.dataclass
class KVPlan:
    world: int
    rank: int
    n_blocks: int
    BH: int
    first: int
    count: int
    n_before: int
    n_after: int
    col_idx_ext: np.ndarray          # the rank's CSR entries in extended key blocks
    need_bh: np.ndarray              # remote blocks to fetch, grouped by owner
    need_j: np.ndarray
    need_pos: np.ndarray
    need_count_by_rank: List[int]

    @property
    def n_k_ext(self) -> int:
        return self.n_before + self.count + self.n_after


def plan_kv(world: int, rank: int, n_blocks: int, BH: int, row_ptr: np.ndarray, col_idx: np.ndarray) -> KVPlan:
    """Key/value exchange plan of this rank's CSR (host arrays)."""
    L = _sigs()
    g = _Geom(world, rank, n_blocks, BH)
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    ci = np.ascontiguousarray(col_idx if len(col_idx) else np.zeros(1, np.int32), dtype=np.int32)
    nnz = int(rp[-1])
    first, count = shard_range(world, rank, n_blocks, BH)
    ext = np.zeros(max(nnz, 1), np.int32)
    cap = max(nnz, 1)
    nbh, nj, npos = (np.zeros(cap, np.int32) for _ in range(3))
    cnt = np.zeros(world, np.int32)
    nbf, naf = ctypes.c_int32(0), ctypes.c_int32(0)
    _b._check("bsa_shard_plan_kv", L.bsa_shard_plan_kv(
        ctypes.byref(g), _np_ptr(rp), _np_ptr(ci), _np_ptr(ext), _np_ptr(nbh), _np_ptr(nj), _np_ptr(npos), cap,
        _np_ptr(cnt), ctypes.byref(nbf), ctypes.byref(naf)))
    n = int(cnt.sum())
    return KVPlan(world, rank, n_blocks, BH, first, count, int(nbf.value), int(naf.value), ext[:nnz],
                  nbh[:n].copy(), nj[:n].copy(), npos[:n].copy(), [int(x) for x in cnt])


def exchange_kv(k_local: torch.Tensor, v_local: torch.Tensor, plan: KVPlan, block: int, group=None,
                ops: Optional[DeviceOps] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """The sparse all-to-all: requests (head, key block) to each owner, then
    the blocks themselves, placed with the local shard into the extended key
    range [B, H, n_k_ext*block, D] in this rank's memory."""
    ops = ops or DeviceOps()
    world, rank = _world(group)
    assert (world, rank) == (plan.world, plan.rank)
    B, H, Nl, D = k_local.shape
    BH, cnt, first = B * H, plan.count, plan.first
    assert Nl == cnt * block and BH == plan.BH
    dev = k_local.device
    # 1. requests: how many blocks each peer wants from me, then which
    recv_counts = _a2a_counts(plan.need_count_by_rank, dev, group)
    req = torch.as_tensor(np.stack([plan.need_bh, plan.need_j], 1).reshape(-1).astype(np.int32), device=dev)
    got = _a2a(req, plan.need_count_by_rank, recv_counts, 2, group).cpu().numpy().reshape(-1, 2)
    # 2. the requested K and V blocks, gathered into one buffer [n, 2 (K, V), block, D]
    n_send = got.shape[0]
    send = torch.empty((n_send * 2 * block, D), dtype=k_local.dtype, device=dev)
    if n_send:
        src = (got[:, 0].astype(np.int64) * Nl + (got[:, 1].astype(np.int64) - first) * block)
        dst = np.arange(n_send, dtype=np.int64) * 2 * block
        ops.copy_blocks(k_local.reshape(-1, D), send, src, dst, block)
        ops.copy_blocks(v_local.reshape(-1, D), send, src, dst + block, block)
    unit = 2 * block * D * k_local.element_size() // 4
    recv = _a2a(send, recv_counts, plan.need_count_by_rank, unit, group).reshape(-1, D)
    # 3. the extended range: own shard in the middle, received blocks at their slots
    Ne = plan.n_k_ext * block
    k_ext = torch.zeros((B, H, Ne, D), dtype=k_local.dtype, device=dev)
    v_ext = torch.zeros_like(k_ext)
    own_src = (np.arange(BH, dtype=np.int64)[:, None] * Nl + np.arange(cnt, dtype=np.int64)[None, :] * block)
    own_dst = (np.arange(BH, dtype=np.int64)[:, None] * Ne
               + (plan.n_before + np.arange(cnt, dtype=np.int64))[None, :] * block)
    for loc, ext in ((k_local, k_ext), (v_local, v_ext)):
        ops.copy_blocks(loc.reshape(-1, D), ext.reshape(-1, D), own_src.reshape(-1), own_dst.reshape(-1), block)
    n_recv = len(plan.need_bh)
    if n_recv:
        src = np.arange(n_recv, dtype=np.int64) * 2 * block
        dst = plan.need_bh.astype(np.int64) * Ne + plan.need_pos.astype(np.int64) * block
        ops.copy_blocks(recv, k_ext.reshape(-1, D), src, dst, block)
        ops.copy_blocks(recv, v_ext.reshape(-1, D), src + block, dst, block)
    return k_ext, v_ext


def forward_kv_exchange(q_local: torch.Tensor, k_local: torch.Tensor, v_local: torch.Tensor, row_ptr, col_idx,
                        block: int, n_blocks: int, scale: Optional[float] = None, causal: bool = False,
                        row_flags: Optional[np.ndarray] = None, group=None, plan: Optional[KVPlan] = None,
                        ops: Optional[DeviceOps] = None):
    """Sequence-sharded forward by key/value exchange.  row_ptr / col_idx:
    this rank's CSR (host numpy or any tensor; entries are global key-block
    ids), n_blocks: blocks of the whole sequence.  Returns (O, LSE, plan) for
    the rank's query rows."""
    ops = ops or DeviceOps()
    world, rank = _world(group)
    B, H, Nl, D = q_local.shape
    rp = np.asarray(row_ptr.cpu() if torch.is_tensor(row_ptr) else row_ptr, np.int32)
    ci = np.asarray(col_idx.cpu() if torch.is_tensor(col_idx) else col_idx, np.int32)
    if plan is None:
        plan = plan_kv(world, rank, n_blocks, B * H, rp, ci)
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    k_ext, v_ext = exchange_kv(k_local, v_local, plan, block, group=group, ops=ops)
    o, lse = ops.forward_ex(q_local, k_ext, v_ext, rp, plan.col_idx_ext, block, scale, causal, row_flags,
                            plan.n_before)
    return o, lse, plan


# ---------------------------------------------------------------- partial outputs + merge
@dataclasses.dataclass
class PartialPlan:
    world: int
    rank: int
    count: int
    local_row_ptr: np.ndarray
    local_col_idx: np.ndarray
    guest_q: np.ndarray          # local CSR rows shipped out, grouped by peer
    guest_ptr: np.ndarray
    guest_col: np.ndarray        # their entries in the peer's numbering
    guest_rows_by_rank: List[int]
    guest_entries_by_rank: List[int]


def plan_partial(world: int, rank: int, n_blocks: int, BH: int, row_ptr: np.ndarray, col_idx: np.ndarray,
                 causal: bool, row_flags: Optional[np.ndarray] = None) -> PartialPlan:
    L = _sigs()
    g = _Geom(world, rank, n_blocks, BH)
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    ci = np.ascontiguousarray(col_idx if len(col_idx) else np.zeros(1, np.int32), dtype=np.int32)
    fl = None if row_flags is None else np.ascontiguousarray(row_flags, dtype=np.uint8)
    nnz = int(rp[-1])
    cap = max(nnz, 1)
    _, count = shard_range(world, rank, n_blocks, BH)
    lrp = np.zeros(BH * count + 1, np.int32)
    lci, gq, gcol = (np.zeros(cap, np.int32) for _ in range(3))
    gptr = np.zeros(cap + 1, np.int32)
    grows, gents = np.zeros(world, np.int32), np.zeros(world, np.int32)
    _b._check("bsa_shard_plan_partial", L.bsa_shard_plan_partial(
        ctypes.byref(g), _np_ptr(rp), _np_ptr(ci), _np_ptr(fl), int(bool(causal)), _np_ptr(lrp), _np_ptr(lci),
        _np_ptr(gq), _np_ptr(gptr), _np_ptr(gcol), cap, _np_ptr(grows), _np_ptr(gents)))
    ng = int(grows.sum())
    return PartialPlan(world, rank, count, lrp, lci[:int(lrp[-1])].copy(), gq[:ng].copy(), gptr[:ng + 1].copy(),
                       gcol[:int(gptr[ng])].copy(), [int(x) for x in grows], [int(x) for x in gents])


def guest_layout(hdr: np.ndarray, ent: np.ndarray, BH: int):
    """Where received guest rows go at their key owner.  hdr: [n, 2] (head,
    entry count) per guest query block in arrival order, ent: their entries
    (owner's key numbering) concatenated.  Guests of head bh take slots 0, 1,
    ... of that head in arrival order; every head gets gmax slots.  Returns
    (gmax, row_of [n] = the guest CSR row bh*gmax + slot of each arrival,
    row_ptr [BH*gmax + 1], col_idx) of the guest CSR; unused slots are empty
    rows."""
    n = hdr.shape[0]
    slot = np.zeros(n, np.int64)
    per_head = np.zeros(BH, np.int64)
    for x in range(n):
        slot[x] = per_head[hdr[x, 0]]
        per_head[hdr[x, 0]] += 1
    gmax = int(per_head.max()) if n else 0
    row_of = hdr[:, 0].astype(np.int64) * gmax + slot if n else np.zeros(0, np.int64)
    lens = np.zeros(BH * gmax, np.int64)
    lens[row_of] = hdr[:, 1] if n else 0
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ci = np.zeros(max(int(rp[-1]), 1), np.int32)
    starts = np.concatenate([[0], np.cumsum(hdr[:, 1] if n else [])]).astype(np.int64)
    for x in range(n):
        ci[rp[row_of[x]]:rp[row_of[x]] + hdr[x, 1]] = ent[starts[x]:starts[x + 1]]
    return gmax, row_of, rp, ci


def forward_partial_merge(q_local: torch.Tensor, k_local: torch.Tensor, v_local: torch.Tensor, row_ptr, col_idx,
                          block: int, n_blocks: int, scale: Optional[float] = None, causal: bool = False,
                          row_flags: Optional[np.ndarray] = None, group=None, plan: Optional[PartialPlan] = None,
                          ops: Optional[DeviceOps] = None):
    """Sequence-sharded forward by local attention plus a merge of partial
    outputs.  Arguments as forward_kv_exchange.  Returns (O, LSE, plan)."""
    ops = ops or DeviceOps()
    world, rank = _world(group)
    B, H, Nl, D = q_local.shape
    BH = B * H
    dev = q_local.device
    rp = np.asarray(row_ptr.cpu() if torch.is_tensor(row_ptr) else row_ptr, np.int32)
    ci = np.asarray(col_idx.cpu() if torch.is_tensor(col_idx) else col_idx, np.int32)
    if plan is None:
        plan = plan_partial(world, rank, n_blocks, BH, rp, ci, causal, row_flags)
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    cnt = plan.count
    # 1. the local part (fp32 O: partial results are merged before rounding)
    o, lse = ops.forward_ex(q_local, k_local, v_local, plan.local_row_ptr, plan.local_col_idx, block, scale, causal,
                            row_flags, 0, out_f32=True)
    # 2. guest rows to their key owners: (head, entry count) and the entries
    send_rows, send_ents = plan.guest_rows_by_rank, plan.guest_entries_by_rank
    recv_rows = _a2a_counts(send_rows, dev, group)
    recv_ents = _a2a_counts(send_ents, dev, group)
    gq = plan.guest_q.astype(np.int64)
    glen = np.diff(plan.guest_ptr).astype(np.int32)
    hdr = torch.as_tensor(np.stack([(gq // cnt).astype(np.int32), glen], 1).reshape(-1), device=dev)
    hdr_in = _a2a(hdr, send_rows, recv_rows, 2, group).cpu().numpy().reshape(-1, 2)
    ent_in = _a2a(torch.as_tensor(plan.guest_col.astype(np.int32), device=dev), send_ents, recv_ents, 1,
                  group).cpu().numpy()
    # 3. their query blocks
    n_out = len(gq)
    qsend = torch.empty((n_out * block, D), dtype=q_local.dtype, device=dev)
    src_q = (gq // cnt) * Nl + (gq % cnt) * block
    ops.copy_blocks(q_local.reshape(-1, D), qsend, src_q, np.arange(n_out, dtype=np.int64) * block, block)
    unit = block * D * q_local.element_size() // 4
    qrecv = _a2a(qsend, send_rows, recv_rows, unit, group).reshape(-1, D)
    # 4. the guests' attention on this rank's keys (no causal cut: the plan
    #    sent only blocks wholly before each causal row)
    n_in = hdr_in.shape[0]
    gmax, row_of, grp, gci = guest_layout(hdr_in, ent_in, BH)
    partial_out = []
    if gmax:
        qg = torch.zeros((B, H, gmax * block, D), dtype=q_local.dtype, device=dev)
        ops.copy_blocks(qrecv, qg.reshape(-1, D), np.arange(n_in, dtype=np.int64) * block, row_of * block, block)
        og, lg = ops.forward_ex(qg, k_local, v_local, grp, gci, block, scale, False, None, 0, out_f32=True)
        # results back in arrival order
        res_o = torch.empty((n_in * block, D), dtype=og.dtype, device=dev)
        res_l = torch.empty((n_in, block), dtype=lg.dtype, device=dev)
        ops.copy_blocks(og.reshape(-1, D), res_o, row_of * block, np.arange(n_in, dtype=np.int64) * block, block)
        # LSE: one row of `block` values per query block
        ops.copy_blocks(lg.reshape(-1, block), res_l, row_of, np.arange(n_in, dtype=np.int64), 1)
        partial_out = [res_o, res_l]
    else:
        partial_out = [torch.empty((0, D), dtype=o.dtype, device=dev),
                       torch.empty((0, block), dtype=lse.dtype, device=dev)]
    # 5. the partial results go home and are merged, one peer at a time
    unit_o = block * D * o.element_size() // 4
    unit_l = block * lse.element_size() // 4
    back_o = _a2a(partial_out[0], recv_rows, send_rows, unit_o, group).reshape(-1, D)
    back_l = _a2a(partial_out[1], recv_rows, send_rows, unit_l, group).reshape(-1)
    o2, l2 = o.reshape(-1, D), lse.reshape(-1)
    off = 0
    for p in range(world):
        n = send_rows[p]
        if n == 0:
            continue
        rows = gq[off:off + n]
        dst = (rows // cnt) * Nl + (rows % cnt) * block
        ops.merge(o2, l2, back_o[off * block:(off + n) * block], back_l[off * block:(off + n) * block], dst, block)
        off += n
    return ops.to_bf16(o), lse, plan
