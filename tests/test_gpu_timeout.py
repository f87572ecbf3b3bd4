"""Hang detection on the GPU, without a hang.

Every wait inside the forward kernel is bounded by the library's wait limit.
The test hook bsa_debug_stall_next_forward makes the next forward's work
distributor stop after a few work items without publishing the end of the
work -- a flag that nothing will ever set -- so every other role of each CTA
waits until the limit runs out.  The launch must then leave through its
normal exit (in-flight copies and MMAs drained, tensor memory freed), report
bit 1 (timeout) in the device error word, and leave the context usable: the
next forward on the same inputs matches the fp64 oracle.

Nothing here faults or hangs a GPU: the stalled waits end after 5 ms.
"""

import numpy as np
import pytest
import torch

import bsa_inputs
import oracle
from parity import assert_close, bits, compare, oracle_csr

pytestmark = pytest.mark.gpu

W = {w.name: w for w in bsa_inputs.WORKLOADS}
ERR_TIMEOUT = 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_flashattention_bsa_gb300 import build
    build.build()
    import block_sparse_flashattention_bsa_gb300 as bsa
    bsa.device_error()
    yield
    bsa.set_wait_limit(0)
    bsa.debug_stall_next_forward(-1)


def _inputs(w):
    import block_sparse_flashattention_bsa_gb300 as bsa
    d = bsa_inputs.make_qkv(w)
    dev = torch.device("cuda")
    q, k, v = (d[x].to(dev) for x in "qkv")
    pat = bsa.Pattern(w.n_blocks, w.window_left, w.window_right, w.causal, w.global_blocks,
                      w.global_rows_attend_all)
    rp, ci = bsa.build_mask_csr(pat, w.B, w.H, device=dev)
    return d, q, k, v, rp, ci


def _check_against_oracle(w, d, o, lse):
    rp_ref, ci_ref = oracle_csr(w)
    rows = np.arange(w.B * w.H * w.N, dtype=np.int64)
    O_ref, L_ref = oracle.attention_rows(bits(d["q"]), bits(d["k"]), bits(d["v"]), rp_ref, ci_ref, w.block,
                                         w.scale, w.causal, rows=rows)
    assert_close(compare(o, lse, O_ref, L_ref, rows, w.D), w.name)


# Each CTA's distributor stops before its (stall + 1)-th claim, so a stall of
# 1 stalls every CTA that got any work (launches here give a CTA one or two
# items), and 0 stalls every CTA before its first claim.
@pytest.mark.parametrize("name,kw,stall", [
    ("window_16k", dict(H=4, N=128 * 64), 1),          # block 128, rows of 5 blocks
    ("window_global_64k", dict(H=2, N=128 * 96), 0),   # nothing handed out at all
    ("tiny_window_global", dict(H=8, N=64 * 64), 1),   # block 64: the paired form
])
def test_stalled_forward_times_out_and_context_survives(name, kw, stall):
    import block_sparse_flashattention_bsa_gb300 as bsa
    w = bsa_inputs.small_workload(W[name], **kw)
    d, q, k, v, rp, ci = _inputs(w)
    bsa.set_wait_limit(5_000_000)  # 5 ms
    bsa.debug_stall_next_forward(stall)
    o, lse = bsa.forward(q, k, v, rp, ci, w.block, scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    assert bsa.device_error() == ERR_TIMEOUT
    # the hook is one-shot; the default limit is back for the rerun
    bsa.set_wait_limit(0)
    o, lse = bsa.forward(q, k, v, rp, ci, w.block, scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    assert bsa.device_error() == 0
    _check_against_oracle(w, d, o, lse)


def test_short_limit_without_stall_changes_nothing():
    """A 1 ms limit is far above any real wait of a small launch: no timeout,
    same results as the oracle."""
    import block_sparse_flashattention_bsa_gb300 as bsa
    w = bsa_inputs.small_workload(W["long_window_128k"], H=2, N=128 * 48)
    d, q, k, v, rp, ci = _inputs(w)
    bsa.set_wait_limit(1_000_000)
    try:
        o, lse = bsa.forward(q, k, v, rp, ci, w.block, scale=w.scale, causal=w.causal)
        torch.cuda.synchronize()
    finally:
        bsa.set_wait_limit(0)
    assert bsa.device_error() == 0
    _check_against_oracle(w, d, o, lse)
