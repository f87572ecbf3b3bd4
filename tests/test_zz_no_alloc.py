"""bsa_forward_noalloc -- the forward pass for callers that cannot let the
library allocate device memory (serving loops that must not hit the
device-wide synchronisation of cudaMalloc / cudaFree, applications that own
every byte of device memory through their own pools).  It takes its schedule
scratch from a fixed array inside libbsa.so.

Checked through the C ABI against bsa_forward on the same inputs, on two
calls in a row with different problems (the shared array keeps the previous
call's contents, so the second call must not depend on them), within the
tolerances of the parity tests.  Collected last on purpose; it also passes
when run alone in a fresh process.
"""

import ctypes

import pytest
import torch

import bsa_inputs
from parity import TOL_LSE, TOL_MAX_O, TOL_MEAN_O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_flashattention_bsa_gb300 import build
    build.build()
    import block_sparse_flashattention_bsa_gb300 as m
    L = m.lib()
    P = ctypes.c_void_p
    from block_sparse_flashattention_bsa_gb300._binding import _Shape
    L.bsa_forward_noalloc.argtypes = [ctypes.POINTER(_Shape), P, P, P, P, P, P, P, ctypes.c_float, ctypes.c_int32, P]
    L.bsa_forward_noalloc.restype = ctypes.c_int
    return m


def _case(bsa, w):
    d = bsa_inputs.make_qkv(w)
    q, k, v = (d[x].cuda() for x in "qkv")
    pat = bsa.Pattern(w.n_blocks, w.window_left, w.window_right, w.causal, w.global_blocks,
                      w.global_rows_attend_all)
    rp, ci = bsa.build_mask_csr(pat, w.B, w.H, device=q.device)
    return q, k, v, rp, ci


def _noalloc(bsa, w, q, k, v, rp, ci):
    from block_sparse_flashattention_bsa_gb300._binding import _Shape
    sh = _Shape(w.B, w.H, w.N, w.D, w.block)
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=q.device)
    st = bsa.lib().bsa_forward_noalloc(
        ctypes.byref(sh), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(rp.data_ptr()), ctypes.c_void_p(ci.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), ctypes.c_float(w.scale),
        int(w.causal), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, bsa.lib().bsa_status_string(st)
    return o, lse


def test_noalloc_matches_forward_two_calls_in_a_row(bsa):
    w1 = bsa_inputs.small_workload(bsa_inputs.workload("window_global_64k"), H=4, N=128 * 96)
    w2 = bsa_inputs.small_workload(bsa_inputs.workload("tiny_window_global"), H=3)
    for w in (w1, w2):
        q, k, v, rp, ci = _case(bsa, w)
        o_ref, l_ref = bsa.forward(q, k, v, rp, ci, w.block, scale=w.scale, causal=w.causal)
        o, lse = _noalloc(bsa, w, q, k, v, rp, ci)
        torch.cuda.synchronize()
        d_o = (o.double() - o_ref.double()).abs()
        assert float(d_o.max()) <= TOL_MAX_O and float(d_o.mean()) <= TOL_MEAN_O
        assert float((lse.double() - l_ref.double()).abs().max()) <= TOL_LSE


def test_noalloc_block64_matches_oracle(bsa):
    """64-token blocks run the padded form here (no pairing workspace): all rows
    against the fp64 oracle."""
    import numpy as np

    import oracle
    w = bsa_inputs.small_workload(bsa_inputs.workload("tiny_window_global"), H=3)
    q, k, v, rp, ci = _case(bsa, w)
    o, lse = _noalloc(bsa, w, q, k, v, rp, ci)
    torch.cuda.synchronize()
    d = bsa_inputs.make_qkv(w)
    rp1, ci1 = oracle.Pattern.from_workload(w).csr()
    rp_ref, ci_ref = oracle.replicate_csr(rp1, ci1, w.B * w.H)
    np.testing.assert_array_equal(rp.cpu().numpy(), rp_ref)
    np.testing.assert_array_equal(ci.cpu().numpy(), ci_ref)
    O_ref, L_ref = oracle.attention_rows(bsa_inputs.bf16_bits(d["q"]), bsa_inputs.bf16_bits(d["k"]),
                                         bsa_inputs.bf16_bits(d["v"]), rp_ref, ci_ref,
                                         w.block, w.scale, w.causal)
    d_o = np.abs(o.reshape(-1, w.D).double().cpu().numpy() - O_ref)
    assert d_o.max() <= TOL_MAX_O and d_o.mean() <= TOL_MEAN_O
    assert np.abs(lse.reshape(-1).double().cpu().numpy() - L_ref).max() <= TOL_LSE


def test_noalloc_rejects_too_many_rows(bsa):
    from block_sparse_flashattention_bsa_gb300._binding import _Shape
    fake = ctypes.c_void_p(1 << 20)  # rejected on the host before any device access
    sh = _Shape(1, 64, 128 * 8192, 128, 128)  # 64 * 8192 rows > BSA_NOALLOC_MAX_ROWS
    st = bsa.lib().bsa_forward_noalloc(ctypes.byref(sh), fake, fake, fake, fake, fake, fake, fake,
                                       ctypes.c_float(0.1), 0, None)
    assert st == -3  # BSA_ERR_CAPACITY
