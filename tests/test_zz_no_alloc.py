"""bsa_forward_noalloc -- the forward pass for callers that cannot let the
library allocate device memory (serving loops that must not hit the
device-wide synchronisation of cudaMalloc / cudaFree, applications that own
every byte of device memory through their own pools).  It takes its schedule
scratch from a fixed array inside libbsa.so.

Checked through the C ABI against bsa_forward on the same inputs, on two
calls in a row with different problems (the shared array keeps the previous
call's contents, so the second call must not depend on them), within the
tolerances of the parity tests; both block sizes against the fp64 oracle;
its device-side errors read through bsa_device_error; and the device's free
memory unchanged across a call on a larger problem than any before.
Collected last on purpose; it also passes when run alone in a fresh process.
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


def _oracle_all_rows(w, d, rp, ci, o, lse):
    import numpy as np

    import oracle
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


def test_noalloc_block128_matches_oracle(bsa):
    """The 128-token-block instance against the fp64 oracle, every row."""
    w = bsa_inputs.small_workload(bsa_inputs.workload("window_global_64k"), H=2, N=128 * 80)
    q, k, v, rp, ci = _case(bsa, w)
    o, lse = _noalloc(bsa, w, q, k, v, rp, ci)
    torch.cuda.synchronize()
    _oracle_all_rows(w, bsa_inputs.make_qkv(w), rp, ci, o, lse)


def test_noalloc_errors_reach_device_error(bsa):
    """A skipped out-of-range col_idx entry is reported by bsa_device_error
    (the error word lives in the fixed array) and the word is cleared by the
    read; the valid entries still give the oracle's result."""
    import numpy as np

    import oracle
    w = bsa_inputs.Workload("oob", 1, 2, 128 * 6, 128, 128, seed=3)
    nb = w.n_blocks
    rp_good, ci_good = oracle.replicate_csr(*oracle.Pattern(nb, 1, 1).csr(), w.B * w.H)
    rp_bad, ci_bad = [0], []
    for r in range(len(rp_good) - 1):
        ci_bad += [nb + 5] + ci_good[rp_good[r]:rp_good[r + 1]].tolist()
        rp_bad.append(len(ci_bad))
    d = bsa_inputs.make_qkv(w)
    q, k, v = (d[x].cuda() for x in "qkv")
    rp_t = torch.tensor(rp_bad, dtype=torch.int32, device=q.device)
    ci_t = torch.tensor(ci_bad, dtype=torch.int32, device=q.device)
    bsa.device_error()  # start clean
    o, lse = _noalloc(bsa, w, q, k, v, rp_t, ci_t)
    assert bsa.device_error() & 2
    assert bsa.device_error() == 0
    O_ref, L_ref = oracle.attention_rows(bsa_inputs.bf16_bits(d["q"]), bsa_inputs.bf16_bits(d["k"]),
                                         bsa_inputs.bf16_bits(d["v"]), rp_good, ci_good, w.block, w.scale, False)
    assert np.abs(o.reshape(-1, w.D).double().cpu().numpy() - O_ref).max() <= TOL_MAX_O
    assert np.abs(lse.reshape(-1).double().cpu().numpy() - L_ref).max() <= TOL_LSE


def test_noalloc_call_leaves_device_memory_unchanged(bsa):
    """After one warm-up call (which loads the kernels and looks up the
    array), a call on a larger problem than any before changes the device's
    free memory by nothing: the library allocated no device memory for it."""
    w_small = bsa_inputs.small_workload(bsa_inputs.workload("window_16k"), H=2, N=128 * 16)
    w_big = bsa_inputs.small_workload(bsa_inputs.workload("window_16k"), H=8, N=128 * 256)
    small = _case(bsa, w_small)
    big = _case(bsa, w_big)
    o_s = torch.empty_like(small[0])
    l_s = torch.empty(small[0].shape[:3], dtype=torch.float32, device=small[0].device)
    o_b = torch.empty_like(big[0])
    l_b = torch.empty(big[0].shape[:3], dtype=torch.float32, device=big[0].device)
    bsa.forward_noalloc(*small, w_small.block, scale=w_small.scale, causal=w_small.causal, out=o_s, lse=l_s)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    bsa.forward_noalloc(*big, w_big.block, scale=w_big.scale, causal=w_big.causal, out=o_b, lse=l_b)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert bsa.device_error() == 0


def test_noalloc_rejects_too_many_rows(bsa):
    from block_sparse_flashattention_bsa_gb300._binding import _Shape
    fake = ctypes.c_void_p(1 << 20)  # rejected on the host before any device access
    sh = _Shape(1, 64, 128 * 8192, 128, 128)  # 64 * 8192 rows > BSA_NOALLOC_MAX_ROWS
    st = bsa.lib().bsa_forward_noalloc(ctypes.byref(sh), fake, fake, fake, fake, fake, fake, fake,
                                       ctypes.c_float(0.1), 0, None)
    assert st == -3  # BSA_ERR_CAPACITY
