"""GPU parity of the FP8-score path (e4m3 Q and K, "Flash MSA Sparse
Attention Kernels Explained", section "The Future of Attention Kernels").

* bsa_quantize_e4m3: bit-exact against the oracle's codec (round to nearest
  even on the fp32 product, saturation, signed zeros, ties), at full size;
* bsa_forward_fp8: against the oracle's exact attention on the decoded e4m3
  Q and K (inputs quantised by the oracle, never by the CUDA path), with the
  bf16 path's tolerances -- both sides see the same quantised inputs, so only
  the kernel's own roundings differ -- every row at small sizes (block 128,
  and block 64 in the paired form) and sampled rows at the full window_16k
  size.
"""

import numpy as np
import pytest
import torch

import bsa_inputs
import oracle
from parity import assert_close, bits, compare, oracle_csr

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


def _codes_equal(got: torch.Tensor, want: np.ndarray):
    g = got.cpu().numpy().reshape(-1)
    bad = np.nonzero(g != want.reshape(-1))[0]
    assert bad.size == 0, "%d codes differ, first at %d: %#x vs %#x" % (bad.size, bad[0], g[bad[0]],
                                                                        want.reshape(-1)[bad[0]])


def test_quantize_bit_exact_edge_values():
    import block_sparse_flashattention_bsa_gb300 as bsa
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (np.unique(vals)[:-1] + np.unique(vals)[1:]) / 2          # exact ties, exact in bf16
    x = np.concatenate([mids, -mids, vals, -vals, [0.0, -0.0, 449.0, 500.0, 1e4, -1e4, 3e38, -3e38,
                                                    1e-30, -1e-30, 2.0 ** -10, -(2.0 ** -10)]])
    x = np.concatenate([x, np.zeros((-len(x)) % 16)]).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    for inv in (1.0, 0.5, 3.0, 1.0 / 3.0):
        got = bsa.quantize_e4m3(xb.cuda(), inv)
        _codes_equal(got, oracle.quantize_e4m3(bits(xb), inv))


def test_quantize_bit_exact_full_size():
    import block_sparse_flashattention_bsa_gb300 as bsa
    w = W["window_16k"]
    d = bsa_inputs.make_qkv(w)
    q = d["q"]
    amax = float(q.abs().max())
    inv = 448.0 / amax
    got = bsa.quantize_e4m3(q.cuda(), inv)
    _codes_equal(got, oracle.quantize_e4m3(bits(q), inv))
    # scaled so a share of the products saturates and a share lands in the subnormals
    for inv2 in (448.0 / (0.25 * amax), 2.0 ** -6):
        got = bsa.quantize_e4m3(q[:, :2].contiguous().cuda(), inv2)
        _codes_equal(got, oracle.quantize_e4m3(bits(q[:, :2].contiguous()), inv2))


def _fp8_case(w, rows=None, csr=None, causal=None):
    """Q, K quantised by the oracle; the forward on the GPU; the oracle's
    attention on the same codes."""
    import block_sparse_flashattention_bsa_gb300 as bsa
    d = bsa_inputs.make_qkv(w)
    q, k, v = d["q"], d["k"], d["v"]
    inv_q = 448.0 / float(q.abs().max())
    inv_k = 448.0 / float(k.abs().max())
    q8 = oracle.quantize_e4m3(bits(q), inv_q).reshape(q.shape)
    k8 = oracle.quantize_e4m3(bits(k), inv_k).reshape(k.shape)
    if csr is None:
        csr = oracle_csr(w, q, k)
    rp, ci = csr
    causal = w.causal if causal is None else causal
    dev = torch.device("cuda")
    rp_d = torch.as_tensor(rp, dtype=torch.int32, device=dev)
    ci_d = torch.as_tensor(ci if len(ci) else np.zeros(1, np.int32), dtype=torch.int32, device=dev)
    o, lse = bsa.forward_fp8(torch.from_numpy(q8).to(dev), torch.from_numpy(k8).to(dev), v.to(dev), rp_d, ci_d,
                             w.block, 1.0 / inv_q, 1.0 / inv_k, scale=w.scale, causal=causal)
    torch.cuda.synchronize()
    err = bsa.device_error()
    if rows is None:
        rows = np.arange(w.B * w.H * w.N, dtype=np.int64)
    O_ref, L_ref = oracle.attention_rows_fp8(q8, k8, bits(v), rp, ci, w.block, 1.0 / inv_q, 1.0 / inv_k,
                                             w.scale, causal, rows=rows)
    return compare(o, lse, O_ref, L_ref, rows, w.D), err


@pytest.mark.parametrize("causal", [True, False])
def test_fp8_forward_window_all_rows(causal):
    w = bsa_inputs.small_workload(W["window_16k"], H=2, N=128 * 24, seed=61)
    stats, err = _fp8_case(w, causal=causal)
    assert err == 0
    assert_close(stats, "fp8 window causal=%s" % causal)


def test_fp8_forward_random_lists_all_rows():
    rng = np.random.default_rng(71)
    w = bsa_inputs.small_workload(W["window_16k"], B=1, H=3, N=128 * 20, seed=72)
    nb = w.N // w.block
    lists = [sorted(rng.choice(nb, size=int(rng.integers(0, nb + 1)), replace=False).tolist())
             for _ in range(w.B * w.H * nb)]
    rp = np.concatenate([[0], np.cumsum([len(l) for l in lists])]).astype(np.int32)
    ci = np.array([j for l in lists for j in l], dtype=np.int32)
    for causal in (False, True):
        stats, err = _fp8_case(w, csr=(rp, ci), causal=causal)
        assert err == 0
        assert_close(stats, "fp8 random causal=%s" % causal)


def test_fp8_forward_block64_paired_all_rows():
    w = bsa_inputs.small_workload(W["content_topk"], B=1, H=2, N=64 * 96, seed=81)
    stats, err = _fp8_case(w)
    assert err == 0
    assert_close(stats, "fp8 content top-k block 64")


def test_fp8_forward_window_16k_sampled():
    w = W["window_16k"]
    rows = bsa_inputs.sample_rows(w).numpy()
    stats, err = _fp8_case(w, rows=rows)
    assert err == 0
    assert_close(stats, "fp8 window_16k sampled")
