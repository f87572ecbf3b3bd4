"""GPU parity of FP8 scores with one scale per (head, block).

bsa_quantize_e4m3_blocks must give the oracle's codes and descale factors
bit for bit (quantize_e4m3_blocks: amax per block, inv = fp32(448 / amax),
codes = e4m3(fp32(x * inv)), descale = fp32(amax / 448)).  The forward on
those codes (bsa_forward_fp8_blocks) is checked against the oracle's exact
fp64 attention of the decoded codes times their block factors
(attention_rows_fp8_blocks) at the bf16 forward's tolerances: both sides see
the same quantised inputs, so the quantisation itself is not part of the
comparison.  Cases: window masks (causal and not), random unsorted lists
with empty rows, the paired block-64 form on the clustered top-k inputs,
blocks with very different magnitudes, and sampled full-size rows of the
16K window workload.
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


def _quantize_both(x_cpu, block):
    import block_sparse_flashattention_bsa_gb300 as bsa
    BH = x_cpu.shape[0] * x_cpu.shape[1]
    codes_ref, desc_ref = oracle.quantize_e4m3_blocks(bits(x_cpu).reshape(BH, x_cpu.shape[2], x_cpu.shape[3]), block)
    codes, desc = bsa.quantize_e4m3_blocks(x_cpu.cuda(), block)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(codes.cpu().numpy().reshape(codes_ref.shape), codes_ref)
    np.testing.assert_array_equal(desc.cpu().numpy().reshape(desc_ref.shape), desc_ref)
    return codes, desc, codes_ref, desc_ref


@pytest.mark.parametrize("block,D", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_block_quantization_bit_exact(block, D):
    g = torch.Generator().manual_seed(block + D)
    nb = 12
    x = (torch.randn(2, 3, nb * block, D, generator=g) * 2).to(torch.bfloat16)
    x[0, 1, 3 * block:4 * block] = 0                       # an all-zero block
    x[1, 2, 5 * block:6 * block] *= 300                    # a peaked block
    x[1, 0, 7 * block:8 * block] *= 1e-3                   # a tiny one
    _quantize_both(x, block)


def _fp8_blocks_case(w, csr=None, causal=None, rows=None, data=None):
    import block_sparse_flashattention_bsa_gb300 as bsa
    d = bsa_inputs.make_qkv(w) if data is None else data
    BH = w.B * w.H
    q8, qd, q8r, qdr = _quantize_both(d["q"], w.block)
    k8, kd, k8r, kdr = _quantize_both(d["k"], w.block)
    if csr is None:
        rp, ci = oracle_csr(w, d["q"], d["k"])
    else:
        rp, ci = csr
    causal = w.causal if causal is None else causal
    dev = torch.device("cuda")
    o, lse = bsa.forward_fp8_blocks(q8, k8, d["v"].to(dev), qd.reshape(-1), kd.reshape(-1),
                                    torch.as_tensor(rp, device=dev),
                                    torch.as_tensor(ci if len(ci) else np.zeros(1, np.int32), device=dev),
                                    w.block, scale=w.scale, causal=causal)
    torch.cuda.synchronize()
    err = bsa.device_error()
    if rows is None:
        rows = np.arange(BH * w.N, dtype=np.int64)
    O, L = oracle.attention_rows_fp8_blocks(q8r, k8r, bits(d["v"]).reshape(BH, w.N, w.D), qdr, kdr, rp, ci,
                                            w.block, w.scale, causal, rows=rows)
    return compare(o, lse, O, L, rows, w.D), err


@pytest.mark.parametrize("causal", [True, False])
def test_fp8_blocks_window_all_rows(causal):
    w = bsa_inputs.small_workload(W["window_16k"], H=2, N=128 * 24, seed=161)
    stats, err = _fp8_blocks_case(w, causal=causal)
    assert err == 0
    assert_close(stats, "fp8 blocks window causal=%s" % causal)


def test_fp8_blocks_random_lists_all_rows():
    rng = np.random.default_rng(171)
    w = bsa_inputs.small_workload(W["window_16k"], B=1, H=3, N=128 * 20, seed=172)
    nb = w.n_blocks
    lists = [list(rng.choice(nb, size=int(rng.integers(0, nb + 1)), replace=False)) for _ in range(w.B * w.H * nb)]
    rp = np.concatenate([[0], np.cumsum([len(l) for l in lists])]).astype(np.int32)
    ci = np.array([j for l in lists for j in l], dtype=np.int32)
    for causal in (False, True):
        stats, err = _fp8_blocks_case(w, csr=(rp, ci), causal=causal)
        assert err == 0
        assert_close(stats, "fp8 blocks random causal=%s" % causal)


def test_fp8_blocks_paired_block64_all_rows():
    w = bsa_inputs.small_workload(W["content_topk"], B=1, H=2, N=64 * 96, seed=181)
    stats, err = _fp8_blocks_case(w)
    assert err == 0
    assert_close(stats, "fp8 blocks content top-k block 64")


def test_fp8_blocks_uneven_magnitudes():
    """Blocks whose magnitudes differ (factors e^N(0, 0.7) per block, up to
    about 10x apart): per-block factors differ too, and the per-step logit
    scale must follow them.  (Much wider spreads make logits of hundreds,
    where the fp32 accumulation of the e4m3 tensor-core products alone moves
    LSE by ~1e-3.)"""
    w = bsa_inputs.small_workload(W["window_global_64k"], H=2, N=128 * 32, seed=191)
    d = bsa_inputs.make_qkv(w)
    g = torch.Generator().manual_seed(5)
    f = torch.exp(torch.randn(w.B, w.H, w.n_blocks, 1, 1, generator=g) * 0.7)
    for x in ("q", "k"):
        d[x] = (d[x].float().reshape(w.B, w.H, w.n_blocks, w.block, w.D) * f).reshape(d[x].shape).to(torch.bfloat16)
    # peaked rows give O close to single V rows: V at half scale keeps |O| < 4,
    # where bf16's half-ulp (0.0078) leaves room inside max |dO| <= 1e-2
    d["v"] = (d["v"].float() * 0.5).to(torch.bfloat16)
    stats, err = _fp8_blocks_case(w, data=d)
    assert err == 0
    assert_close(stats, "fp8 blocks uneven magnitudes")


def test_fp8_blocks_window_16k_sampled():
    w = W["window_16k"]
    rows = bsa_inputs.sample_rows(w, n_random_blocks=6).numpy()
    stats, err = _fp8_blocks_case(w, rows=rows)
    assert err == 0
    assert_close(stats, "fp8 blocks window_16k sampled")
