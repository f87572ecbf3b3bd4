"""Pins of the oracle's e4m3 codec and of its FP8-score attention.

FP8 scores ("Flash MSA Sparse Attention Kernels Explained", section "The
Future of Attention Kernels") take Q and K as OCP E4M3 codes.  The codec is
pinned to values the OCP 8-bit floating point format fixes (largest finite
448, smallest normal 2^-6, smallest subnormal 2^-9, NaN at S.1111.111), to
PyTorch's float8_e4m3fn conversion (a library routine, compared inside its
non-saturating range), and to round-trip and tie properties.  The attention
is pinned to the brute-force full-mask oracle on the decoded inputs and to
the invariance that only the product of the descale factors matters.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import brute


def test_decode_landmarks():
    d = oracle.e4m3_decode(np.array([0x7E, 0x08, 0x01, 0x38, 0x30, 0x77, 0x3F, 0x07, 0x00, 0x80, 0xC0, 0xFE]))
    want = [448.0, 2.0 ** -6, 2.0 ** -9, 1.0, 0.5, 240.0, 1.875, 7 * 2.0 ** -9, 0.0, -0.0, -2.0, -448.0]
    assert list(d) == want
    assert np.signbit(d[9]) and not np.signbit(d[8])
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF]))).all()
    # no infinities: every other code is finite
    codes = np.arange(256, dtype=np.uint8)
    fin = np.isfinite(oracle.e4m3_decode(codes))
    assert fin.sum() == 254


def test_decode_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    d = oracle.e4m3_decode(codes)
    t = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(d), np.isnan(t))
    ok = ~np.isnan(d)
    assert np.array_equal(d[ok], t[ok]) and np.array_equal(np.signbit(d[ok]), np.signbit(t[ok]))


def _midpoints():
    v = np.unique(oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)))  # 0 .. 448, ascending
    mid = (v[:-1] + v[1:]) / 2
    return np.concatenate([mid, -mid]).astype(np.float32)


def test_encode_matches_torch_float8():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(100000) * s for s in (1e-4, 1e-3, 1e-2, 0.1, 1.0, 10.0, 100.0)])
    x = np.concatenate([x.astype(np.float32), _midpoints(), np.float32([0.0, -0.0, 1e-30, -1e-30])])
    x = x[np.abs(x) < 464]  # beyond, torch returns NaN where the format saturates
    a = oracle.e4m3_encode(x)
    b = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(a, b)


def test_encode_ties_go_to_even_code():
    mid = _midpoints()
    c = oracle.e4m3_encode(mid)
    assert np.all(c & 1 == 0)
    # and every midpoint lands on one of its two neighbours
    lo = oracle.e4m3_encode(np.nextafter(mid, np.float32(0)))
    hi = oracle.e4m3_encode(np.nextafter(mid, np.float32(np.inf) * np.sign(mid)))
    assert np.all((c == lo) | (c == hi)) and np.all(lo != hi)


def test_encode_saturates_and_keeps_sign():
    x = np.float32([448.0, 449.0, 463.9, 464.0, 1e6, np.inf, -500.0, -np.inf, -0.0, -1e-12])
    assert list(oracle.e4m3_encode(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x80, 0x80]
    assert oracle.e4m3_encode(np.float32([np.nan]))[0] & 0x7F == 0x7F


def test_round_trip_every_finite_code():
    codes = np.arange(256, dtype=np.uint8)
    d = oracle.e4m3_decode(codes)
    ok = ~np.isnan(d)
    assert np.array_equal(oracle.e4m3_encode(d[ok].astype(np.float32)), codes[ok])


def test_quantize_multiplies_by_inv_scale():
    rng = np.random.default_rng(3)
    x = torch.randn(4096).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    xf = x.float().numpy()
    assert np.array_equal(oracle.quantize_e4m3(bits, 1.0), oracle.e4m3_encode(xf))
    for k in (-3, 2, 5):  # powers of two: the product is exact
        assert np.array_equal(oracle.quantize_e4m3(bits, 2.0 ** k), oracle.e4m3_encode(xf * np.float32(2.0 ** k)))
    # a product that rounds in fp32 before the e4m3 rounding
    s = np.float32(1.0 / 3.0)
    want = oracle.e4m3_encode((xf * s).astype(np.float32))
    assert np.array_equal(oracle.quantize_e4m3(bits, float(s)), want)
    d = oracle.e4m3_decode(oracle.quantize_e4m3(bits, 4.0))
    assert np.all(np.abs(d - 4 * xf) <= np.maximum(np.abs(4 * xf) / 16, 2.0 ** -10) + 1e-12)
    del rng


def test_bf16_bits_of_e4m3_are_exact():
    codes = np.arange(256, dtype=np.uint8)
    d = oracle.e4m3_decode(codes)
    ok = ~np.isnan(d)
    b = oracle.e4m3_to_bf16_bits(codes[ok])
    assert np.array_equal(brute.bf16_to_f64(b), d[ok])


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_attention_equals_brute_force(causal):
    rng = np.random.default_rng(5 + causal)
    N, D, block = 256, 16, 64
    nb = N // block
    q8 = oracle.e4m3_encode((rng.standard_normal((1, N, D)) * 8).astype(np.float32))
    k8 = oracle.e4m3_encode((rng.standard_normal((1, N, D)) * 8).astype(np.float32))
    v = torch.randn(1, N, D).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    lists = [sorted(rng.choice(nb, size=rng.integers(0, nb + 1), replace=False).tolist()) for _ in range(nb)]
    row_ptr = np.concatenate([[0], np.cumsum([len(l) for l in lists])]).astype(np.int32)
    col_idx = np.array([j for l in lists for j in l], dtype=np.int32)
    qd, kd, scale = 0.125, 0.25, 1 / np.sqrt(D)
    o, lse = oracle.attention_rows_fp8(q8, k8, v, row_ptr, col_idx, block, qd, kd, scale, causal)
    allowed = brute.expand_block_mask(brute.block_mask_from_csr(row_ptr, col_idx, nb), block, causal)
    o_ref, l_ref = brute.masked_attention(oracle.e4m3_decode(q8[0]) * qd, oracle.e4m3_decode(k8[0]) * kd,
                                          brute.bf16_to_f64(v[0]), allowed, scale)
    assert np.allclose(o, o_ref, rtol=0, atol=1e-12)
    both = np.isinf(lse) & np.isinf(l_ref)
    assert np.array_equal(np.isinf(lse), np.isinf(l_ref))
    assert np.allclose(lse[~both], l_ref[~both], rtol=0, atol=1e-12)


def test_fp8_attention_depends_on_descale_product_only():
    rng = np.random.default_rng(9)
    N, D, block = 128, 32, 64
    q8 = oracle.e4m3_encode(rng.standard_normal((1, N, D)).astype(np.float32) * 4)
    k8 = oracle.e4m3_encode(rng.standard_normal((1, N, D)).astype(np.float32) * 4)
    v = torch.randn(1, N, D).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    rp = np.array([0, 1, 3], dtype=np.int32)
    ci = np.array([0, 0, 1], dtype=np.int32)
    a = oracle.attention_rows_fp8(q8, k8, v, rp, ci, block, 2.0, 0.25, 0.1, True)
    b = oracle.attention_rows_fp8(q8, k8, v, rp, ci, block, 1.0, 1.0, 0.05, True)
    c = oracle.attention_rows_fp8(q8, k8, v, rp, ci, block, 1.0, 1.0, 0.1, True)
    assert np.allclose(a[0], b[0], atol=1e-13) and np.allclose(a[1], b[1], atol=1e-13)
    assert not np.allclose(a[0], c[0], atol=1e-6)
