"""The C-ABI library builds, loads, exports every symbol include/bsa.h
declares, and rejects invalid arguments on the host (no GPU needed: every
call here returns before touching a device)."""

import ctypes
import json
import os
import re

import numpy as np
import pytest

import bsa_inputs
from parity import ex_pair as _ex_pair, random_ex_specs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "pattern_masks.json")))


@pytest.fixture(scope="module")
def L():
    from block_sparse_flashattention_bsa_gb300 import build as B
    B.build()
    import block_sparse_flashattention_bsa_gb300 as bsa
    return bsa.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "bsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bsa_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n


def test_version_and_status_strings(L):
    assert L.bsa_version() == 102
    for st in (0, -1, -2, -3, -4, -5):
        assert L.bsa_status_string(st)
    assert L.bsa_status_string(0) == b"ok"


@pytest.mark.parametrize("w", [w for w in bsa_inputs.WORKLOADS if not w.is_topk], ids=lambda w: w.name)
def test_pattern_nnz_closed_form(L, w):
    import block_sparse_flashattention_bsa_gb300 as bsa
    p = bsa.Pattern(w.n_blocks, w.window_left, w.window_right, w.causal, w.global_blocks,
                    w.global_rows_attend_all)
    assert bsa.pattern_nnz(p, w.B, w.H) == GOLDEN[w.name]["nnz_per_head"] * w.B * w.H
    # the count-only form of bsa_build_mask_csr (col_idx NULL) launches nothing
    n = ctypes.c_int64(-1)
    st = L.bsa_build_mask_csr(ctypes.byref(p._c()), w.B, w.H, None, None, 0, ctypes.byref(n), None)
    assert st == 0 and n.value == GOLDEN[w.name]["nnz_per_head"] * w.B * w.H


def test_invalid_arguments_rejected_on_host(L):
    import block_sparse_flashattention_bsa_gb300 as bsa
    from block_sparse_flashattention_bsa_gb300._binding import _Shape
    INVALID, UNSUP = -1, -2
    n = ctypes.c_int64(0)
    bad_window = bsa.Pattern(8, -1, 0)
    assert L.bsa_pattern_nnz(ctypes.byref(bad_window._c()), 1, 1, ctypes.byref(n)) == INVALID
    bad_global = bsa.Pattern(8, 1, 1, global_blocks=(9,))
    assert L.bsa_pattern_nnz(ctypes.byref(bad_global._c()), 1, 1, ctypes.byref(n)) == INVALID
    assert L.bsa_pattern_nnz(None, 1, 1, ctypes.byref(n)) == INVALID
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: rejected before launch
    ragged = _Shape(1, 1, 1000, 128, 128)  # N % block != 0
    assert L.bsa_forward(ctypes.byref(ragged), fake, fake, fake, fake, fake, fake, fake,
                         ctypes.c_float(0.1), 0, None) == INVALID
    d96 = _Shape(1, 1, 1024, 96, 128)
    assert L.bsa_forward(ctypes.byref(d96), fake, fake, fake, fake, fake, fake, fake,
                         ctypes.c_float(0.1), 0, None) == UNSUP
    ok = _Shape(1, 1, 1024, 128, 128)
    assert L.bsa_forward(ctypes.byref(ok), None, fake, fake, fake, fake, fake, fake,
                         ctypes.c_float(0.1), 0, None) == INVALID
    mis = ctypes.c_void_p((1 << 20) + 8)  # not 16-byte aligned
    assert L.bsa_forward(ctypes.byref(ok), mis, fake, fake, fake, fake, fake, fake,
                         ctypes.c_float(0.1), 0, None) == INVALID
    assert L.bsa_forward(ctypes.byref(ok), fake, fake, fake, fake, fake, fake, fake,
                         ctypes.c_float(-1.0), 0, None) == INVALID
    assert L.bsa_forward(ctypes.byref(ok), fake, fake, fake, fake, fake, fake, fake,
                         ctypes.c_float(0.1), 2, None) == INVALID
    # top-k: k larger than the number of blocks, or beyond the built limit
    small = _Shape(1, 1, 1024, 128, 64)
    assert L.bsa_topk_blocks(ctypes.byref(small), fake, fake, 17, 1, fake, fake, 1 << 20, None) == INVALID
    big = _Shape(1, 1, 64 * 100, 128, 64)
    assert L.bsa_topk_blocks(ctypes.byref(big), fake, fake, 40, 1, fake, fake, 1 << 20, None) == UNSUP
    # capacity check happens on the host too
    assert L.bsa_topk_blocks(ctypes.byref(small), fake, fake, 4, 1, fake, fake, 10, None) == -3
    p = bsa.Pattern(8, 1, 1)
    assert L.bsa_build_mask_csr(ctypes.byref(p._c()), 1, 1, fake, fake, 3, ctypes.byref(n), None) == -3


def test_product_path_refuses_without_library(tmp_path, monkeypatch):
    """With no libbsa.so the binding raises instead of computing anything."""
    from block_sparse_flashattention_bsa_gb300 import _binding
    monkeypatch.setattr(_binding, "_LIB_FILE", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_binding, "_lib", None)
    with pytest.raises(RuntimeError):
        _binding.lib()


# ------------------------------------------------------------ per-head patterns
EX_GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "pattern_ex_masks.json")))


@pytest.mark.parametrize("name", [k for k in EX_GOLDEN if not k.startswith("_")])
def test_pattern_ex_count_matches_golden(L, name):
    import block_sparse_flashattention_bsa_gb300 as bsa
    p, _ = _ex_pair(EX_GOLDEN[name]["pattern"])
    assert bsa.mask_heads_nnz([p], 1, 1) == EX_GOLDEN[name]["nnz"]
    assert bsa.mask_heads_nnz([p], 3, 5) == EX_GOLDEN[name]["nnz"] * 15


def test_heads_count_matches_oracle(L):
    import block_sparse_flashattention_bsa_gb300 as bsa
    import oracle
    rng = np.random.default_rng(11)
    for trial in range(30):
        nb = int(rng.integers(1, 60))
        specs = random_ex_specs(rng, nb, int(rng.integers(1, 9)))
        pairs = [_ex_pair(s) for s in specs]
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 12))
        hp = [int(x) for x in rng.integers(0, len(specs), size=H)] if trial % 2 else None
        rp, _ = oracle.heads_csr([o for _, o in pairs], B, H, hp)
        assert bsa.mask_heads_nnz([p for p, _ in pairs], B, H, hp) == int(rp[-1]), (trial, specs)


def test_heads_invalid_arguments_rejected_on_host(L):
    import block_sparse_flashattention_bsa_gb300 as bsa
    from block_sparse_flashattention_bsa_gb300._binding import _PatternEx

    def status(pats, H=2, hp=None, B=1):
        arr = (_PatternEx * max(1, len(pats)))()
        keep = [arr]
        for x, p in enumerate(pats):
            p._fill(arr[x], keep)
        hpa = None if hp is None else (ctypes.c_int32 * len(hp))(*hp)
        n = ctypes.c_int64(0)
        return L.bsa_build_mask_csr_heads(arr, len(pats), hpa, B, H, None, None, 0, ctypes.byref(n), None)

    ok = bsa.PatternEx(16, windows=[(1, 1, 2)], stride=4)
    assert status([ok]) == 0
    assert status([bsa.PatternEx(16, windows=[(1, 1, 0)])]) == -1          # dilation 0
    assert status([bsa.PatternEx(16, windows=[(-1, 1, 1)])]) == -1         # negative extent
    assert status([bsa.PatternEx(16, stride=-2)]) == -1                    # negative stride
    assert status([bsa.PatternEx(16, global_blocks=[16])]) == -1           # global out of range
    assert status([ok, bsa.PatternEx(17)]) == -1                           # n_blocks differ
    assert status([ok], hp=[0, 1]) == -1                                   # head -> missing pattern
    assert status([ok] * 9, H=9) == -1                                     # more than 8 patterns
    assert status([ok], H=1025) == -1                                      # too many heads
    assert status([ok], B=0) == -1
    many = [bsa.PatternEx(300, global_blocks=list(range(64)))] * 5         # 320 globals > 256
    assert status(many) == -1
    assert L.bsa_build_mask_csr_heads(None, 1, None, 1, 1, None, None, 0, None, None) == -1
    # n_windows above the limit, set through the raw struct
    arr = (_PatternEx * 1)()
    ok._fill(arr[0], [])
    arr[0].n_windows = 5
    assert L.bsa_build_mask_csr_heads(arr, 1, None, 1, 1, None, None, 0, None, None) == -1
    assert L.bsa_build_mask_csr_heads(arr, 0, None, 1, 1, None, None, 0, None, None) == -1
    # too small col_capacity is refused before any device work (the pointers
    # are never dereferenced)
    arr[0].n_windows = 1
    fake = ctypes.c_void_p(256)
    assert L.bsa_build_mask_csr_heads(arr, 1, None, 1, 1, fake, fake, 1, None, None) == -3
    with pytest.raises(bsa.BsaError):
        bsa.mask_heads_nnz([bsa.PatternEx(16, windows=[(1, 1, 0)])], 1, 1)


def test_backward_invalid_arguments_rejected_on_host(L):
    """bsa_backward checks everything on the host before touching a device
    (the pointers below are never dereferenced)."""
    from block_sparse_flashattention_bsa_gb300._binding import _Shape
    P = ctypes.c_void_p
    good = P(4096)  # 16-byte aligned, never dereferenced

    def call(sh=(1, 2, 1024, 128, 128), ptrs=None, lse=good, cap=10, scale=0.1, causal=1, mis=None):
        s = _Shape(*sh)
        p = [good] * 11 if ptrs is None else ptrs
        if mis is not None:
            p = list(p)
            p[mis] = P(4096 + 8)  # 8-byte aligned only
        q, k, v, o, do, rp, ci, dq, dk, dv = p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7], p[8], p[9]
        return L.bsa_backward(ctypes.byref(s), q, k, v, o, do, lse, rp, ci, cap, dq, dk, dv,
                              ctypes.c_float(scale), causal, None)

    assert call(sh=(1, 2, 1000, 128, 128)) == -1           # N not a multiple of the block
    assert call(sh=(1, 2, 1024, 128, 32)) == -2            # block 32: not built
    assert call(sh=(1, 2, 1024, 96, 128)) == -2            # head dim
    assert call(ptrs=[None] + [good] * 10) == -1           # null q
    assert call(lse=None) == -1
    assert call(mis=0) == -1 and call(mis=7) == -1         # misaligned q, dq
    assert call(cap=-1) == -1
    assert call(scale=0.0) == -1 and call(scale=float("inf")) == -1
    assert call(causal=2) == -1


def test_fp8_invalid_arguments_rejected_on_host(L):
    """bsa_forward_fp8 and bsa_quantize_e4m3 check their arguments on the
    host before touching a device (the pointers are never dereferenced)."""
    from block_sparse_flashattention_bsa_gb300._binding import _Shape
    P = ctypes.c_void_p
    good = P(4096)

    def fwd(sh=(1, 2, 1024, 128, 128), q=good, lse=good, qd=1.0, kd=1.0, scale=0.1, causal=0):
        s = _Shape(*sh)
        return L.bsa_forward_fp8(ctypes.byref(s), q, good, good, good, good, good, lse, ctypes.c_float(qd),
                                 ctypes.c_float(kd), ctypes.c_float(scale), causal, None)

    assert fwd(sh=(1, 2, 1024, 64, 128)) == -2              # FP8 scores: D = 128 only
    assert fwd(sh=(1, 2, 1024, 128, 256)) == -2             # block 256
    assert fwd(sh=(1, 2, 1000, 128, 128)) == -1             # N not a multiple of the block
    assert fwd(q=None) == -1 and fwd(lse=None) == -1
    assert fwd(q=P(4096 + 8)) == -1                          # misaligned
    assert fwd(qd=0.0) == -1 and fwd(kd=-1.0) == -1 and fwd(qd=float("nan")) == -1
    assert fwd(scale=0.0) == -1 and fwd(scale=float("inf")) == -1
    assert fwd(qd=1e30, kd=1e30) == -1                        # the product overflows fp32
    assert fwd(causal=3) == -1

    def quant(x=good, y=good, n=4096, inv=1.0):
        return L.bsa_quantize_e4m3(x, y, n, ctypes.c_float(inv), None)

    assert quant(n=0) == -1 and quant(n=4104) == -1           # n a positive multiple of 16
    assert quant(x=None) == -1 and quant(y=P(4096 + 4)) == -1
    assert quant(inv=0.0) == -1 and quant(inv=float("inf")) == -1



def test_binding_rejects_wrong_tensors_before_any_call(L):
    """The Python marshalling refuses host tensors and wrong dtypes (no device needed)."""
    import torch

    import block_sparse_flashattention_bsa_gb300 as bsa
    x = torch.zeros(1, 2, 128, 128, dtype=torch.bfloat16)
    rp = torch.zeros(3, dtype=torch.int32)
    with pytest.raises(ValueError):
        bsa.forward(x, x, x, rp, rp, 128)
    with pytest.raises(ValueError):
        bsa.quantize_e4m3(x, 1.0)
    codes = torch.zeros(1, 2, 128, 128, dtype=torch.uint8)
    with pytest.raises(ValueError):
        bsa.forward_fp8(codes, codes, x, rp, rp, 128, 1.0, 1.0)
    with pytest.raises(ValueError):  # e4m3 codes must be bytes
        bsa.forward_fp8(x, x, x, rp, rp, 128, 1.0, 1.0)


def test_wait_limit_setting_host_only(L):
    """The wait limit is a host-side setting: range-checked, 0 restores 2 s."""
    import block_sparse_flashattention_bsa_gb300 as bsa
    assert bsa.get_wait_limit() == 2_000_000_000
    assert L.bsa_set_wait_limit(999) == -1
    assert L.bsa_set_wait_limit(601 * 10 ** 9) == -1
    bsa.set_wait_limit(5_000_000)
    assert bsa.get_wait_limit() == 5_000_000
    bsa.set_wait_limit(0)
    assert bsa.get_wait_limit() == 2_000_000_000
    assert L.bsa_debug_stall_next_forward(-2) == -1
    bsa.debug_stall_next_forward(3)
    bsa.debug_stall_next_forward(-1)  # cancel: nothing may stay pending for later tests
