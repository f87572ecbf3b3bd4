"""The C-ABI library builds, loads, exports every symbol include/bsa.h
declares, and rejects invalid arguments on the host (no GPU needed: every
call here returns before touching a device)."""

import ctypes
import json
import os
import re

import pytest

import bsa_inputs

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
    return sorted(set(re.findall(r"\b(bsa_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n


def test_version_and_status_strings(L):
    assert L.bsa_version() == 100
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
