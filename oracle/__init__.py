"""fp64 CPU oracle for block-sparse attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
binding) never imports it, and it imports nothing from the product path; the
only shared code is the seeded input module ``bsa_inputs``.

Two independent implementations live here:

* ``bsa_oracle.c`` (built into ``liboracle.so``): the pattern masks (plain
  window, and dilated windows / stride) by brute force, exact fp64 masked attention for any list of query rows, its
  fp64 backward (dQ, dK, dV of sum(dO * O)), and the
  fp32 content-based top-k selection in its stated order.
* the e4m3 codec below (numpy): OCP 8-bit floating point E4M3, decode and
  round-to-nearest-even encode with saturation, for the FP8-score forward.
* ``brute.py``: a literal numpy version for tiny shapes -- a full N x N token
  mask filled with -inf, full-row softmax -- used to cross-check the C code.

Parity status of each function is recorded in the module docstrings of the
tests that pin it; functions without a pin say "parity unpinned" here.  All
functions below are pinned (see tests/test_oracle_*.py).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: the top-k scores are compared bit-exactly, so the
# compiler must not fuse the stated multiplies and adds.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
          "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (idempotent)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


class _Pattern(ctypes.Structure):
    _fields_ = [("n_blocks", ctypes.c_int32), ("window_left", ctypes.c_int32),
                ("window_right", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("n_global", ctypes.c_int32), ("global_blocks", ctypes.POINTER(ctypes.c_int32)),
                ("global_rows_attend_all", ctypes.c_int32), ("global_rows_noncausal", ctypes.c_int32)]


class _PatternEx(ctypes.Structure):
    _fields_ = [("n_blocks", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("n_windows", ctypes.c_int32),
                ("window_left", ctypes.c_int32 * 4), ("window_right", ctypes.c_int32 * 4),
                ("window_dilation", ctypes.c_int32 * 4),
                ("stride", ctypes.c_int32), ("n_global", ctypes.c_int32),
                ("global_blocks", ctypes.POINTER(ctypes.c_int32)),
                ("global_rows_attend_all", ctypes.c_int32)]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_set_num_threads.argtypes = [ctypes.c_int]
        lib.orc_pattern_allows.argtypes = [ctypes.POINTER(_Pattern), i32, i32]
        lib.orc_pattern_allows.restype = ctypes.c_int
        lib.orc_pattern_csr.argtypes = [ctypes.POINTER(_Pattern), P, P]
        lib.orc_pattern_csr.restype = i64
        lib.orc_pattern_ex_allows.argtypes = [ctypes.POINTER(_PatternEx), i32, i32]
        lib.orc_pattern_ex_allows.restype = ctypes.c_int
        lib.orc_pattern_ex_csr.argtypes = [ctypes.POINTER(_PatternEx), P, P]
        lib.orc_pattern_ex_csr.restype = i64
        lib.orc_attention_rows.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, f64, i32,
                                           i64, P, P, P, P]
        lib.orc_attention_rows.restype = None
        lib.orc_attention_backward.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P, f64, i32,
                                               i64, P, P, i64, P, P, P]
        lib.orc_attention_backward.restype = None
        lib.orc_block_means.argtypes = [i32, i32, i32, i32, P, P]
        lib.orc_block_scores.argtypes = [i32, i32, i32, P, P, P]
        lib.orc_topk_csr.argtypes = [i32, i32, P, i32, i32, P, P]
        lib.orc_topk_csr.restype = i64
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


def attention_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, dout: np.ndarray,
                       row_ptr: np.ndarray, col_idx: np.ndarray, block: int, scale: float,
                       causal: bool, qrows: Optional[np.ndarray] = None,
                       krows: Optional[np.ndarray] = None, row_flags: Optional[np.ndarray] = None):
    """Gradients of sum(dO * O) of the masked attention, fp64.

    q, k, v, dout: fp64 arrays [BH, N, D] (widen bf16 inputs exactly first).
    qrows / krows: flat row ids bh*N + t (default: all).  ``row_flags``:
    optional uint8 per CSR row, bit 0 = that row takes no causal cut (the
    forward's attention_rows reading).  Returns (dQ [n_q, D], dK [n_k, D],
    dV [n_k, D]).
    """
    BH, N, D = q.shape
    qd, kd, vd, dd = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v, dout))
    allr = np.arange(BH * N, dtype=np.int64)
    qr = np.ascontiguousarray(allr if qrows is None else qrows, dtype=np.int64)
    kr = np.ascontiguousarray(allr if krows is None else krows, dtype=np.int64)
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    ci = np.ascontiguousarray(col_idx if len(col_idx) else np.zeros(1, np.int32), dtype=np.int32)
    dq = np.zeros((len(qr), D))
    dk = np.zeros((len(kr), D))
    dv = np.zeros((len(kr), D))
    fl = None
    if row_flags is not None:
        fl = np.ascontiguousarray(row_flags, dtype=np.uint8)
        assert fl.shape[0] == rp.shape[0] - 1, "one flag per CSR row"
    _load().orc_attention_backward(BH, N, D, int(block), _ptr(qd), _ptr(kd), _ptr(vd), _ptr(dd), _ptr(rp),
                                   _ptr(ci), _ptr(fl), float(scale), int(bool(causal)), len(qr), _ptr(qr),
                                   _ptr(dq), len(kr), _ptr(kr), _ptr(dk), _ptr(dv))
    return dq, dk, dv


class Pattern:
    """A block mask recipe: window [i-wl, i+wr], global blocks, causal;
    global query rows attend to all blocks (global_rows_attend_all), without
    the causal cut when global_rows_noncausal is also set."""

    def __init__(self, n_blocks: int, window_left: int = 0, window_right: int = 0,
                 causal: bool = False, global_blocks: Sequence[int] = (),
                 global_rows_attend_all: bool = False, global_rows_noncausal: bool = False):
        self.n_blocks = int(n_blocks)
        self.window_left = int(window_left)
        self.window_right = int(window_right)
        self.causal = bool(causal)
        self.global_blocks = tuple(int(g) for g in global_blocks)
        self.global_rows_attend_all = bool(global_rows_attend_all)
        self.global_rows_noncausal = bool(global_rows_noncausal)

    @classmethod
    def from_workload(cls, w) -> "Pattern":
        return cls(w.n_blocks, w.window_left, w.window_right, w.causal, w.global_blocks,
                   w.global_rows_attend_all, getattr(w, "global_rows_noncausal", False))

    def _c(self):
        g = np.asarray(self.global_blocks, dtype=np.int32)
        self._g = g  # keep alive
        return _Pattern(self.n_blocks, self.window_left, self.window_right, int(self.causal),
                        len(g), g.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                        int(self.global_rows_attend_all), int(self.global_rows_noncausal))

    def row_flags(self) -> np.ndarray:
        """uint8 [n_blocks] of one (batch, head): 1 for the global query rows
        that take no causal cut (global_rows_attend_all and
        global_rows_noncausal), else 0."""
        f = np.zeros(self.n_blocks, dtype=np.uint8)
        if self.global_rows_attend_all and self.global_rows_noncausal:
            for g in self.global_blocks:
                f[g] = 1
        return f

    def allows(self, i: int, j: int) -> bool:
        c = self._c()
        return bool(_load().orc_pattern_allows(ctypes.byref(c), int(i), int(j)))

    def csr(self) -> Tuple[np.ndarray, np.ndarray]:
        """CSR (row_ptr [nb+1], col_idx [nnz]) of one (batch, head)."""
        lib = _load()
        c = self._c()
        nnz = lib.orc_pattern_csr(ctypes.byref(c), None, None)
        row_ptr = np.zeros(self.n_blocks + 1, dtype=np.int32)
        col_idx = np.zeros(max(nnz, 1), dtype=np.int32)
        lib.orc_pattern_csr(ctypes.byref(c), _ptr(row_ptr), _ptr(col_idx))
        return row_ptr, col_idx[:nnz]


class PatternEx:
    """Dilated windows (left, right, dilation), a stride, global blocks,
    causal; brute-forced by orc_pattern_ex_allows."""

    def __init__(self, n_blocks: int, windows: Sequence[Tuple[int, int, int]] = (),
                 stride: int = 0, causal: bool = False, global_blocks: Sequence[int] = (),
                 global_rows_attend_all: bool = False):
        assert len(windows) <= 4
        self.n_blocks = int(n_blocks)
        self.windows = tuple((int(l), int(r), int(d)) for l, r, d in windows)
        self.stride = int(stride)
        self.causal = bool(causal)
        self.global_blocks = tuple(int(g) for g in global_blocks)
        self.global_rows_attend_all = bool(global_rows_attend_all)

    def _c(self):
        c = _PatternEx()
        g = np.asarray(self.global_blocks, dtype=np.int32)
        self._g = g  # keep alive
        c.n_blocks, c.causal, c.n_windows = self.n_blocks, int(self.causal), len(self.windows)
        for w, (l, r, d) in enumerate(self.windows):
            c.window_left[w], c.window_right[w], c.window_dilation[w] = l, r, d
        c.stride = self.stride
        c.n_global = len(g)
        c.global_blocks = g.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        c.global_rows_attend_all = int(self.global_rows_attend_all)
        return c

    def allows(self, i: int, j: int) -> bool:
        c = self._c()
        return bool(_load().orc_pattern_ex_allows(ctypes.byref(c), int(i), int(j)))

    def csr(self) -> Tuple[np.ndarray, np.ndarray]:
        """CSR (row_ptr [nb+1], col_idx [nnz]) of one head."""
        lib = _load()
        c = self._c()
        nnz = lib.orc_pattern_ex_csr(ctypes.byref(c), None, None)
        row_ptr = np.zeros(self.n_blocks + 1, dtype=np.int32)
        col_idx = np.zeros(max(nnz, 1), dtype=np.int32)
        lib.orc_pattern_ex_csr(ctypes.byref(c), _ptr(row_ptr), _ptr(col_idx))
        return row_ptr, col_idx[:nnz]


def heads_csr(patterns: Sequence[PatternEx], B: int, H: int,
              head_pattern: Optional[Sequence[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """CSR over rows r = (b*H + h)*nb + i with head h following
    patterns[head_pattern[h]] (default h % len(patterns)), the same for every b."""
    per = [p.csr() for p in patterns]
    hp = list(head_pattern) if head_pattern is not None else [h % len(patterns) for h in range(H)]
    nb = patterns[0].n_blocks
    lens, cols = [], []
    for _b in range(B):
        for h in range(H):
            rp, ci = per[hp[h]]
            lens.append(np.diff(rp))
            cols.append(ci)
    lens = np.concatenate(lens) if lens else np.zeros(0, np.int32)
    row_ptr = np.zeros(B * H * nb + 1, dtype=np.int32)
    row_ptr[1:] = np.cumsum(lens)
    col_idx = np.concatenate(cols).astype(np.int32) if cols else np.zeros(0, np.int32)
    return row_ptr, col_idx


def replicate_csr(row_ptr: np.ndarray, col_idx: np.ndarray, BH: int) -> Tuple[np.ndarray, np.ndarray]:
    """The per-(b, h) CSR repeated for BH heads (rows r = bh*nb + i)."""
    nb = row_ptr.shape[0] - 1
    nnz = int(row_ptr[-1])
    rp = np.zeros(BH * nb + 1, dtype=np.int64)
    for bh in range(BH):
        rp[bh * nb + 1: (bh + 1) * nb + 1] = row_ptr[1:].astype(np.int64) + bh * nnz
    return rp.astype(np.int32), np.tile(col_idx, BH).astype(np.int32)


def attention_rows(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray,
                   row_ptr: np.ndarray, col_idx: np.ndarray, block: int, scale: float,
                   causal: bool, rows: Optional[np.ndarray] = None,
                   return_counts: bool = False, row_flags: Optional[np.ndarray] = None):
    """Exact fp64 masked attention.

    q_bits/k_bits/v_bits: uint16 bf16 bit patterns shaped [B, H, N, D] (or
    [BH, N, D]); CSR over rows r = bh*nb + i.  ``rows``: flat row ids bh*N + t
    (default: every row).  ``row_flags``: optional uint8 per CSR row, bit 0 =
    that row takes no causal cut.  Returns (O [n_rows, D] fp64, LSE [n_rows]
    fp64[, counts]).
    """
    lib = _load()
    N, D = q_bits.shape[-2], q_bits.shape[-1]
    BH = int(np.prod(q_bits.shape[:-2]))
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    ci = np.ascontiguousarray(col_idx, dtype=np.int32)
    if ci.size == 0:
        ci = np.zeros(1, dtype=np.int32)
    if rows is None:
        rows = np.arange(BH * N, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.shape[0]
    out = np.empty((n, D), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    cnt = np.empty(n, dtype=np.int64) if return_counts else None
    fl = None
    if row_flags is not None:
        fl = np.ascontiguousarray(row_flags, dtype=np.uint8)
        assert fl.shape[0] == rp.shape[0] - 1, "one flag per CSR row"
    lib.orc_attention_rows(BH, N, D, int(block), _ptr(q), _ptr(k), _ptr(v), _ptr(rp), _ptr(ci), _ptr(fl),
                           float(scale), int(bool(causal)), n, _ptr(rows), _ptr(out), _ptr(lse),
                           _ptr(cnt))
    if return_counts:
        return out, lse, cnt
    return out, lse


def block_means(x_bits: np.ndarray, block: int) -> np.ndarray:
    """fp32 block means [BH, nb, D] in the stated pairwise-tree order."""
    lib = _load()
    N, D = x_bits.shape[-2], x_bits.shape[-1]
    BH = int(np.prod(x_bits.shape[:-2]))
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    out = np.empty((BH, N // block, D), dtype=np.float32)
    lib.orc_block_means(BH, N, D, int(block), _ptr(x), _ptr(out))
    return out


def block_scores(qbar: np.ndarray, kbar: np.ndarray) -> np.ndarray:
    """fp32 block scores [BH, nb, nb] in the stated order."""
    lib = _load()
    BH, nb, D = qbar.shape
    qb = np.ascontiguousarray(qbar, dtype=np.float32)
    kb = np.ascontiguousarray(kbar, dtype=np.float32)
    out = np.empty((BH, nb, nb), dtype=np.float32)
    lib.orc_block_scores(BH, nb, D, _ptr(qb), _ptr(kb), _ptr(out))
    return out


def topk_csr_from_scores(scores: np.ndarray, topk: int, include_diag: bool = True):
    lib = _load()
    BH, nb, _ = scores.shape
    s = np.ascontiguousarray(scores, dtype=np.float32)
    nnz = lib.orc_topk_csr(BH, nb, _ptr(s), int(topk), int(include_diag), None, None)
    rp = np.zeros(BH * nb + 1, dtype=np.int32)
    ci = np.zeros(max(nnz, 1), dtype=np.int32)
    lib.orc_topk_csr(BH, nb, _ptr(s), int(topk), int(include_diag), _ptr(rp), _ptr(ci))
    return rp, ci[:nnz]


def topk_csr(q_bits: np.ndarray, k_bits: np.ndarray, block: int, topk: int,
             include_diag: bool = True):
    """Content-based block selection: (row_ptr, col_idx, scores)."""
    qbar = block_means(q_bits, block)
    kbar = block_means(k_bits, block)
    scores = block_scores(qbar, kbar)
    rp, ci = topk_csr_from_scores(scores, topk, include_diag)
    return rp, ci, scores


# ---------------------------------------------------------------- e4m3
# Scores computed in FP8 ("Flash MSA Sparse Attention Kernels Explained",
# section "The Future of Attention Kernels") take e4m3 Q and K.  The format is
# the OCP 8-bit floating point E4M3 ("FN": 1 sign, 4 exponent bits with bias
# 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, so the largest finite
# value is 1.75 * 2^8 = 448; exponent field 0 holds the subnormals m/8 * 2^-6).

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """fp64 values of e4m3 codes (uint8); NaN for S.1111.111."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """e4m3 codes of fp32 values: nearest representable value, ties to the
    even code, magnitudes above 448 saturated to 448, the sign of zero kept,
    NaN to S.1111.111."""
    x = np.asarray(x, dtype=np.float32)
    neg = np.signbit(x)
    a = np.abs(x.astype(np.float64))
    nan = np.isnan(a)
    a = np.where(nan, 0.0, np.minimum(a, E4M3_MAX))
    # quantum of the binade of a: 2^(e-3) for a normal a = 1.f * 2^e, 2^-9 below 2^-6
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(ex - 1, -6)
    q = np.exp2(e - 3.0)
    val = np.rint(a / q) * q          # round half to even on the exact quotient
    val = np.minimum(val, E4M3_MAX)   # cannot exceed 448: a <= 448 and 448 is a grid point
    # code of val
    _, ev = np.frexp(np.where(val > 0, val, 1.0))
    ev = ev - 1
    normal = val >= 2.0 ** -6
    mant_n = np.rint((val / np.exp2(ev) - 1.0) * 8.0)
    code_n = ((ev + 7) << 3) + mant_n
    code_s = np.rint(val / 2.0 ** -9)
    code = np.where(normal, code_n, code_s).astype(np.int64)
    code = np.where(nan, 0x7F, code)
    return (code | (neg.astype(np.int64) << 7)).astype(np.uint8)


def quantize_e4m3(x_bits: np.ndarray, inv_scale: float) -> np.ndarray:
    """e4m3 codes of bf16 values (uint16 bit patterns) times inv_scale, the
    product rounded once to fp32."""
    x = (np.asarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    return e4m3_encode(x * np.float32(inv_scale))


def e4m3_to_bf16_bits(codes) -> np.ndarray:
    """bf16 bit patterns of e4m3 values (every finite e4m3 value is a bf16 value)."""
    v = e4m3_decode(codes).astype(np.float32)
    bits = v.view(np.uint32)
    assert not np.any(bits & 0xFFFF), "e4m3 value not exact in bf16"
    return (bits >> 16).astype(np.uint16)


def attention_rows_fp8(q8: np.ndarray, k8: np.ndarray, v_bits: np.ndarray, row_ptr: np.ndarray,
                       col_idx: np.ndarray, block: int, q_descale: float, k_descale: float,
                       scale: float, causal: bool, rows: Optional[np.ndarray] = None):
    """Exact fp64 masked attention with FP8 scores: Q = e4m3(q8) * q_descale,
    K = e4m3(k8) * k_descale, logits Q K^T * scale, V bf16.  The descale
    factors only scale the logits, so this is attention_rows on the decoded
    codes with scale * q_descale * k_descale."""
    return attention_rows(e4m3_to_bf16_bits(q8), e4m3_to_bf16_bits(k8), v_bits, row_ptr, col_idx, block,
                          float(scale) * float(q_descale) * float(k_descale), causal, rows=rows)


# ---------------------------------------------------------------- fp64 inputs, general geometry
def attention_blocks_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, row_ptr: np.ndarray,
                         col_idx: np.ndarray, block: int, scale: float, causal: bool,
                         rows: Optional[np.ndarray] = None, row_flags: Optional[np.ndarray] = None,
                         q_block_offset: int = 0):
    """Exact masked attention on fp64 inputs, one query block at a time (numpy).

    q: [BH, Nq, D]; k, v: [BH, Nk, D] (fp64 values).  CSR rows r = bh*nbq + i
    (nbq = Nq / block) list key blocks j in [0, Nk / block).  Query token t of
    block i sits at key position (i + q_block_offset) * block + (t mod block):
    with causal, key token u of block j is allowed only if j*block + u <= that
    position, unless the row's flag bit 0 is set.  The block mask is taken as a
    set; entries outside the key blocks are ignored.  ``rows``: flat row ids
    bh*Nq + t (default all).  Returns (O [n, D], LSE [n]); a row with no
    allowed key gives O = 0 and LSE = -inf.

    The same definition as orc_attention_rows (the Attention(Q, K, V) formula
    of "Flash MSA Sparse Attention vs Full Attention", "The Mechanics"),
    written for inputs that are not bf16 values and for a key range held apart
    from the query range, as a sequence shard sees it.
    """
    BH, Nq, D = q.shape
    Nk = k.shape[1]
    nbq, nbk = Nq // block, Nk // block
    if rows is None:
        rows = np.arange(BH * Nq, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), D))
    lse = np.full(len(rows), -np.inf)
    # group the requested rows by their query block
    qblk = rows // block
    order = np.argsort(qblk, kind="stable")
    uniq, starts = np.unique(qblk[order], return_index=True)
    ends = np.append(starts[1:], len(order))
    for ub, s0, s1 in zip(uniq, starts, ends):
        sel = order[s0:s1]
        bh, i = int(ub) // nbq, int(ub) % nbq
        r = bh * nbq + i
        js = sorted(set(int(j) for j in col_idx[row_ptr[r]:row_ptr[r + 1]] if 0 <= j < nbk))
        if not js:
            continue
        t = rows[sel] - bh * Nq                       # query rows within the head
        keys = np.concatenate([np.arange(j * block, (j + 1) * block) for j in js])
        s = (q[bh, t] @ k[bh, keys].T) * scale        # [n, n_keys]
        row_causal = causal and not (row_flags is not None and (int(row_flags[r]) & 1))
        if row_causal:
            pos = (i + q_block_offset) * block + (t % block)
            s = np.where(keys[None, :] <= pos[:, None], s, -np.inf)
        m = s.max(axis=1)
        ok = np.isfinite(m)
        mm = np.where(ok, m, 0.0)
        p = np.exp(s - mm[:, None])
        l = p.sum(axis=1)
        o = (p @ v[bh, keys]) / np.where(l > 0, l, 1.0)[:, None]
        o[~ok] = 0.0
        out[sel] = o
        lse[sel] = np.where(ok, mm + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return out, lse


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """fp64 values of bf16 bit patterns (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- merge of partial results
def merge_partials(outs: Sequence[np.ndarray], lses: Sequence[np.ndarray]):
    """Combine partial attention results over disjoint key sets.

    Part p holds O_p (softmax over its keys, times V) and LSE_p (log of its
    sum of exponentials).  The whole row has LSE = log sum_p exp(LSE_p) and
    O = sum_p exp(LSE_p - LSE) O_p: the online-softmax rescale of "Flash MSA
    Sparse Attention vs Full Attention", "The Mechanics", applied to whole
    partial results -- the merge of partial outputs that "How Do Sparse
    Attention Kernels Work in GPU Clusters?" ("Distributed Sparse
    Attention", local attention plus a global merge) calls for.  Parts with
    LSE = -inf (no key) contribute nothing; a row with no key in any part
    gives O = 0, LSE = -inf.
    """
    L = np.stack([np.asarray(x, dtype=np.float64) for x in lses])          # [P, n]
    O = np.stack([np.asarray(x, dtype=np.float64) for x in outs])          # [P, n, D]
    m = L.max(axis=0)
    ok = np.isfinite(m)
    mm = np.where(ok, m, 0.0)
    w = np.exp(L - mm[None, :])                                           # exp(-inf) = 0
    tot = w.sum(axis=0)
    lse = np.where(ok, mm + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    o = (w[:, :, None] * O).sum(axis=0) / np.where(tot > 0, tot, 1.0)[:, None]
    o[~ok] = 0.0
    return o, lse


# ---------------------------------------------------------------- per-block e4m3
def quantize_e4m3_blocks(x_bits: np.ndarray, block: int):
    """e4m3 codes of bf16 values with one scale per (head, block of tokens).

    x_bits: uint16 bf16 bit patterns [BH, N, D].  For each block of `block`
    tokens of a head: amax = max |x| over its block x D values; inv =
    fp32(448 / amax) (one rounding; 1 when amax is 0); codes =
    e4m3(fp32(x * inv)) as in quantize_e4m3; descale = fp32(amax / 448) (1
    when amax is 0).  Returns (codes uint8 [BH, N, D], descale fp32 [BH, nb]).
    One scale per block instead of per tensor keeps peaked blocks from
    crushing the others' precision (scores "in FP8": "Flash MSA Sparse
    Attention Kernels Explained", "The Future of Attention Kernels").
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    BH, N, D = x_bits.shape
    nb = N // block
    x = (x_bits.astype(np.uint32) << 16).view(np.float32).reshape(BH, nb, block, D)
    amax = np.abs(x).max(axis=(2, 3)).astype(np.float32)                  # exact
    zero = amax == 0
    safe = np.where(zero, np.float32(1.0), amax).astype(np.float32)
    inv = np.where(zero, np.float32(1.0), np.float32(448.0) / safe).astype(np.float32)
    desc = np.where(zero, np.float32(1.0), safe / np.float32(448.0)).astype(np.float32)
    prod = (x * inv[:, :, None, None]).astype(np.float32)                 # one fp32 rounding
    codes = e4m3_encode(prod).reshape(BH, N, D)
    return codes, desc


def attention_rows_fp8_blocks(q8: np.ndarray, k8: np.ndarray, v_bits: np.ndarray, q_descale: np.ndarray,
                              k_descale: np.ndarray, row_ptr: np.ndarray, col_idx: np.ndarray, block: int,
                              scale: float, causal: bool, rows: Optional[np.ndarray] = None):
    """Exact fp64 attention with per-block FP8 scores: Q = e4m3(q8) times the
    descale of its (head, query block), K likewise per key block, logits
    Q K^T * scale, V bf16.  q8, k8, v_bits: [BH, N, D]; descales [BH, nb]."""
    BH, N, D = q8.shape
    qd = np.repeat(np.asarray(q_descale, dtype=np.float64), block, axis=1)[:, :, None]
    kd = np.repeat(np.asarray(k_descale, dtype=np.float64), block, axis=1)[:, :, None]
    q = e4m3_decode(q8).reshape(BH, N, D) * qd
    k = e4m3_decode(k8).reshape(BH, N, D) * kd
    v = bf16_to_f64(v_bits).reshape(BH, N, D)
    return attention_blocks_f64(q, k, v, row_ptr, col_idx, block, scale, causal, rows=rows)

