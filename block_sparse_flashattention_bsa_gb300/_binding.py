"""ctypes marshalling for libbsa.so (argument checks live in the C library)."""

from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Sequence, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_FILE = os.path.join(_HERE, "libbsa.so")
_lock = threading.Lock()
_lib = None

BSA_OK = 0
MAX_GLOBAL_BLOCKS = 64


class BsaError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__("%s failed: %s (status %d)" % (fn, text, status))
        self.status = status


class _Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("N", ctypes.c_int32),
                ("D", ctypes.c_int32), ("block", ctypes.c_int32)]


class _Pattern(ctypes.Structure):
    _fields_ = [("n_blocks", ctypes.c_int32), ("window_left", ctypes.c_int32),
                ("window_right", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("n_global", ctypes.c_int32), ("global_blocks", ctypes.POINTER(ctypes.c_int32)),
                ("global_rows_attend_all", ctypes.c_int32), ("global_rows_noncausal", ctypes.c_int32)]


class _ForwardArgs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("D", ctypes.c_int32), ("block", ctypes.c_int32),
                ("n_q_blocks", ctypes.c_int32), ("n_k_blocks", ctypes.c_int32),
                ("q_block_offset", ctypes.c_int32),
                ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("row_ptr", ctypes.c_void_p), ("col_idx", ctypes.c_void_p), ("row_flags", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("scale", ctypes.c_float),
                ("causal", ctypes.c_int32), ("out_fp32", ctypes.c_int32)]


MAX_WINDOWS = 4


class _PatternEx(ctypes.Structure):
    _fields_ = [("n_blocks", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("n_windows", ctypes.c_int32),
                ("window_left", ctypes.c_int32 * MAX_WINDOWS),
                ("window_right", ctypes.c_int32 * MAX_WINDOWS),
                ("window_dilation", ctypes.c_int32 * MAX_WINDOWS),
                ("stride", ctypes.c_int32), ("n_global", ctypes.c_int32),
                ("global_blocks", ctypes.POINTER(ctypes.c_int32)),
                ("global_rows_attend_all", ctypes.c_int32)]


def lib_path() -> str:
    return _LIB_FILE


def lib():
    """The loaded libbsa.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_FILE):
                raise RuntimeError("libbsa.so is not built (run python -m "
                                   "block_sparse_flashattention_bsa_gb300.build)")
            L = ctypes.CDLL(_LIB_FILE)
            P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            PS, PP = ctypes.POINTER(_Shape), ctypes.POINTER(_Pattern)
            PX = ctypes.POINTER(_PatternEx)
            sigs = {
                "bsa_version": ([], ctypes.c_int),
                "bsa_status_string": ([ctypes.c_int], ctypes.c_char_p),
                "bsa_pattern_nnz": ([PP, i32, i32, ctypes.POINTER(i64)], ctypes.c_int),
                "bsa_build_mask_csr": ([PP, i32, i32, P, P, i64, ctypes.POINTER(i64), P], ctypes.c_int),
                "bsa_pattern_row_flags": ([PP, i32, i32, P, P], ctypes.c_int),
                "bsa_forward_ex": ([ctypes.POINTER(_ForwardArgs), P], ctypes.c_int),
                "bsa_build_mask_csr_heads": ([PX, i32, P, i32, i32, P, P, i64, ctypes.POINTER(i64), P],
                                             ctypes.c_int),
                "bsa_topk_blocks": ([PS, P, P, i32, i32, P, P, i64, P], ctypes.c_int),
                "bsa_forward": ([PS, P, P, P, P, P, P, P, ctypes.c_float, i32, P], ctypes.c_int),
                "bsa_forward_fp8": ([PS, P, P, P, P, P, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                     i32, P], ctypes.c_int),
                "bsa_quantize_e4m3": ([P, P, i64, ctypes.c_float, P], ctypes.c_int),
                "bsa_quantize_e4m3_blocks": ([PS, P, P, P, P], ctypes.c_int),
                "bsa_forward_fp8_blocks": ([PS, P, P, P, P, P, P, P, P, P, ctypes.c_float, i32, P], ctypes.c_int),
                "bsa_backward_ex": ([PS, P, P, P, P, P, P, P, P, i64, P, P, P, P, ctypes.c_float, i32, P],
                                    ctypes.c_int),
                "bsa_backward": ([PS, P, P, P, P, P, P, P, P, i64, P, P, P, ctypes.c_float, i32, P],
                                 ctypes.c_int),
                "bsa_validate_csr": ([PS, P, P, P, P], ctypes.c_int),
                "bsa_device_error": ([ctypes.POINTER(i32)], ctypes.c_int),
                "bsa_set_wait_limit": ([i64], ctypes.c_int),
                "bsa_get_wait_limit": ([], i64),
                "bsa_debug_stall_next_forward": ([i32], ctypes.c_int),
                "bsa_forward_noalloc": ([PS, P, P, P, P, P, P, P, ctypes.c_float, i32, P], ctypes.c_int),
                "bsa_release_workspace": ([], None),
            }
            for name, (args, res) in sigs.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


def _check(fn: str, status: int) -> None:
    if status != BSA_OK:
        raise BsaError(fn, status, lib().bsa_status_string(status).decode())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class Pattern:
    """Fixed block-mask pattern: window [i - window_left, i + window_right],
    global key blocks (seen by every row), optional global query rows (see
    every block) and causal cut j <= i.  global_rows_noncausal: the global
    query rows also skip the causal cut (they see the whole sequence); the
    forward then needs the rows' flags (pattern_row_flags, forward_ex)."""

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

    def _c(self):
        arr = (ctypes.c_int32 * max(1, len(self.global_blocks)))(*self.global_blocks)
        self._keep = arr
        return _Pattern(self.n_blocks, self.window_left, self.window_right, int(self.causal),
                        len(self.global_blocks), ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32)),
                        int(self.global_rows_attend_all), int(self.global_rows_noncausal))


class PatternEx:
    """Fixed pattern of dilated windows, a stride and global blocks.

    windows: up to four (left, right, dilation) triples; window w holds the
    key blocks i + dilation * t for -left <= t <= right.  stride s > 0 adds
    every key block j with (i - j) a multiple of s.  Global blocks, global
    query rows and the causal cut j <= i as in Pattern."""

    def __init__(self, n_blocks: int, windows: Sequence[Tuple[int, int, int]] = (),
                 stride: int = 0, causal: bool = False, global_blocks: Sequence[int] = (),
                 global_rows_attend_all: bool = False):
        if len(windows) > MAX_WINDOWS:
            raise ValueError("at most %d windows" % MAX_WINDOWS)
        self.n_blocks = int(n_blocks)
        self.windows = tuple((int(l), int(r), int(d)) for l, r, d in windows)
        self.stride = int(stride)
        self.causal = bool(causal)
        self.global_blocks = tuple(int(g) for g in global_blocks)
        self.global_rows_attend_all = bool(global_rows_attend_all)

    def _fill(self, c: _PatternEx, keep: list) -> None:
        arr = (ctypes.c_int32 * max(1, len(self.global_blocks)))(*self.global_blocks)
        keep.append(arr)
        c.n_blocks, c.causal, c.n_windows = self.n_blocks, int(self.causal), len(self.windows)
        for w, (l, r, d) in enumerate(self.windows):
            c.window_left[w], c.window_right[w], c.window_dilation[w] = l, r, d
        c.stride = self.stride
        c.n_global = len(self.global_blocks)
        c.global_blocks = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
        c.global_rows_attend_all = int(self.global_rows_attend_all)


def _pattern_ex_args(patterns: Sequence[PatternEx], H: int, head_pattern: Optional[Sequence[int]]):
    arr = (_PatternEx * max(1, len(patterns)))()
    keep: list = [arr]
    for x, p in enumerate(patterns):
        p._fill(arr[x], keep)
    hp = None
    if head_pattern is not None:
        if len(head_pattern) != H:
            raise ValueError("head_pattern needs one entry per head")
        hp = (ctypes.c_int32 * H)(*[int(x) for x in head_pattern])
        keep.append(hp)
    return arr, hp, keep


def mask_heads_nnz(patterns: Sequence[PatternEx], B: int, H: int,
                   head_pattern: Optional[Sequence[int]] = None) -> int:
    """Entries of the per-head CSR (host only, no device work)."""
    arr, hp, _keep = _pattern_ex_args(patterns, H, head_pattern)
    n = ctypes.c_int64(0)
    _check("bsa_build_mask_csr_heads", lib().bsa_build_mask_csr_heads(
        arr, len(patterns), hp, B, H, None, None, 0, ctypes.byref(n), None))
    return int(n.value)


def build_mask_csr_heads(patterns: Sequence[PatternEx], B: int, H: int,
                         head_pattern: Optional[Sequence[int]] = None, device="cuda", stream=None,
                         row_ptr: Optional[torch.Tensor] = None,
                         col_idx: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Block CSR with head h following patterns[head_pattern[h]] (default
    h % len(patterns)), the same for every batch element, built on the device."""
    nnz = mask_heads_nnz(patterns, B, H, head_pattern)
    R = B * H * patterns[0].n_blocks
    if row_ptr is None:
        row_ptr = torch.empty(R + 1, dtype=torch.int32, device=device)
    if col_idx is None:
        col_idx = torch.empty(max(nnz, 1), dtype=torch.int32, device=device)
    arr, hp, _keep = _pattern_ex_args(patterns, H, head_pattern)
    n = ctypes.c_int64(0)
    _check("bsa_build_mask_csr_heads", lib().bsa_build_mask_csr_heads(
        arr, len(patterns), hp, B, H, _ptr(row_ptr), _ptr(col_idx), col_idx.numel(),
        ctypes.byref(n), _stream(stream)))
    return row_ptr, col_idx[:nnz]


def _shape(q: torch.Tensor, block: int) -> _Shape:
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, D] tensors")
    B, H, N, D = q.shape
    return _Shape(B, H, N, D, int(block))


def _require_bf16_cuda(*ts: torch.Tensor) -> None:
    for t in ts:
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("expected contiguous bf16 CUDA tensors")


def pattern_nnz(pattern: Pattern, B: int, H: int) -> int:
    n = ctypes.c_int64(0)
    _check("bsa_pattern_nnz", lib().bsa_pattern_nnz(ctypes.byref(pattern._c()), B, H, ctypes.byref(n)))
    return int(n.value)


def build_mask_csr(pattern: Pattern, B: int, H: int, device="cuda", stream=None,
                   row_ptr: Optional[torch.Tensor] = None,
                   col_idx: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Block CSR of `pattern` replicated over B*H heads, built on the device."""
    nnz = pattern_nnz(pattern, B, H)
    R = B * H * pattern.n_blocks
    if row_ptr is None:
        row_ptr = torch.empty(R + 1, dtype=torch.int32, device=device)
    if col_idx is None:
        col_idx = torch.empty(max(nnz, 1), dtype=torch.int32, device=device)
    n = ctypes.c_int64(0)
    _check("bsa_build_mask_csr", lib().bsa_build_mask_csr(
        ctypes.byref(pattern._c()), B, H, _ptr(row_ptr), _ptr(col_idx), col_idx.numel(),
        ctypes.byref(n), _stream(stream)))
    return row_ptr, col_idx[:nnz]


def pattern_row_flags(pattern: Pattern, B: int, H: int, device="cuda", stream=None,
                      out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """uint8 [B*H*n_blocks] on the device: 1 for the rows of global query
    blocks that take no causal cut, 0 elsewhere."""
    R = B * H * pattern.n_blocks
    if out is None:
        out = torch.empty(R, dtype=torch.uint8, device=device)
    _check("bsa_pattern_row_flags", lib().bsa_pattern_row_flags(ctypes.byref(pattern._c()), B, H, _ptr(out),
                                                                _stream(stream)))
    return out


def topk_blocks(q: torch.Tensor, k: torch.Tensor, block: int, topk: int, include_diag: bool = True,
                stream=None, row_ptr: Optional[torch.Tensor] = None,
                col_idx: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Content-based block CSR.  col_idx is returned at full capacity; its
    first row_ptr[-1] entries are valid."""
    _require_bf16_cuda(q, k)
    sh = _shape(q, block)
    R = sh.B * sh.H * (sh.N // block)
    cap = R * (topk + int(bool(include_diag)))
    if row_ptr is None:
        row_ptr = torch.empty(R + 1, dtype=torch.int32, device=q.device)
    if col_idx is None:
        col_idx = torch.empty(cap, dtype=torch.int32, device=q.device)
    _check("bsa_topk_blocks", lib().bsa_topk_blocks(
        ctypes.byref(sh), _ptr(q), _ptr(k), int(topk), int(bool(include_diag)), _ptr(row_ptr),
        _ptr(col_idx), col_idx.numel(), _stream(stream)))
    return row_ptr, col_idx


def forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, row_ptr: torch.Tensor,
            col_idx: torch.Tensor, block: int, scale: Optional[float] = None, causal: bool = False,
            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
            stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Block-sparse attention forward: returns (O bf16 [B,H,N,D], LSE fp32 [B,H,N])."""
    _require_bf16_cuda(q, k, v)
    sh = _shape(q, block)
    if scale is None:
        scale = 1.0 / math.sqrt(sh.D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    _check("bsa_forward", lib().bsa_forward(
        ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(row_ptr), _ptr(col_idx), _ptr(out),
        _ptr(lse), float(scale), int(bool(causal)), _stream(stream)))
    return out, lse


def forward_ex(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, row_ptr: torch.Tensor,
               col_idx: torch.Tensor, block: int, scale: Optional[float] = None, causal: bool = False,
               row_flags: Optional[torch.Tensor] = None, q_block_offset: int = 0,
               out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
               out_dtype=torch.bfloat16, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """The forward with its geometry spelled out: q [B,H,Nq,D] and k, v
    [B,H,Nk,D] may differ in length (a query shard against its local plus
    received key blocks); query block i sits at key-block position
    i + q_block_offset for the causal cut; row_flags (uint8 per CSR row, bit 0)
    lifts the causal cut for single rows; out_dtype torch.float32 writes O in
    fp32 (partial results to merge).  Returns (O [B,H,Nq,D], LSE [B,H,Nq])."""
    _require_bf16_cuda(q, k, v)
    if q.dim() != 4 or k.shape != v.shape or k.dim() != 4 or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("expected q [B,H,Nq,D] and k, v [B,H,Nk,D]")
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if Nq % block or Nk % block:
        raise ValueError("query and key lengths must be multiples of the block size")
    if row_flags is not None and (not row_flags.is_cuda or row_flags.dtype != torch.uint8
                                  or row_flags.numel() != B * H * (Nq // block)):
        raise ValueError("row_flags: uint8 CUDA tensor with one entry per CSR row")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out_dtype: torch.bfloat16 or torch.float32")
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if out.dtype != out_dtype or out.shape != q.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of q's shape in out_dtype")
    if lse is None:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    a = _ForwardArgs(B, H, D, int(block), Nq // block, Nk // block, int(q_block_offset),
                     q.data_ptr(), k.data_ptr(), v.data_ptr(), row_ptr.data_ptr(), col_idx.data_ptr(),
                     row_flags.data_ptr() if row_flags is not None else None, out.data_ptr(), lse.data_ptr(),
                     float(scale), int(bool(causal)), int(out_dtype == torch.float32))
    _check("bsa_forward_ex", lib().bsa_forward_ex(ctypes.byref(a), _stream(stream)))
    return out, lse


_E4M3_DTYPES = (torch.uint8, torch.float8_e4m3fn)


def _require_byte_cuda(*ts: torch.Tensor) -> None:
    for t in ts:
        if not t.is_cuda or t.dtype not in _E4M3_DTYPES or not t.is_contiguous():
            raise ValueError("expected contiguous uint8 / float8_e4m3fn CUDA tensors")


def quantize_e4m3(x: torch.Tensor, inv_scale: float, out: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """e4m3 codes (uint8, shape of x) of x * inv_scale: fp32 product, round to
    nearest even, saturate to +-448.  x: contiguous bf16 CUDA tensor, numel % 16 == 0."""
    _require_bf16_cuda(x)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _require_byte_cuda(out)
    if out.numel() != x.numel():
        raise ValueError("out must have x's number of elements")
    _check("bsa_quantize_e4m3", lib().bsa_quantize_e4m3(_ptr(x), _ptr(out), x.numel(), float(inv_scale),
                                                        _stream(stream)))
    return out


def forward_fp8(q8: torch.Tensor, k8: torch.Tensor, v: torch.Tensor, row_ptr: torch.Tensor,
                col_idx: torch.Tensor, block: int, q_descale: float, k_descale: float,
                scale: Optional[float] = None, causal: bool = False, out: Optional[torch.Tensor] = None,
                lse: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """The forward with FP8 scores: q8, k8 e4m3 codes [B,H,N,D] (uint8 or
    float8_e4m3fn), logits (q8 . k8) * q_descale * k_descale * scale; v bf16.
    Returns (O bf16 [B,H,N,D], LSE fp32 [B,H,N])."""
    _require_byte_cuda(q8, k8)
    _require_bf16_cuda(v)
    sh = _shape(v, block)
    if tuple(q8.shape) != tuple(v.shape) or tuple(k8.shape) != tuple(v.shape):
        raise ValueError("q8, k8 and v must have one shape")
    if scale is None:
        scale = 1.0 / math.sqrt(sh.D)
    if out is None:
        out = torch.empty_like(v)
    if lse is None:
        lse = torch.empty(v.shape[:3], dtype=torch.float32, device=v.device)
    _check("bsa_forward_fp8", lib().bsa_forward_fp8(
        ctypes.byref(sh), _ptr(q8), _ptr(k8), _ptr(v), _ptr(row_ptr), _ptr(col_idx), _ptr(out), _ptr(lse),
        float(q_descale), float(k_descale), float(scale), int(bool(causal)), _stream(stream)))
    return out, lse


def quantize_e4m3_blocks(x: torch.Tensor, block: int, out: Optional[torch.Tensor] = None,
                         descale: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-(head, block) e4m3 codes of x [B,H,N,D] bf16: returns (codes uint8
    [B,H,N,D], descale fp32 [B,H,N/block]); x ~ codes * descale of its block."""
    _require_bf16_cuda(x)
    sh = _shape(x, block)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if descale is None:
        descale = torch.empty((sh.B, sh.H, sh.N // block), dtype=torch.float32, device=x.device)
    _require_byte_cuda(out)
    _check("bsa_quantize_e4m3_blocks", lib().bsa_quantize_e4m3_blocks(ctypes.byref(sh), _ptr(x), _ptr(out),
                                                                      _ptr(descale), _stream(stream)))
    return out, descale


def forward_fp8_blocks(q8: torch.Tensor, k8: torch.Tensor, v: torch.Tensor, q_descale: torch.Tensor,
                       k_descale: torch.Tensor, row_ptr: torch.Tensor, col_idx: torch.Tensor, block: int,
                       scale: Optional[float] = None, causal: bool = False, out: Optional[torch.Tensor] = None,
                       lse: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """The forward with FP8 scores and one descale factor per (head, block):
    logits (q8 . k8) * q_descale[i] * k_descale[j] * scale."""
    _require_byte_cuda(q8, k8)
    _require_bf16_cuda(v)
    sh = _shape(v, block)
    nblk = sh.B * sh.H * (sh.N // block)
    for t in (q_descale, k_descale):
        if not t.is_cuda or t.dtype != torch.float32 or t.numel() != nblk or not t.is_contiguous():
            raise ValueError("descale factors: contiguous fp32 CUDA tensors with one entry per (head, block)")
    if scale is None:
        scale = 1.0 / math.sqrt(sh.D)
    if out is None:
        out = torch.empty_like(v)
    if lse is None:
        lse = torch.empty(v.shape[:3], dtype=torch.float32, device=v.device)
    _check("bsa_forward_fp8_blocks", lib().bsa_forward_fp8_blocks(
        ctypes.byref(sh), _ptr(q8), _ptr(k8), _ptr(v), _ptr(q_descale), _ptr(k_descale), _ptr(row_ptr),
        _ptr(col_idx), _ptr(out), _ptr(lse), float(scale), int(bool(causal)), _stream(stream)))
    return out, lse


def backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor, dout: torch.Tensor,
             lse: torch.Tensor, row_ptr: torch.Tensor, col_idx: torch.Tensor, block: int,
             scale: Optional[float] = None, causal: bool = False, stream=None,
             row_flags: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """dQ, dK, dV of sum(dout * out) for the attention `forward` computed with
    the same CSR (out, lse are its results).  row_flags: the forward's per-row
    causal flags (uint8 per CSR row, bit 0 lifts the causal cut), if it had
    any (pattern_row_flags)."""
    _require_bf16_cuda(q, k, v, out, dout)
    sh = _shape(q, block)
    if scale is None:
        scale = 1.0 / math.sqrt(sh.D)
    if row_flags is not None and (not row_flags.is_cuda or row_flags.dtype != torch.uint8
                                  or row_flags.numel() != sh.B * sh.H * (sh.N // sh.block)):
        raise ValueError("row_flags: uint8 CUDA tensor with one entry per CSR row")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    _check("bsa_backward_ex", lib().bsa_backward_ex(
        ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(row_ptr),
        _ptr(col_idx), col_idx.numel(), _ptr(row_flags), _ptr(dq), _ptr(dk), _ptr(dv), float(scale),
        int(bool(causal)), _stream(stream)))
    return dq, dk, dv


def validate_csr(q_shape, block: int, row_ptr: torch.Tensor, col_idx: torch.Tensor,
                 stream=None) -> int:
    """Debug CSR check; returns the error bits (synchronises)."""
    B, H, N, D = q_shape
    sh = _Shape(B, H, N, D, int(block))
    err = torch.zeros(1, dtype=torch.int32, device=row_ptr.device)
    _check("bsa_validate_csr", lib().bsa_validate_csr(ctypes.byref(sh), _ptr(row_ptr), _ptr(col_idx),
                                                      _ptr(err), _stream(stream)))
    return int(err.item())


def device_error() -> int:
    """Read and clear the device error word (synchronises the device)."""
    code = ctypes.c_int32(0)
    st = lib().bsa_device_error(ctypes.byref(code))
    if st not in (BSA_OK, -5):
        _check("bsa_device_error", st)
    return int(code.value)


def release_workspace() -> None:
    lib().bsa_release_workspace()


def set_wait_limit(ns: int) -> None:
    """Limit (nanoseconds) of every pipeline wait inside the kernels launched
    after this call; a longer wait aborts the launch and sets bit 1 of the
    device error word.  0 restores the default (2 s)."""
    _check("bsa_set_wait_limit", lib().bsa_set_wait_limit(int(ns)))


def get_wait_limit() -> int:
    return int(lib().bsa_get_wait_limit())


def debug_stall_next_forward(n_items: int) -> None:
    """Test hook: the next forward-family call hands out at most n_items work
    items per CTA and then stalls until the wait limit runs out (-1 cancels)."""
    _check("bsa_debug_stall_next_forward", lib().bsa_debug_stall_next_forward(int(n_items)))


def forward_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, row_ptr: torch.Tensor,
                    col_idx: torch.Tensor, block: int, scale: Optional[float] = None, causal: bool = False,
                    out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                    stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """bsa_forward_noalloc: the forward with the library allocating nothing
    (its scratch is a fixed array inside libbsa.so).  Pass `out` and `lse` to
    keep the call free of any allocation on the torch side as well."""
    _require_bf16_cuda(q, k, v)
    sh = _shape(q, block)
    if scale is None:
        scale = 1.0 / math.sqrt(sh.D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    _check("bsa_forward_noalloc", lib().bsa_forward_noalloc(
        ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(row_ptr), _ptr(col_idx), _ptr(out),
        _ptr(lse), float(scale), int(bool(causal)), _stream(stream)))
    return out, lse


def block_sparse_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block: int,
                           pattern: Optional[Pattern] = None, topk: int = 0,
                           include_diag: bool = True, causal: Optional[bool] = None,
                           scale: Optional[float] = None, stream=None):
    """Mask (pattern or content top-k) + forward.  Returns (O, LSE, row_ptr, col_idx)."""
    B, H, N, D = q.shape
    if pattern is not None:
        row_ptr, col_idx = build_mask_csr(pattern, B, H, device=q.device, stream=stream)
        if causal is None:
            causal = pattern.causal
        if pattern.global_rows_noncausal:
            flags = pattern_row_flags(pattern, B, H, device=q.device, stream=stream)
            o, lse = forward_ex(q, k, v, row_ptr, col_idx, block, scale=scale, causal=bool(causal),
                                row_flags=flags, stream=stream)
            return o, lse, row_ptr, col_idx
    elif topk > 0:
        row_ptr, col_idx = topk_blocks(q, k, block, topk, include_diag, stream=stream)
    else:
        raise ValueError("give a pattern or topk > 0")
    o, lse = forward(q, k, v, row_ptr, col_idx, block, scale=scale, causal=bool(causal), stream=stream)
    return o, lse, row_ptr, col_idx
