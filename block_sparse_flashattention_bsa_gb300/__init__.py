"""Block-sparse FlashAttention forward for GB300 (sm_103a).

A thin ctypes binding over ``libbsa.so`` (declared in ``include/bsa.h``).
Every step of the computation runs in the library's CUDA kernels; this module
only marshals torch tensors (device memory) and the current CUDA stream into
the C ABI and turns status codes into exceptions.  There is no fallback: if
the library is missing or the device is not sm_103, calls raise.

Entry points (same names as the C ABI, minus the ``bsa_`` prefix):

* :func:`build_mask_csr`  pattern (window / globals / causal) -> block CSR
* :func:`build_mask_csr_heads`  per-head patterns (:class:`PatternEx`: dilated
  windows, stride, globals, causal) -> block CSR
* :func:`topk_blocks`     content-based block CSR (pooled Q.K top-k + diagonal)
* :func:`forward`         block-sparse attention forward -> (O bf16, LSE fp32)
* :func:`forward_ex`      the same with key blocks apart from the query blocks
  (sequence shards), a query offset and per-row causal flags
  (:func:`pattern_row_flags`: global query rows of a causal model)
* :func:`forward_fp8`     the same with FP8 scores (e4m3 Q and K, per-tensor
  descale factors); :func:`quantize_e4m3` makes the e4m3 inputs;
  :func:`forward_fp8_blocks` / :func:`quantize_e4m3_blocks` take one
  descale factor per (head, block)
* :func:`backward`        its gradients (dQ, dK, dV) through the same mask
* :func:`forward_noalloc`  the forward with no allocation by the library
* :func:`validate_csr`, :func:`device_error`, :func:`pattern_nnz`
* :func:`set_wait_limit` (hang detection), :func:`debug_stall_next_forward`
  (its test hook)
* :func:`block_sparse_attention`  convenience: mask + forward in one call
"""

from ._binding import (  # noqa: F401
    BsaError,
    Pattern,
    PatternEx,
    backward,
    block_sparse_attention,
    build_mask_csr,
    build_mask_csr_heads,
    debug_stall_next_forward,
    device_error,
    forward,
    forward_ex,
    forward_fp8,
    forward_fp8_blocks,
    forward_noalloc,
    get_wait_limit,
    lib,
    lib_path,
    mask_heads_nnz,
    pattern_nnz,
    pattern_row_flags,
    quantize_e4m3,
    quantize_e4m3_blocks,
    release_workspace,
    set_wait_limit,
    topk_blocks,
    validate_csr,
)
