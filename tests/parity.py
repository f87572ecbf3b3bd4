"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded bf16 inputs, and compare.

Tolerances (fixed by the target): max |dO| <= 1e-2, mean |dO| <= 1e-3,
max |dLSE| <= 1e-3; CSR and top-k selections bit-exact.
"""

from __future__ import annotations

import numpy as np
import torch

import bsa_inputs
import oracle

TOL_MAX_O = 1e-2
TOL_MEAN_O = 1e-3
TOL_LSE = 1e-3


def bits(t: torch.Tensor) -> np.ndarray:
    return bsa_inputs.bf16_bits(t.cpu())


def oracle_csr(w, q_cpu=None, k_cpu=None):
    if w.is_topk:
        rp, ci, _ = oracle.topk_csr(bits(q_cpu), bits(k_cpu), w.block, w.topk, w.include_diag)
        return rp, ci
    rp1, ci1 = oracle.Pattern.from_workload(w).csr()
    return oracle.replicate_csr(rp1, ci1, w.B * w.H)


def gpu_pattern(w):
    import block_sparse_flashattention_bsa_gb300 as bsa
    return bsa.Pattern(w.n_blocks, w.window_left, w.window_right, w.causal, w.global_blocks,
                       w.global_rows_attend_all)


def gpu_csr(w, q_dev, k_dev):
    import block_sparse_flashattention_bsa_gb300 as bsa
    if w.is_topk:
        rp, ci = bsa.topk_blocks(q_dev, k_dev, w.block, w.topk, w.include_diag)
        return rp, ci[: int(rp[-1].item())]
    return bsa.build_mask_csr(gpu_pattern(w), w.B, w.H, device=q_dev.device)


def compare(o_gpu: torch.Tensor, lse_gpu: torch.Tensor, O_ref: np.ndarray, L_ref: np.ndarray,
            rows: np.ndarray, D: int):
    """o_gpu [.., N, D] bf16 and lse_gpu [.., N] fp32 on any device; reference
    rows given as flat row ids.  Returns (max|dO|, mean|dO|, max|dLSE|, max|O|)."""
    rows_t = torch.as_tensor(rows, dtype=torch.int64)
    o = o_gpu.reshape(-1, D).index_select(0, rows_t.to(o_gpu.device)).double().cpu().numpy()
    l = lse_gpu.reshape(-1).index_select(0, rows_t.to(lse_gpu.device)).double().cpu().numpy()
    d_o = np.abs(o - O_ref)
    both_inf = np.isneginf(l) & np.isneginf(L_ref)
    d_l = np.where(both_inf, 0.0, np.abs(l - L_ref))
    return float(d_o.max()), float(d_o.mean()), float(d_l.max()), float(np.abs(O_ref).max())


def assert_close(stats, what=""):
    mx, mean, dl, omax = stats
    assert mx <= TOL_MAX_O, "%s max|dO| %.3g > %g (max|O| %.3g)" % (what, mx, TOL_MAX_O, omax)
    assert mean <= TOL_MEAN_O, "%s mean|dO| %.3g > %g" % (what, mean, TOL_MEAN_O)
    assert dl <= TOL_LSE, "%s max|dLSE| %.3g > %g" % (what, dl, TOL_LSE)


def run_forward_case(w, rows=None, data=None, csr=None, causal=None, check_csr=True):
    """Full path for workload w: CSR on the GPU (bit-exact vs the oracle's),
    forward on the GPU, oracle on `rows` (default: all rows)."""
    import block_sparse_flashattention_bsa_gb300 as bsa
    if data is None:
        data = bsa_inputs.make_qkv(w)
    q, k, v = data["q"], data["k"], data["v"]
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    if csr is None:
        rp_ref, ci_ref = oracle_csr(w, q, k)
        rp_g, ci_g = gpu_csr(w, qd, kd)
        if check_csr:
            np.testing.assert_array_equal(rp_g.cpu().numpy(), rp_ref)
            np.testing.assert_array_equal(ci_g.cpu().numpy(), ci_ref)
        rp_use, ci_use = rp_g, ci_g
    else:
        rp_ref, ci_ref = csr
        rp_use = torch.as_tensor(rp_ref, dtype=torch.int32, device=dev)
        ci_use = torch.as_tensor(ci_ref if len(ci_ref) else np.zeros(1, np.int32), dtype=torch.int32,
                                 device=dev)
    causal = w.causal if causal is None else causal
    o, lse = bsa.forward(qd, kd, vd, rp_use, ci_use, w.block, scale=w.scale, causal=causal)
    torch.cuda.synchronize()
    err = bsa.device_error()
    if rows is None:
        rows = np.arange(w.B * w.H * w.N, dtype=np.int64)
    O_ref, L_ref = oracle.attention_rows(bits(q), bits(k), bits(v), rp_ref, ci_ref, w.block, w.scale,
                                         causal, rows=rows)
    return compare(o, lse, O_ref, L_ref, rows, w.D), err


def random_ex_specs(rng, nb, n):
    """n random dilated-window / stride / global pattern specs over nb blocks."""
    specs = []
    for _ in range(n):
        nw = int(rng.integers(0, 5))
        specs.append(dict(
            n_blocks=nb,
            windows=[[int(rng.integers(0, 5)), int(rng.integers(0, 5)), int(rng.integers(1, 6))]
                     for _ in range(nw)],
            stride=int(rng.choice([0, 0, 1, 3, 7, nb + 3])),
            causal=bool(rng.integers(0, 2)),
            global_blocks=sorted(set(int(x) for x in rng.integers(0, nb, size=int(rng.integers(0, 4))))),
            global_rows_attend_all=bool(rng.integers(0, 2))))
    return specs


def ex_pair(spec):
    """The same dilated-window / stride pattern for the library and the oracle."""
    import block_sparse_flashattention_bsa_gb300 as bsa
    args = (spec["n_blocks"], [tuple(w) for w in spec["windows"]], spec["stride"], spec["causal"],
            spec["global_blocks"], spec["global_rows_attend_all"])
    return bsa.PatternEx(*args), oracle.PatternEx(*args)
