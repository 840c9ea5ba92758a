"""Shared helpers for the GPU parity tests (imported by tests only)."""

import numpy as np
import pytest
import torch

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}   # max-abs on attention outputs
# The tensor-core decode of grouped bf16 heads: scores and the P.V product accumulate in fp32
# from bf16 operands (q, K and V are bf16 values, so exact), and P goes into the product as a
# bf16 pair hi + lo: hi = bf16(P) leaves at most 2^-9 P, lo = bf16(P - hi) at most 2^-9 of
# that, so each weight is off by at most 2^-18 P and the output by at most 2^-18 * max|v|
# (1.7e-5 for the unit-variance values here, |v| < 4.5) plus the fp32 roundings.  Measured
# worst against the fp64 oracle: 1.8e-6 (ragged lengths, D 64/128/256, groups 2-8, and the
# SnapKV, long-context and grouped-H2O full-size layers).
TOL_SPLIT_P = 2e-5


def lib():
    from kv_cache_compression_kvc_gb300 import build, kvc
    build.build()
    kvc.load()
    return kvc


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of stored values (fp32 or bf16) to float64 on the host."""
    return t.detach().to("cpu").double().numpy()


def assert_close(got, ref, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"
    return err


def assert_rel(got, ref, rtol, atol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bad = np.abs(got - ref) > rtol * np.abs(ref) + atol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside rtol {rtol} atol {atol}; "
                           f"worst {float(np.max(np.abs(got - ref))):.3e}")


def topk_sets_agree(idx_gpu, idx_ref, score_ref, k, band=1e-4):
    """End-to-end index check: the two selections may differ only at positions whose oracle
    score lies within a relative band of the k-th largest oracle score (near-ties decided by
    rounding).  Returns the number of such tolerated differences."""
    a, b = set(int(x) for x in idx_gpu), set(int(x) for x in idx_ref)
    diff = a ^ b
    if not diff:
        return 0
    s = np.asarray(score_ref, dtype=np.float64)
    kth = np.sort(s)[::-1][k - 1]
    for i in diff:
        if i >= len(s) or abs(s[i] - kth) > band * abs(kth):
            raise AssertionError(f"index {i} differs and its score {s[i] if i < len(s) else None} "
                                 f"is not within {band} of the threshold {kth}")
    return len(diff)


def cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
