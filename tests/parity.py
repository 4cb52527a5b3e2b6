"""Comparison helpers shared by the GPU parity tests (test infrastructure).

Tolerances, fixed before any GPU result was seen:
  attention, float32 output : |gpu - oracle| <= 2e-3 per element
      (bf16 inputs, fp32 accumulation; the oracle accumulates in float64);
  attention, bf16 output    : |gpu - oracle| <= 2e-3 + 2^-8 |oracle|
      (plus the half-ulp of round-to-nearest into bf16's 8-bit significand);
  sampler tokens            : bit-exact wherever the oracle's Gumbel margin
      (best minus second-best perturbed score, float64) is >= 1e-5; the GPU
      computes the perturbation in fp32, whose error is far below 1e-5;
  top-k sets                : bit-exact (support of the probabilities);
  probabilities             : |gpu - oracle| <= 1e-6 + 2e-5 |oracle|
      (fp32 expf and a sum of at most 2048 fp32 terms).
"""
from __future__ import annotations

import math

import numpy as np
import torch

ATTN_ABS_TOL = 2e-3
MARGIN_EXCLUSION = 1e-5


def attn_tolerance(ref: np.ndarray, out_dtype: torch.dtype) -> np.ndarray:
    if out_dtype == torch.float32:
        return np.full_like(ref, ATTN_ABS_TOL)
    return ATTN_ABS_TOL + 2.0 ** -8 * np.abs(ref)


def assert_attn_close(got: torch.Tensor, ref: np.ndarray, what: str = "attention"):
    g = got.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(ref).all(), f"{what}: oracle produced non-finite values"
    err = np.abs(g - ref)
    tol = attn_tolerance(ref, got.dtype)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance, max err {err.max():.3e}, "
                             f"first at {idx.tolist()}")
    return float(err.max())


def assert_tokens_match(got: torch.Tensor | np.ndarray, ref: dict, what: str = "tokens",
                        max_excluded: int | None = None):
    """Tokens equal wherever the oracle's margin is >= MARGIN_EXCLUSION.  At most max_excluded draws (default:
    1% of all draws, at least 1) may fall under the exclusion, so that a comparison cannot pass by skipping."""
    g = got.cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    compare = ref["margins"] >= MARGIN_EXCLUSION
    n_excl = int((~compare).sum())
    limit = max(1, compare.size // 100) if max_excluded is None else max_excluded
    if n_excl > limit:
        raise AssertionError(f"{what}: {n_excl} of {compare.size} draws fall under the margin exclusion "
                             f"(at most {limit} allowed)")
    mism = compare & (g != ref["tokens"])
    if mism.any():
        idx = np.argwhere(mism)[:5]
        raise AssertionError(f"{what}: {int(mism.sum())} of {int(compare.sum())} compared draws differ; "
                             f"first at {idx.tolist()}: gpu {g[tuple(idx[0])]} oracle {ref['tokens'][tuple(idx[0])]}")
    return int(compare.sum()), int((~compare).sum())


def assert_probs_match(got: torch.Tensor, ref: dict, what: str = "probs"):
    g = got.cpu().numpy().astype(np.float64)
    r = ref["probs"]
    support_g, support_r = g != 0, r != 0
    if not np.array_equal(support_g, support_r):
        idx = np.argwhere(support_g != support_r)[:5]
        raise AssertionError(f"{what}: top-k sets differ at {idx.tolist()}")
    err = np.abs(g - r)
    tol = 1e-6 + 2e-5 * np.abs(r)
    if not (err <= tol).all():
        raise AssertionError(f"{what}: max err {err.max():.3e}")


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)
