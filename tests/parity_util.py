"""Helpers shared by the GPU parity tests: host copies, error norms and the
routing comparison rule.

Routing comparison: when both sides compute their own fp32 logits (tensor
cores on the GPU, BLAS on the CPU) the two differ by rounding, so a token
whose K-th and (K+1)-th keys are closer than that difference has two correct
answers.  Such tokens must still get a valid top-K (every selected key at
least every unselected key minus the tolerance); all other tokens must match
exactly.  Routing from the same fp32 logits is compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

BF16_TOL = 5e-3     # normwise relative error of bf16 outputs and gradients


def np32(t):
    return None if t is None else t.detach().float().cpu().numpy()


def host_params(p: dict) -> dict:
    return {k: np32(v) for k, v in p.items()}


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))


def routing_agreement(keys: np.ndarray, idx_gpu: np.ndarray, idx_ref: np.ndarray, tol: float) -> np.ndarray:
    """Boolean mask of tokens whose selected sets agree.  Asserts that every
    disagreeing token is a near tie within ``tol`` and that the GPU's set is
    a valid top-K of the oracle's keys within ``tol``."""
    n, k = idx_ref.shape
    same = (np.sort(idx_gpu, 1) == np.sort(idx_ref, 1)).all(axis=1)
    for t in np.nonzero(~same)[0]:
        sel = np.zeros(keys.shape[1], dtype=bool)
        sel[idx_gpu[t]] = True
        assert len(set(idx_gpu[t].tolist())) == k, f"token {t}: repeated expert"
        assert keys[t, sel].min() >= keys[t, ~sel].max() - tol, f"token {t}: not a top-K within {tol}"
    return same


def to_dev(p: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}


def check_rows(got, want, tol: float, key: str = ""):
    """Normwise relative error of the whole array within ``tol``, and per row
    (token): the 99th percentile of ``||got_t - want_t||`` over the root mean
    square row norm of ``want`` within ``2 * tol``, so that a few wrong rows
    cannot hide in the pooled norm."""
    from oracle_pool import per_token_error
    got, want = np.asarray(got), np.asarray(want)
    e = rel(got, want)
    assert e < tol, (key, e)
    pt = per_token_error(got, want)
    assert np.quantile(pt, 0.99) <= 2 * tol, (key, float(pt.max()), int(np.argmax(pt)))
