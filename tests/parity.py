"""Shared helpers of the GPU parity tests: moving seeded inputs to the device, calling
the oracle on the same bytes, and the comparison rules.

Tolerances:
  * candidate ids: bit-exact;
  * unary logits and fp32 edge scores: |gpu - ref| <= 2e-3 * (1 + |ref|), NaN where the
    reference is NaN;
  * the bf16 projection: at most one bf16 step from the oracle. The oracle rounds an
    exact sum once; the kernel rounds an fp32 sum, which can land on the other side of a
    rounding boundary.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from draft_candidate_selector_gb300 import workloads as wl

RTOL = 2e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (any device)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_device(inp: wl.Inputs, dev) -> dict:
    return dict(
        logits=torch.from_numpy(inp.logits).to(dev),
        hidden=inp.hidden.to(dev),
        w_proj=inp.w_proj.to(dev),
        pred_cb=inp.pred_cb.to(dev),
        succ_cb=inp.succ_cb.to(dev),
        anchors=torch.from_numpy(inp.anchors).to(dev),
    )


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str) -> None:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(gpu), nan_ref), f"{what}: NaN positions differ"
    g, r = gpu[~nan_ref], ref[~nan_ref]
    same_inf = (g == r)
    err = np.where(same_inf, 0.0, np.abs(g - r))
    bound = RTOL * (1.0 + np.abs(r))
    bad = ~(err <= bound)
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} values out of tolerance; "
                             f"first: gpu={g[i]!r} ref={r[i]!r} err={err[i]:.3g}")


def assert_ids_equal(gpu: np.ndarray, ref: np.ndarray, what: str) -> None:
    gpu = np.asarray(gpu)
    ref = np.asarray(ref)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    if not np.array_equal(gpu, ref):
        idx = np.argwhere(gpu != ref)[0]
        raise AssertionError(f"{what}: ids differ at {tuple(idx)}: gpu={gpu[tuple(idx[:-1])]} "
                             f"ref={ref[tuple(idx[:-1])]}")


def _ordered(b: np.ndarray) -> np.ndarray:
    """bf16 bits -> integers in value order, so adjacent bf16 values differ by 1."""
    b = b.astype(np.int32)
    return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + b)


def assert_bf16_within_one_step(gpu_bits: np.ndarray, ref_bits: np.ndarray, what: str,
                                max_fraction: float = 0.01) -> None:
    d = np.abs(_ordered(gpu_bits) - _ordered(ref_bits))
    assert d.max(initial=0) <= 1, f"{what}: a value is {d.max()} bf16 steps from the oracle"
    frac = float((d > 0).mean()) if d.size else 0.0
    assert frac <= max_fraction, f"{what}: {frac:.4f} of values differ by one bf16 step"


def oracle_topk_rows(logits: np.ndarray, K: int, rows: np.ndarray):
    """Oracle top-k of selected flat rows of logits [R, S, V]."""
    flat = logits.reshape(-1, logits.shape[-1])
    return oracle.topk(flat[rows], K)


def sample_rows(n_rows: int, k: int, seed: int, extra=()) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = set(int(x) for x in rng.choice(n_rows, size=min(k, n_rows), replace=False))
    pick.update([0, n_rows - 1, n_rows // 2])
    pick.update(int(x) for x in extra if 0 <= x < n_rows)
    return np.array(sorted(pick), dtype=np.int64)


def sample_requests(R: int, k: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = set(int(x) for x in rng.choice(R, size=min(k, R), replace=False))
    pick.update([0, R - 1])
    return np.array(sorted(pick), dtype=np.int64)
