"""Shared helpers of the GPU parity tests: moving seeded inputs to the device, calling
the oracle on the same bytes, and the comparison rules.

Tolerances:
  * candidate ids: bit-exact;
  * unary logits and fp32 edge scores: |gpu - ref| <= 2e-3 * (1 + |ref|), NaN where the
    reference is NaN;
  * the bf16 projection h = bf16(sum_i W[j,i] x[i]), where s is the exact sum and
    A = sum_i |W[j,i] x[i]|:
      - every entry satisfies |h - s| <= 2^-8 |s| + H 2^-24 A. That is the bf16 rounding
        plus the worst-case error of an fp32 sum of H products (H unit roundoffs on the
        sum of magnitudes). Near zero, where a bf16 step is tiny, only the second term
        matters;
      - at least 99% of entries are within one bf16 step of the oracle's correctly
        rounded value;
      - the RMS of (h - s) is at most 2^-9 of the RMS of s (half a bf16 step).
    A wrong tile, swizzle or K block moves many entries by far more and fails the last
    two checks.
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
    with np.errstate(invalid="ignore"):      # inf - inf where both are the same infinity
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


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_projection(gpu_bits: np.ndarray, hidden_bits: np.ndarray, w_bits: np.ndarray,
                      what: str) -> None:
    """The projection tolerance described in the module docstring."""
    H = hidden_bits.shape[-1]
    ref_bits, exact = oracle.projection(hidden_bits, w_bits, want_exact=True)
    x = bits_to_f64(hidden_bits).reshape(-1, H)
    w = bits_to_f64(w_bits)
    A = (np.abs(x) @ np.abs(w).T).reshape(exact.shape)
    g = bits_to_f64(gpu_bits).reshape(exact.shape)
    err = np.abs(g - exact)
    bound = 2.0 ** -8 * np.abs(exact) + H * 2.0 ** -24 * A
    steps = np.abs(_ordered(np.asarray(gpu_bits).reshape(exact.shape)) - _ordered(ref_bits))
    near = float((steps <= 1).mean())
    rms_rel = float(np.sqrt(np.mean((g - exact) ** 2)) / max(np.sqrt(np.mean(exact ** 2)), 1e-300))
    use = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0), np.where(err > 0, np.inf, 0.0))
    stats = (f"max |h-s| = {err.max():.3g}, max bound use = {use.max():.3g}, "
             f"within one step: {near:.5f}, rms rel err = {rms_rel:.3g}")
    assert np.all(err <= bound), f"{what}: entry outside the summation bound; {stats}"
    assert near >= 0.99, f"{what}: too many entries off by more than one bf16 step; {stats}"
    assert rms_rel <= 2.0 ** -9, f"{what}: RMS error above half a bf16 step; {stats}"


def sample_rows(n_rows: int, k: int, seed: int, extra=()) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = set(int(x) for x in rng.choice(n_rows, size=min(k, n_rows), replace=False))
    pick.update([0, n_rows - 1, n_rows // 2])
    pick.update(int(x) for x in extra if 0 <= x < n_rows)
    return np.array(sorted(pick), dtype=np.int64)


def assert_lmhead_valid(gpu_ids: np.ndarray, gpu_unary: np.ndarray, hidden_bits: np.ndarray,
                        lm_head_bits: np.ndarray, K: int, what: str, softcap: float = 0.0,
                        scale: float = 1.0) -> float:
    """Candidates from fp32 tensor-core logits, checked against the exact logits.

    tol_v = 2 * H * 2^-24 * sum_i |x_i w_vi| bounds how far two fp32 sums can reorder.
    (a) every chosen id is in range and distinct, and its exact logit is within tol of the
        exact K-th best;
    (b) every id that beats the exact (K+1)-th best by more than tol is chosen;
    (c) the chosen order never puts a logit below the next one by more than tol;
    (d) the unary values are within 2e-3 * (1 + |ref|) of the processed exact logits.
    Returns the fraction of rows whose ids equal the oracle's exactly.
    """
    H = hidden_bits.shape[-1]
    V = lm_head_bits.shape[0]
    ax = np.abs(bits_to_f64(hidden_bits).reshape(-1, H))
    ref_ids, _, exact = oracle.lmhead_topk(hidden_bits.reshape(-1, H), lm_head_bits, K,
                                           softcap=softcap, scale=scale, want_logits=True)
    tol = np.empty((ax.shape[0], V))
    for v0 in range(0, V, 4096):             # in chunks: the LM head may be gigabytes
        aw = np.abs(bits_to_f64(lm_head_bits[v0:v0 + 4096]).reshape(-1, H))
        tol[:, v0:v0 + aw.shape[0]] = 2.0 * H * 2.0 ** -24 * (ax @ aw.T)
    gi = np.asarray(gpu_ids).reshape(-1, K)
    gu = np.asarray(gpu_unary, dtype=np.float64).reshape(-1, K)
    same = 0
    for r in range(gi.shape[0]):
        ids = gi[r]
        assert np.all((ids >= 0) & (ids < V)), f"{what}: row {r} has an id out of range"
        assert len(set(ids.tolist())) == K, f"{what}: row {r} repeats an id"
        L = exact[r]
        order = ref_ids[r]
        kth = L[order[K - 1]]
        nxt = np.sort(L)[::-1][K] if V > K else -np.inf
        t = tol[r]
        assert np.all(L[ids] + t[ids] + t[order[K - 1]] >= kth), f"{what}: row {r} chose a loser"
        must = np.nonzero(L > nxt + t + t.max())[0]
        assert set(must.tolist()) <= set(ids.tolist()), f"{what}: row {r} missed a clear winner"
        assert np.all(L[ids[:-1]] + t[ids[:-1]] + t[ids[1:]] >= L[ids[1:]]), \
            f"{what}: row {r} out of order"
        v = L[ids].astype(np.float32).astype(np.float64)
        ref_u = (softcap * np.tanh(v / softcap) if softcap > 0 else v) * scale
        assert np.all(np.abs(gu[r] - ref_u) <= RTOL * (1 + np.abs(ref_u)) + 2 * t[ids] * scale), \
            f"{what}: row {r} unary off"
        same += int(np.array_equal(ids, order))
    return same / gi.shape[0]


def assert_lmhead_valid_every_row(ids: torch.Tensor, unary: torch.Tensor, hidden: torch.Tensor,
                                  lm_head: torch.Tensor, K: int, what: str,
                                  softcap: float = 0.0, scale: float = 1.0,
                                  chunk: int = 256) -> None:
    """Every row of an LM-head top-k at full size, against plain fp32 logits on the device.

    The reference f is torch's fp32 GEMM of the bf16 inputs widened to fp32 (TF32 off): each
    product is exact and only the fp32 sums round, as in the kernel. With
    t_v = 2 * H * 2^-24 * sum_i |x_i w_vi| (the tolerance of assert_lmhead_valid), the
    kernel's sum k_v and f_v each lie within t_v / 2 of the exact logit. The kernel keeps
    k_v <= k_c for every v left out and c chosen, so f_v - t_v <= f_c + t_c. Checked on every
    row, with a factor 2 of margin on t:
    (a) the ids are in range and distinct;
    (b) max over left-out v of (f_v - 2 t_v) <= min over chosen c of (f_c + 2 t_c);
    (c) the unary values are non-increasing, and equal raw values keep ids ascending;
    (d) each unary value is within 2 scale t_c (plus 1e-5 relative, the fp32 soft cap) of the
        processed reference logit of its id.
    """
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        H = hidden.shape[-1]
        V = lm_head.shape[0]
        x = hidden.reshape(-1, H)
        n = x.shape[0]
        gi = ids.reshape(n, K).long()
        gu = unary.reshape(n, K).float()
        assert bool(((gi >= 0) & (gi < V)).all()), f"{what}: an id out of range"
        srt = gi.sort(dim=1).values
        assert bool((srt[:, 1:] != srt[:, :-1]).all()), f"{what}: a row repeats an id"
        assert bool((gu[:, 1:] <= gu[:, :-1]).all()), f"{what}: unary values not non-increasing"
        if softcap == 0.0 and scale == 1.0:
            tie = gu[:, 1:] == gu[:, :-1]
            assert bool((~tie | (gi[:, 1:] > gi[:, :-1])).all()), \
                f"{what}: equal values out of id order"
        w32 = lm_head.float()
        wabs = w32.abs()
        for r0 in range(0, n, chunk):
            xc = x[r0:r0 + chunk].float()
            f = xc @ w32.t()                                           # [rows, V] fp32
            t = (2.0 * H * 2.0 ** -24) * (xc.abs() @ wabs.t())         # [rows, V]
            ic = gi[r0:r0 + chunk]
            fc, tc = f.gather(1, ic), t.gather(1, ic)
            low = f - 2.0 * t
            low.scatter_(1, ic, float("-inf"))
            bad = low.max(dim=1).values > (fc + 2.0 * tc).min(dim=1).values
            assert not bool(bad.any()), \
                f"{what}: row {r0 + int(bad.nonzero()[0])} left out a clear winner"
            ref_u = (softcap * torch.tanh(fc / softcap) if softcap > 0 else fc) * scale
            uc = gu[r0:r0 + chunk]
            off = (uc - ref_u).abs() > 2.0 * scale * tc + 1e-5 * (1 + ref_u.abs())
            assert not bool(off.any()), \
                f"{what}: row {r0 + int(off.nonzero()[0, 0])} unary off the reference"
            del f, t, low
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def float_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bits of float32 values that are exactly representable in bf16 (checked)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0)
    return (u >> 16).astype(np.uint16)
