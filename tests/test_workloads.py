"""The seeded input generator: shapes, dtypes, determinism, thread independence and the
planted ties of the small tie workload. CPU only."""

import numpy as np
import torch

from draft_candidate_selector_gb300 import workloads as wl


def test_tiny_shapes_and_determinism():
    a = wl.make_inputs("tiny", seed=0)
    b = wl.make_inputs("tiny", seed=0)
    w = a.workload
    assert a.logits.shape == (w.R, w.S, w.V) and a.logits.dtype == np.float32
    assert a.hidden.shape == (w.R, w.S, w.H) and a.hidden.dtype == torch.bfloat16
    assert a.w_proj.shape == (w.rank, w.H)
    assert a.pred_cb.shape == (w.V, w.rank) and a.succ_cb.shape == (w.V, w.rank)
    assert a.anchors.shape == (w.R,) and a.anchors.dtype == np.int32
    assert np.all((a.anchors >= 0) & (a.anchors < w.V))
    assert np.array_equal(a.logits, b.logits)
    assert torch.equal(a.hidden, b.hidden) and torch.equal(a.pred_cb, b.pred_cb)
    c = wl.make_inputs("tiny", seed=1)
    assert not np.array_equal(a.logits, c.logits)


def test_thread_count_does_not_change_logits():
    w = wl.custom_workload(3, 15, 8, 4099, 64, 16)
    x1 = wl.make_logits(w, seed=5, threads=1)
    x4 = wl.make_logits(w, seed=5, threads=4)
    assert np.array_equal(x1, x4)


def test_distribution_scales():
    w = wl.custom_workload(4, 8, 8, 8192, 1024, 64, logit_std=4.0)
    inp = wl.make_inputs(w, seed=3)
    assert abs(inp.logits.std() - 4.0) < 0.05
    assert abs(inp.hidden.float().std().item() - 1.0) < 0.02
    assert abs(inp.w_proj.float().std().item() - 1 / 32) < 0.002
    assert abs(inp.pred_cb.float().std().item() - 1 / 8) < 0.002


def test_planted_ties():
    w = wl.WORKLOADS["small_ties"]
    rows = wl.tie_rows(w, 0)
    assert len(rows) == 1                       # ceil(1% of 56 rows)
    x = wl.make_logits(w, seed=0).reshape(w.rows, w.V)
    for r in rows:
        vals, counts = np.unique(x[r], return_counts=True)
        top2 = vals[-2:]
        assert counts[-1] == w.K // 2           # group A at the top
        assert counts[-2] == w.K + 3            # group B straddles the K-th place
        assert top2[1] == top2[0] + 1


def test_softcap_and_zipf_recipes():
    w = wl.custom_workload(2, 3, 8, 5000, 32, 8, logits="normal_softcap", logit_std=5.0,
                           softcap=30.0)
    x = wl.make_logits(w, seed=0)
    assert np.all(np.abs(x) < 30.0)
    z = wl.custom_workload(2, 3, 8, 5000, 32, 8, logits="zipf_gumbel")
    xz = wl.make_logits(z, seed=0)
    assert np.isfinite(xz).all() and xz.max() < 15 and xz.min() > -20


def test_algorithmic_bytes_large():
    w = wl.WORKLOADS["gemma_large"]
    b = w.algorithmic_bytes()
    assert b["logits"] == 512 * 15 * 262144 * 4
    total = sum(b.values())
    assert 8.3e9 < total < 8.5e9
