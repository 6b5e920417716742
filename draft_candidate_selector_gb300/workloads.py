"""Seeded synthetic workloads for the DFlash2 candidate selector.

This module only draws random inputs. It holds none of the selector's arithmetic:
no top-k, no projection, no edge scores. The tests and the benchmark both take their
inputs from here, so the oracle and the CUDA path always see the same bytes.

Shapes follow the drafter on the "vllm.models.beam.nvidia.dflash2" page:
  * R requests, each with S draft steps. These are the mask positions of a block of
    1 bonus + S mask tokens ("DFlashSpeculator.__init__", query layout).
  * K = selector_top_k and rank = selector_rank
    ("DFlash2BeamModel.__init__", candidate_selector).
  * V = vocab, H = drafter hidden size.

Tensors and layouts. All are row-major and contiguous:
  logits   float32 [R, S, V]   vocab logits, one row per (request, step)
  hidden   bf16    [R, S, H]   drafter hidden states
  w_proj   bf16    [rank, H]   hidden_projection weight, Linear [out, in] convention
  pred_cb  bf16    [V, rank]   predecessor codebook
  succ_cb  bf16    [V, rank]   successor codebook
  anchors  int32   [R]         anchor (bonus) token id of each request

Distributions. "N(0, s)" means a normal with standard deviation s.
  hidden N(0,1); w_proj N(0, 1/sqrt(H)); codebooks N(0, 1/sqrt(rank));
  anchors uniform in [0, V). The logit recipe is chosen per workload (see WORKLOADS).

Random streams. Each tensor, and each block of logit rows, draws from its own numpy
PCG64 stream, keyed by (seed, tensor tag, block index). Blocks are therefore generated
in parallel threads, and the result does not depend on the thread count.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np
import torch

# Tags that key the random streams (arbitrary, fixed).
_TAG_LOGITS = 11
_TAG_HIDDEN = 12
_TAG_W = 13
_TAG_PRED = 14
_TAG_SUCC = 15
_TAG_ANCHOR = 16
_TAG_TIES = 17
_TAG_PERM = 18

# Logit rows per random stream. Fixed, so that the output does not depend on threading.
_ROWS_PER_BLOCK = 16


@dataclass(frozen=True)
class Workload:
    name: str
    R: int
    S: int
    K: int
    V: int
    H: int
    rank: int
    logits: str           # recipe name: "normal", "normal_ties", "zipf_gumbel", "normal_softcap"
    logit_std: float = 1.0
    softcap: float = 0.0
    zipf_s: float = 1.1
    tie_fraction: float = 0.0
    description: str = ""

    @property
    def rows(self) -> int:
        return self.R * self.S

    @property
    def edges_per_call(self) -> int:
        return self.R * self.S * self.K * self.K

    def algorithmic_bytes(self) -> dict:
        """Bytes the method must move once, by tensor.

        Each logit row is read once. Hidden is read once. W is read once. There are
        2K codebook rows per (request, step), or K + 1 at step 0. Ids, unary values,
        the projected state and the edge scores are written once.
        """
        rows, K, rank = self.rows, self.K, self.rank
        gathered_rows = self.R * ((self.S - 1) * 2 * K + (K + 1))
        return {
            "logits": rows * self.V * 4,
            "hidden": rows * self.H * 2,
            "w_proj": self.rank * self.H * 2,
            "gathers": gathered_rows * rank * 2,
            "ids_unary_out": rows * K * 8,
            "h_out": rows * rank * 2,
            "edges_out": rows * K * K * 4,
            "anchors": self.R * 4,
        }


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny", 2, 4, 4, 1024, 256, 16, "normal", logit_std=3.0,
                 description="tiny: R=2 S=4 K=4 V=1024 H=256 rank=16, logits N(0,3)"),
        Workload("small_ties", 8, 7, 8, 32768, 1024, 64, "normal_ties", logit_std=4.0,
                 tie_fraction=0.01,
                 description="R=8 S=7 K=8 V=32768 H=1024 rank=64, logits N(0,4), "
                             "1% of rows with exact ties"),
        Workload("qwen_zipf", 64, 15, 8, 151936, 2048, 128, "zipf_gumbel", zipf_s=1.1,
                 description="R=64 S=15 K=8 V=151936 H=2048 rank=128, "
                             "Gumbel-perturbed Zipf(1.1) logits"),
        Workload("gemma_softcap", 256, 15, 16, 262144, 3840, 128, "normal_softcap",
                 logit_std=5.0, softcap=30.0,
                 description="R=256 S=15 K=16 V=262144 H=3840 rank=128, "
                             "logits 30*tanh(N(0,5)/30)"),
        Workload("gemma_large", 512, 15, 32, 262144, 5376, 256, "normal", logit_std=5.0,
                 description="R=512 S=15 K=32 V=262144 H=5376 rank=256, logits N(0,5)"),
    ]
}

# The order in which the five workloads are listed for the method.
WORKLOAD_ORDER = ["tiny", "small_ties", "qwen_zipf", "gemma_softcap", "gemma_large"]


def _rng(seed: int, tag: int, block: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, block])))


def _to_bf16(x: np.ndarray) -> torch.Tensor:
    """Quantise float32 samples to bf16 (round to nearest even), giving a CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _bf16_normal(seed: int, tag: int, shape, std: float) -> torch.Tensor:
    x = _rng(seed, tag).standard_normal(size=shape, dtype=np.float32)
    x *= np.float32(std)
    return _to_bf16(x)


def tie_rows(w: Workload, seed: int) -> np.ndarray:
    """Flat row indices that receive planted ties: ceil(fraction * rows), at least one."""
    if w.tie_fraction <= 0:
        return np.zeros(0, dtype=np.int64)
    n = max(1, math.ceil(w.tie_fraction * w.rows))
    return np.sort(_rng(seed, _TAG_TIES).choice(w.rows, size=n, replace=False)).astype(np.int64)


def _plant_ties(row: np.ndarray, K: int, rng: np.random.Generator) -> None:
    """Plant exact ties so that the id tie-break decides both membership and order.

    Group A: floor(K/2) positions share the value top+2. All of them are selected, and
    their order among themselves comes from the ids alone.
    Group B: K+3 more positions share the value top+1. Exactly K - floor(K/2) of them
    are selected (the lowest ids), so the cut at K falls inside a tie.
    Here top is the row's largest value rounded up.
    """
    V = row.shape[0]
    na, nb = K // 2, K + 3
    pos = rng.choice(V, size=min(V, na + nb), replace=False)
    top = np.float32(math.ceil(float(np.max(row))))
    row[pos[:na]] = top + np.float32(2.0)
    row[pos[na:]] = top + np.float32(1.0)


def _logit_block(w: Workload, seed: int, block: int, out: np.ndarray) -> None:
    """Fill out[rows_in_block, V] with the logits of one block of rows."""
    nrows, V = out.shape
    rng = _rng(seed, _TAG_LOGITS, block)
    if w.logits in ("normal", "normal_ties", "normal_softcap"):
        rng.standard_normal(size=out.shape, dtype=np.float32, out=out)
        out *= np.float32(w.logit_std)
        if w.logits == "normal_softcap":
            # The softcap the logits processor applies, cap * tanh(x / cap), is part of the
            # input recipe here. The selector sees already-capped logits.
            np.divide(out, np.float32(w.softcap), out=out)
            np.tanh(out, out=out)
            out *= np.float32(w.softcap)
    elif w.logits == "zipf_gumbel":
        # logit[v] = -s * ln(1 + pi(v)) + Gumbel(0, 1), where pi is a per-row random
        # permutation of [0, V) that gives each token its popularity rank.
        ranks = np.arange(V, dtype=np.float64)
        profile = (-w.zipf_s * np.log1p(ranks)).astype(np.float32)
        prng = _rng(seed, _TAG_PERM, block)
        for i in range(nrows):
            perm = prng.permutation(V)
            u = rng.random(V)
            g = -np.log(-np.log(np.maximum(u, 1e-300)))
            out[i] = profile[perm] + g.astype(np.float32)
    else:
        raise ValueError(f"unknown logit recipe {w.logits!r}")


def make_logits(w: Workload, seed: int = 0, out: np.ndarray | None = None,
                threads: int | None = None) -> np.ndarray:
    """Logits [R, S, V] float32. Blocks of rows are filled in parallel threads.

    If `out` is given (for example the numpy view of a pinned host tensor), it is
    filled in place.
    """
    if out is None:
        out = np.empty((w.R, w.S, w.V), dtype=np.float32)
    assert out.shape == (w.R, w.S, w.V) and out.dtype == np.float32
    flat = out.reshape(w.rows, w.V)
    nblocks = (w.rows + _ROWS_PER_BLOCK - 1) // _ROWS_PER_BLOCK

    def fill(b: int) -> None:
        lo = b * _ROWS_PER_BLOCK
        hi = min(w.rows, lo + _ROWS_PER_BLOCK)
        _logit_block(w, seed, b, flat[lo:hi])

    threads = threads or min(32, os.cpu_count() or 1)
    if nblocks == 1 or threads == 1:
        for b in range(nblocks):
            fill(b)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(fill, range(nblocks)))
    if w.tie_fraction > 0:
        trng = _rng(seed, _TAG_TIES, 1)
        for r in tie_rows(w, seed):
            _plant_ties(flat[r], w.K, trng)
    return out


@dataclass
class Inputs:
    workload: Workload
    logits: np.ndarray        # float32 [R, S, V]
    hidden: torch.Tensor      # bf16 [R, S, H] (CPU)
    w_proj: torch.Tensor      # bf16 [rank, H]
    pred_cb: torch.Tensor     # bf16 [V, rank]
    succ_cb: torch.Tensor     # bf16 [V, rank]
    anchors: np.ndarray       # int32 [R]


def make_inputs(w: Workload | str, seed: int = 0, logits_out: np.ndarray | None = None,
                threads: int | None = None) -> Inputs:
    """All selector inputs of a workload, on the host."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    logits = make_logits(w, seed, out=logits_out, threads=threads)
    hidden = _bf16_normal(seed, _TAG_HIDDEN, (w.R, w.S, w.H), 1.0)
    w_proj = _bf16_normal(seed, _TAG_W, (w.rank, w.H), 1.0 / math.sqrt(w.H))
    pred_cb = _bf16_normal(seed, _TAG_PRED, (w.V, w.rank), 1.0 / math.sqrt(w.rank))
    succ_cb = _bf16_normal(seed, _TAG_SUCC, (w.V, w.rank), 1.0 / math.sqrt(w.rank))
    anchors = _rng(seed, _TAG_ANCHOR).integers(0, w.V, size=w.R, dtype=np.int64).astype(np.int32)
    return Inputs(w, logits, hidden, w_proj, pred_cb, succ_cb, anchors)


def custom_workload(R: int, S: int, K: int, V: int, H: int, rank: int, logits: str = "normal",
                    logit_std: float = 3.0, **kw) -> Workload:
    """A workload with arbitrary shapes, for edge-case tests (ragged sizes and the like)."""
    return Workload(f"custom_{R}_{S}_{K}_{V}_{H}_{rank}", R, S, K, V, H, rank, logits,
                    logit_std=logit_std, **kw)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw uint16 bit patterns of a bf16 CPU tensor, as a numpy array (no copy)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
