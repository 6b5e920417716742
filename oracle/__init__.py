"""CPU oracle of the DFlash2 low-rank candidate selector.

TEST INFRASTRUCTURE. Only the tests, the smoke check in __graft_entry__ and the CPU
baseline leg of bench.py may import this package. The product library neither links it
nor calls it, and the two share no code: the arithmetic lives in dflash_oracle.c, plain
fp64 loops written from the page "vllm.models.beam.nvidia.dflash2"
(DFlash2BeamCandidateSelector and DFlash2BeamForCausalLM.compute_candidates).

Functions take and return numpy arrays. bf16 tensors travel as their uint16 bit patterns.

Every function here is pinned by tests/test_oracle_pins.py against brute force, closed
forms, invariants and library routines for special cases (none is "parity unpinned").
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle

class Oracle:
    """ctypes handle on one build of the oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_bf16_round.argtypes = [ctypes.c_double]
        lib.oracle_bf16_round.restype = ctypes.c_uint16
        lib.oracle_topk.argtypes = [p, i64, i64, i32, ctypes.c_double, ctypes.c_double, p, p, i32]
        lib.oracle_topk.restype = i32
        lib.oracle_projection.argtypes = [p, p, i64, i64, i64, p, p, i32]
        lib.oracle_projection.restype = i32
        lib.oracle_edges.argtypes = [p, p, i64, i64, p, p, p, p, i64, i64, i32, p, i32]
        lib.oracle_edges.restype = i32
        lib.oracle_selector.argtypes = [p, p, p, p, p, p, i64, i64, i32, i64, i64, i64,
                                        ctypes.c_double, ctypes.c_double, p, p, p, p, i32]
        lib.oracle_selector.restype = i32
        lib.oracle_lmhead_topk.argtypes = [p, p, i64, i64, i64, i32, ctypes.c_double,
                                           ctypes.c_double, p, p, p, i32]
        lib.oracle_lmhead_topk.restype = i32
        lib.oracle_best_path.argtypes = [p, p, i64, i64, i32, p, p, p, i32]
        lib.oracle_best_path.restype = i32
        self.lib = lib
        self.path = path

    def bf16_round(self, x: float) -> int:
        """Bit pattern of the bf16 nearest to x (ties to even), rounded in one step."""
        return int(self.lib.oracle_bf16_round(float(x)))

    def topk(self, logits: np.ndarray, K: int, threads: int | None = None,
             softcap: float = 0.0, scale: float = 1.0):
        """Top-K of each row of logits[..., V]: ids int32 [..., K], unary float32 [..., K].

        The order is logit descending, then token id ascending (-0 == +0). A NaN with the
        sign clear ranks above +inf, one with the sign set below -inf. unary is the
        processed logit scale * softcap * tanh(x / softcap) (no cap if softcap <= 0).
        """
        x = _c(logits, np.float32)
        V = x.shape[-1]
        lead = x.shape[:-1]
        rows = int(np.prod(lead)) if lead else 1
        ids = np.empty(lead + (K,), dtype=np.int32)
        unary = np.empty(lead + (K,), dtype=np.float32)
        rc = self.lib.oracle_topk(_ptr(x), rows, V, K, float(softcap), float(scale), _ptr(ids),
                                  _ptr(unary), threads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_topk failed (rc={rc}) for V={V}, K={K}")
        return ids, unary

    def lmhead_topk(self, hidden_bits: np.ndarray, lm_head_bits: np.ndarray, K: int,
                    threads: int | None = None, softcap: float = 0.0, scale: float = 1.0,
                    want_logits: bool = False):
        """Top-K of the exact logits hidden . lm_head^T (fp64): ids, processed unary values,
        and, with want_logits, the exact logits [..., V] (float64).

        hidden_bits uint16 [..., H]; lm_head_bits uint16 [V, H].
        """
        x = _c(hidden_bits, np.uint16)
        w = _c(lm_head_bits, np.uint16)
        H = x.shape[-1]
        V = w.shape[0]
        assert w.shape == (V, H)
        lead = x.shape[:-1]
        rows = int(np.prod(lead)) if lead else 1
        ids = np.empty(lead + (K,), dtype=np.int32)
        unary = np.empty(lead + (K,), dtype=np.float32)
        logits = np.empty(lead + (V,), dtype=np.float64) if want_logits else None
        rc = self.lib.oracle_lmhead_topk(_ptr(x), _ptr(w), rows, H, V, K, float(softcap),
                                         float(scale), _ptr(ids), _ptr(unary),
                                         _ptr(logits) if want_logits else None,
                                         threads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_lmhead_topk failed (rc={rc})")
        return (ids, unary, logits) if want_logits else (ids, unary)

    def projection(self, hidden_bits: np.ndarray, w_bits: np.ndarray,
                   threads: int | None = None, want_exact: bool = False):
        """h = bf16(W . hidden) per row: an exact sum, then one rounding.

        hidden_bits is uint16 [..., H] and w_bits uint16 [rank, H]. Returns uint16
        [..., rank], and also the fp64 sums when want_exact is set.
        """
        x = _c(hidden_bits, np.uint16)
        w = _c(w_bits, np.uint16)
        H = x.shape[-1]
        rank = w.shape[0]
        assert w.shape == (rank, H)
        lead = x.shape[:-1]
        rows = int(np.prod(lead)) if lead else 1
        h = np.empty(lead + (rank,), dtype=np.uint16)
        exact = np.empty(lead + (rank,), dtype=np.float64) if want_exact else None
        rc = self.lib.oracle_projection(_ptr(x), _ptr(w), rows, H, rank, _ptr(h),
                                        _ptr(exact) if want_exact else None,
                                        threads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_projection failed (rc={rc})")
        return (h, exact) if want_exact else h

    def edges(self, pred_bits: np.ndarray, succ_bits: np.ndarray, cand: np.ndarray,
              unary: np.ndarray, h_bits: np.ndarray, anchors: np.ndarray,
              threads: int | None = None, allow_bad_ids: bool = False) -> np.ndarray:
        """Edge scores E [R, S, K, K] float32 (q = predecessor index, c = candidate index).

        pred_bits, succ_bits: uint16 [V, rank]; cand int32 [R, S, K]; unary float32
        [R, S, K]; h_bits uint16 [R, S, rank]; anchors int32 [R].
        """
        a = _c(pred_bits, np.uint16)
        b = _c(succ_bits, np.uint16)
        cand = _c(cand, np.int32)
        un = _c(unary, np.float32)
        h = _c(h_bits, np.uint16)
        anc = _c(anchors, np.int32)
        V, rank = a.shape
        assert b.shape == (V, rank)
        R, S, K = cand.shape
        assert un.shape == (R, S, K) and h.shape == (R, S, rank) and anc.shape == (R,)
        out = np.empty((R, S, K, K), dtype=np.float32)
        rc = self.lib.oracle_edges(_ptr(a), _ptr(b), V, rank, _ptr(cand), _ptr(un), _ptr(h),
                                   _ptr(anc), R, S, K, _ptr(out), threads or default_threads())
        if rc < 0 or (rc == 1 and not allow_bad_ids):
            raise ValueError(f"oracle_edges failed (rc={rc})")
        return out

    def selector(self, logits: np.ndarray, hidden_bits: np.ndarray, w_bits: np.ndarray,
                 pred_bits: np.ndarray, succ_bits: np.ndarray, anchors: np.ndarray, K: int,
                 threads: int | None = None, softcap: float = 0.0, scale: float = 1.0):
        """All three steps for logits [R, S, V]: returns (ids, unary, h_bits, edges)."""
        x = _c(logits, np.float32)
        R, S, V = x.shape
        hid = _c(hidden_bits, np.uint16)
        H = hid.shape[-1]
        w = _c(w_bits, np.uint16)
        rank = w.shape[0]
        a = _c(pred_bits, np.uint16)
        b = _c(succ_bits, np.uint16)
        anc = _c(anchors, np.int32)
        ids = np.empty((R, S, K), dtype=np.int32)
        un = np.empty((R, S, K), dtype=np.float32)
        h = np.empty((R, S, rank), dtype=np.uint16)
        e = np.empty((R, S, K, K), dtype=np.float32)
        rc = self.lib.oracle_selector(_ptr(x), _ptr(hid), _ptr(w), _ptr(a), _ptr(b), _ptr(anc),
                                      R, S, K, V, H, rank, float(softcap), float(scale),
                                      _ptr(ids), _ptr(un), _ptr(h), _ptr(e),
                                      threads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_selector failed (rc={rc})")
        return ids, un, h, e


    def best_path(self, edges: np.ndarray, cand: np.ndarray, threads: int | None = None):
        """Max-sum path over edge scores [R, S, K, K] (fp32, the order of the C source):
        returns (path int32 [R, S], tokens int32 [R, S], score float32 [R])."""
        e = _c(edges, np.float32)
        cd = _c(cand, np.int32)
        R, S, K, K2 = e.shape
        assert K == K2 and cd.shape == (R, S, K)
        path = np.empty((R, S), dtype=np.int32)
        tokens = np.empty((R, S), dtype=np.int32)
        score = np.empty((R,), dtype=np.float32)
        rc = self.lib.oracle_best_path(_ptr(e), _ptr(cd), R, S, K, _ptr(path), _ptr(tokens),
                                       _ptr(score), threads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_best_path failed (rc={rc})")
        return path, tokens, score


_default: Oracle | None = None


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def get() -> Oracle:
    """The oracle built from oracle/dflash_oracle.c (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build_oracle())
    return _default


def bf16_round(x: float) -> int:
    return get().bf16_round(x)


def topk(logits, K, threads=None, softcap=0.0, scale=1.0):
    return get().topk(logits, K, threads, softcap, scale)


def projection(hidden_bits, w_bits, threads=None, want_exact=False):
    return get().projection(hidden_bits, w_bits, threads, want_exact)


def edges(pred_bits, succ_bits, cand, unary, h_bits, anchors, threads=None,
          allow_bad_ids=False):
    return get().edges(pred_bits, succ_bits, cand, unary, h_bits, anchors, threads,
                       allow_bad_ids)


def lmhead_topk(hidden_bits, lm_head_bits, K, threads=None, softcap=0.0, scale=1.0,
                want_logits=False):
    return get().lmhead_topk(hidden_bits, lm_head_bits, K, threads, softcap, scale, want_logits)


def selector(logits, hidden_bits, w_bits, pred_bits, succ_bits, anchors, K, threads=None,
             softcap=0.0, scale=1.0):
    return get().selector(logits, hidden_bits, w_bits, pred_bits, succ_bits, anchors, K,
                          threads, softcap, scale)


def best_path(edges, cand, threads=None):
    return get().best_path(edges, cand, threads)


def bits_to_float(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
