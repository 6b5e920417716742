"""GB300-native DFlash2 low-rank candidate selector.

This is the Python binding of libdflash_gb300.so, whose C ABI is in include/dflash.h.
The functions here marshal torch CUDA tensors into pointers and sizes and allocate any
outputs the caller did not pass. Every step of the method runs in the library's
sm_103a kernels, on the current CUDA stream of the tensors' device.

Method (page "vllm.models.beam.nvidia.dflash2"): for request r and step p,
  1. cand_ids, unary = top-K of logits[r, p]        (compute_candidates)
  2. h[r, p] = W_proj . hidden[r, p]                (DFlash2BeamCandidateSelector.hidden_projection)
  3. E[r,p,q,c] = unary[r,p,c]
                  + <pred_cb[cand[r,p-1,q]] * h[r,p], succ_cb[cand[r,p,c]]>
     with the anchor token as the predecessor at p = 0 (DFlash2BeamCandidateSelector)
"""

from __future__ import annotations

import ctypes

import torch

from . import _native
from ._native import DEVICE_BAD_ID, DEVICE_TIMEOUT, DflashError  # noqa: F401

__all__ = [
    "dflash_topk_candidates", "dflash_hidden_projection", "dflash_candidate_edges",
    "dflash_selector", "dflash_selector_forward", "dflash_lmhead_topk", "dflash_selector_lmhead",
    "dflash_best_path",
    "dflash_topk_workspace_bytes",
    "dflash_selector_workspace_bytes", "dflash_lmhead_topk_workspace_bytes",
    "dflash_selector_lmhead_workspace_bytes",
    "dflash_device_status", "dflash_trace_begin", "dflash_trace_end", "DflashError",
    "library_path", "CandidateSelector",
]


def library_path() -> str:
    _native.load()
    return _native._build.LIBRARY


def _stream(dev: torch.device, stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple | None = None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(None if t is None else t.data_ptr())


def dflash_topk_workspace_bytes(R: int, S: int, V: int, K: int) -> int:
    """Workspace bytes dflash_topk_candidates needs on the current device (0 = bad sizes)."""
    return int(_native.load().dflash_topk_workspace_bytes(R, S, V, K))


def dflash_selector_workspace_bytes(R: int, S: int, V: int, K: int) -> int:
    return int(_native.load().dflash_selector_workspace_bytes(R, S, V, K))


def dflash_lmhead_topk_workspace_bytes(R: int, S: int, V: int, K: int) -> int:
    return int(_native.load().dflash_lmhead_topk_workspace_bytes(R, S, V, K))


def dflash_selector_lmhead_workspace_bytes(R: int, S: int, V: int, K: int) -> int:
    return int(_native.load().dflash_selector_lmhead_workspace_bytes(R, S, V, K))


def _workspace(nbytes: int, dev: torch.device, workspace: torch.Tensor | None) -> torch.Tensor:
    if nbytes <= 0:
        _native.check(_native.DFLASH_INVALID_ARGUMENT)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    return workspace


def dflash_topk_candidates(logits: torch.Tensor, K: int, cand_ids: torch.Tensor | None = None,
                           unary: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None, stream=None,
                           softcap: float = 0.0, scale: float = 1.0):
    """Top-K candidate ids (int32) and their logits (fp32) of logits [R, S, V] fp32.

    softcap and scale are the logits processor's options: the reported values are
    scale * softcap * tanh(x / softcap) (no cap when softcap is 0).
    """
    lib = _native.load()
    if logits.dim() != 3:
        raise ValueError("logits must be [R, S, V]")
    _need(logits, "logits", torch.float32)
    R, S, V = logits.shape
    dev = logits.device
    with torch.cuda.device(dev):
        if cand_ids is None:
            cand_ids = torch.empty((R, S, K), dtype=torch.int32, device=dev)
        if unary is None:
            unary = torch.empty((R, S, K), dtype=torch.float32, device=dev)
        _need(cand_ids, "cand_ids", torch.int32, (R, S, K))
        _need(unary, "unary", torch.float32, (R, S, K))
        ws = _workspace(lib.dflash_topk_workspace_bytes(R, S, V, K), dev, workspace)
        _native.check(lib.dflash_topk_candidates(
            _ptr(logits), R, S, V, K, float(softcap), float(scale), _ptr(cand_ids), _ptr(unary),
            _ptr(ws), ws.numel(), _stream(dev, stream)))
    return cand_ids, unary


def dflash_lmhead_topk(hidden: torch.Tensor, lm_head: torch.Tensor, K: int,
                       cand_ids: torch.Tensor | None = None, unary: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, stream=None,
                       softcap: float = 0.0, scale: float = 1.0):
    """Top-K candidates of hidden [R, S, H] . lm_head [V, H]^T without materialised logits."""
    lib = _native.load()
    if hidden.dim() != 3 or lm_head.dim() != 2:
        raise ValueError("hidden must be [R, S, H] and lm_head [V, H]")
    R, S, H = hidden.shape
    V = lm_head.shape[0]
    _need(hidden, "hidden", torch.bfloat16)
    _need(lm_head, "lm_head", torch.bfloat16, (V, H))
    dev = hidden.device
    with torch.cuda.device(dev):
        if cand_ids is None:
            cand_ids = torch.empty((R, S, K), dtype=torch.int32, device=dev)
        if unary is None:
            unary = torch.empty((R, S, K), dtype=torch.float32, device=dev)
        _need(cand_ids, "cand_ids", torch.int32, (R, S, K))
        _need(unary, "unary", torch.float32, (R, S, K))
        ws = _workspace(lib.dflash_lmhead_topk_workspace_bytes(R, S, V, K), dev, workspace)
        _native.check(lib.dflash_lmhead_topk(
            _ptr(hidden), _ptr(lm_head), R, S, H, V, K, float(softcap), float(scale),
            _ptr(cand_ids), _ptr(unary), _ptr(ws), ws.numel(), _stream(dev, stream)))
    return cand_ids, unary


def dflash_hidden_projection(hidden: torch.Tensor, w_proj: torch.Tensor,
                             h_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """h [R, S, rank] bf16 = hidden [R, S, H] bf16 . w_proj [rank, H]^T (fp32 accumulate)."""
    lib = _native.load()
    if hidden.dim() != 3 or w_proj.dim() != 2:
        raise ValueError("hidden must be [R, S, H] and w_proj [rank, H]")
    R, S, H = hidden.shape
    rank = w_proj.shape[0]
    _need(hidden, "hidden", torch.bfloat16)
    _need(w_proj, "w_proj", torch.bfloat16, (rank, H))
    dev = hidden.device
    with torch.cuda.device(dev):
        if h_out is None:
            h_out = torch.empty((R, S, rank), dtype=torch.bfloat16, device=dev)
        _need(h_out, "h_out", torch.bfloat16, (R, S, rank))
        _native.check(lib.dflash_hidden_projection(
            _ptr(hidden), _ptr(w_proj), R, S, H, rank, _ptr(h_out), _stream(dev, stream)))
    return h_out


def dflash_candidate_edges(pred_cb: torch.Tensor, succ_cb: torch.Tensor,
                           cand_ids: torch.Tensor, unary: torch.Tensor, h: torch.Tensor,
                           anchors: torch.Tensor, edges: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """Edge scores E [R, S, K, K] fp32 (q = predecessor index, c = candidate index)."""
    lib = _native.load()
    if cand_ids.dim() != 3:
        raise ValueError("cand_ids must be [R, S, K]")
    R, S, K = cand_ids.shape
    V, rank = pred_cb.shape
    _need(pred_cb, "pred_cb", torch.bfloat16, (V, rank))
    _need(succ_cb, "succ_cb", torch.bfloat16, (V, rank))
    _need(cand_ids, "cand_ids", torch.int32)
    _need(unary, "unary", torch.float32, (R, S, K))
    _need(h, "h", torch.bfloat16, (R, S, rank))
    _need(anchors, "anchors", torch.int32, (R,))
    dev = cand_ids.device
    with torch.cuda.device(dev):
        if edges is None:
            edges = torch.empty((R, S, K, K), dtype=torch.float32, device=dev)
        _need(edges, "edges", torch.float32, (R, S, K, K))
        _native.check(lib.dflash_candidate_edges(
            _ptr(pred_cb), _ptr(succ_cb), _ptr(cand_ids), _ptr(unary), _ptr(h), _ptr(anchors),
            R, S, K, V, rank, _ptr(edges), _stream(dev, stream)))
    return edges


def dflash_selector(logits: torch.Tensor, hidden: torch.Tensor, w_proj: torch.Tensor,
                    pred_cb: torch.Tensor, succ_cb: torch.Tensor, anchors: torch.Tensor,
                    K: int, cand_ids: torch.Tensor | None = None,
                    unary: torch.Tensor | None = None, h_out: torch.Tensor | None = None,
                    edges: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                    stream=None, softcap: float = 0.0, scale: float = 1.0):
    """The whole selector in one library call: returns (cand_ids, unary, h, edges).

    softcap and scale are the logits processor's options (see dflash_topk_candidates).
    """
    lib = _native.load()
    if logits.dim() != 3 or hidden.dim() != 3:
        raise ValueError("logits must be [R, S, V] and hidden [R, S, H]")
    R, S, V = logits.shape
    H = hidden.shape[2]
    rank = w_proj.shape[0]
    _need(logits, "logits", torch.float32)
    _need(hidden, "hidden", torch.bfloat16, (R, S, H))
    _need(w_proj, "w_proj", torch.bfloat16, (rank, H))
    _need(pred_cb, "pred_cb", torch.bfloat16, (V, rank))
    _need(succ_cb, "succ_cb", torch.bfloat16, (V, rank))
    _need(anchors, "anchors", torch.int32, (R,))
    dev = logits.device
    with torch.cuda.device(dev):
        if cand_ids is None:
            cand_ids = torch.empty((R, S, K), dtype=torch.int32, device=dev)
        if unary is None:
            unary = torch.empty((R, S, K), dtype=torch.float32, device=dev)
        if h_out is None:
            h_out = torch.empty((R, S, rank), dtype=torch.bfloat16, device=dev)
        if edges is None:
            edges = torch.empty((R, S, K, K), dtype=torch.float32, device=dev)
        _need(cand_ids, "cand_ids", torch.int32, (R, S, K))
        _need(unary, "unary", torch.float32, (R, S, K))
        _need(h_out, "h_out", torch.bfloat16, (R, S, rank))
        _need(edges, "edges", torch.float32, (R, S, K, K))
        ws = _workspace(lib.dflash_selector_workspace_bytes(R, S, V, K), dev, workspace)
        _native.check(lib.dflash_selector(
            _ptr(logits), _ptr(hidden), _ptr(w_proj), _ptr(pred_cb), _ptr(succ_cb),
            _ptr(anchors), R, S, K, V, H, rank, float(softcap), float(scale), _ptr(cand_ids),
            _ptr(unary), _ptr(h_out), _ptr(edges), _ptr(ws), ws.numel(), _stream(dev, stream)))
    return cand_ids, unary, h_out, edges


def dflash_selector_forward(cand_ids: torch.Tensor, unary: torch.Tensor, hidden: torch.Tensor,
                            anchors: torch.Tensor, w_proj: torch.Tensor, pred_cb: torch.Tensor,
                            succ_cb: torch.Tensor, h_out: torch.Tensor | None = None,
                            edges: torch.Tensor | None = None, stream=None):
    """The selector's forward pass on given candidates: returns (h, edges).

    cand_ids int32 [R, S, K] and unary fp32 [R, S, K] are the candidates and their logits;
    h = hidden . w_proj^T is computed first, then the edge scores [R, S, K, K].
    """
    lib = _native.load()
    if cand_ids.dim() != 3 or hidden.dim() != 3:
        raise ValueError("cand_ids must be [R, S, K] and hidden [R, S, H]")
    R, S, K = cand_ids.shape
    H = hidden.shape[2]
    rank = w_proj.shape[0]
    V = pred_cb.shape[0]
    _need(cand_ids, "cand_ids", torch.int32)
    _need(unary, "unary", torch.float32, (R, S, K))
    _need(hidden, "hidden", torch.bfloat16, (R, S, H))
    _need(anchors, "anchors", torch.int32, (R,))
    _need(w_proj, "w_proj", torch.bfloat16, (rank, H))
    _need(pred_cb, "pred_cb", torch.bfloat16, (V, rank))
    _need(succ_cb, "succ_cb", torch.bfloat16, (V, rank))
    dev = hidden.device
    with torch.cuda.device(dev):
        if h_out is None:
            h_out = torch.empty((R, S, rank), dtype=torch.bfloat16, device=dev)
        if edges is None:
            edges = torch.empty((R, S, K, K), dtype=torch.float32, device=dev)
        _need(h_out, "h_out", torch.bfloat16, (R, S, rank))
        _need(edges, "edges", torch.float32, (R, S, K, K))
        _native.check(lib.dflash_selector_forward(
            _ptr(cand_ids), _ptr(unary), _ptr(hidden), _ptr(anchors), _ptr(w_proj), _ptr(pred_cb),
            _ptr(succ_cb), R, S, K, V, H, rank, _ptr(h_out), _ptr(edges), _stream(dev, stream)))
    return h_out, edges


def dflash_selector_lmhead(hidden: torch.Tensor, lm_head: torch.Tensor, w_proj: torch.Tensor,
                           pred_cb: torch.Tensor, succ_cb: torch.Tensor, anchors: torch.Tensor,
                           K: int, cand_ids: torch.Tensor | None = None,
                           unary: torch.Tensor | None = None, h_out: torch.Tensor | None = None,
                           edges: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None, stream=None,
                           softcap: float = 0.0, scale: float = 1.0):
    """The draft step from the LM head in one library call: returns (cand_ids, unary, h, edges).

    The candidates come straight from hidden [R, S, H] . lm_head [V, H]^T, as in
    dflash_lmhead_topk; no logits are written.
    """
    lib = _native.load()
    if hidden.dim() != 3 or lm_head.dim() != 2:
        raise ValueError("hidden must be [R, S, H] and lm_head [V, H]")
    R, S, H = hidden.shape
    V = lm_head.shape[0]
    rank = w_proj.shape[0]
    _need(hidden, "hidden", torch.bfloat16)
    _need(lm_head, "lm_head", torch.bfloat16, (V, H))
    _need(w_proj, "w_proj", torch.bfloat16, (rank, H))
    _need(pred_cb, "pred_cb", torch.bfloat16, (V, rank))
    _need(succ_cb, "succ_cb", torch.bfloat16, (V, rank))
    _need(anchors, "anchors", torch.int32, (R,))
    dev = hidden.device
    with torch.cuda.device(dev):
        if cand_ids is None:
            cand_ids = torch.empty((R, S, K), dtype=torch.int32, device=dev)
        if unary is None:
            unary = torch.empty((R, S, K), dtype=torch.float32, device=dev)
        if h_out is None:
            h_out = torch.empty((R, S, rank), dtype=torch.bfloat16, device=dev)
        if edges is None:
            edges = torch.empty((R, S, K, K), dtype=torch.float32, device=dev)
        _need(cand_ids, "cand_ids", torch.int32, (R, S, K))
        _need(unary, "unary", torch.float32, (R, S, K))
        _need(h_out, "h_out", torch.bfloat16, (R, S, rank))
        _need(edges, "edges", torch.float32, (R, S, K, K))
        ws = _workspace(lib.dflash_selector_lmhead_workspace_bytes(R, S, V, K), dev, workspace)
        _native.check(lib.dflash_selector_lmhead(
            _ptr(hidden), _ptr(lm_head), _ptr(w_proj), _ptr(pred_cb), _ptr(succ_cb),
            _ptr(anchors), R, S, K, V, H, rank, float(softcap), float(scale), _ptr(cand_ids),
            _ptr(unary), _ptr(h_out), _ptr(edges), _ptr(ws), ws.numel(), _stream(dev, stream)))
    return cand_ids, unary, h_out, edges


def dflash_best_path(edges: torch.Tensor, cand_ids: torch.Tensor, path: torch.Tensor | None = None,
                     tokens: torch.Tensor | None = None, score: torch.Tensor | None = None,
                     stream=None):
    """Max-sum path through edge scores [R, S, K, K]: returns (path int32 [R, S],
    tokens int32 [R, S], score fp32 [R])."""
    lib = _native.load()
    if edges.dim() != 4 or edges.shape[2] != edges.shape[3]:
        raise ValueError("edges must be [R, S, K, K]")
    R, S, K, _ = edges.shape
    _need(edges, "edges", torch.float32)
    _need(cand_ids, "cand_ids", torch.int32, (R, S, K))
    dev = edges.device
    with torch.cuda.device(dev):
        if path is None:
            path = torch.empty((R, S), dtype=torch.int32, device=dev)
        if tokens is None:
            tokens = torch.empty((R, S), dtype=torch.int32, device=dev)
        if score is None:
            score = torch.empty((R,), dtype=torch.float32, device=dev)
        _need(path, "path", torch.int32, (R, S))
        _need(tokens, "tokens", torch.int32, (R, S))
        _need(score, "score", torch.float32, (R,))
        _native.check(lib.dflash_best_path(_ptr(edges), _ptr(cand_ids), R, S, K, _ptr(path),
                                           _ptr(tokens), _ptr(score), _stream(dev, stream)))
    return path, tokens, score


def dflash_device_status(clear: bool = True) -> int:
    """DEVICE_* bits set by kernels on the current device since the last clear."""
    flags = ctypes.c_uint32(0)
    _native.check(_native.load().dflash_device_status(ctypes.byref(flags), int(clear)))
    return int(flags.value)


def dflash_trace_begin(n_calls: int) -> None:
    """Record stage timing events for the next n_calls dflash_selector(_lmhead) calls."""
    _native.check(_native.load().dflash_trace_begin(int(n_calls)))


def dflash_trace_end(max_calls: int) -> list[tuple[float, float, float]]:
    """Per traced call: (projection ms, top-k ms, edges ms). Ends the trace."""
    buf = (ctypes.c_float * (3 * max(1, max_calls)))()
    n = ctypes.c_int(0)
    _native.check(_native.load().dflash_trace_end(buf, int(max_calls), ctypes.byref(n)))
    return [(buf[3 * i], buf[3 * i + 1], buf[3 * i + 2]) for i in range(n.value)]


from .selector import CandidateSelector  # noqa: E402  (uses the functions above)
