"""The top-k entry point that allocates nothing, dflash_topk_candidates_noalloc.

Some callers may not allocate device memory. Examples are a plugin inside an inference
engine that has reserved all device memory for its own pool, and a code path where a
cudaMalloc would synchronise the device or is not allowed. This entry point serves them.
It uses a fixed scratch array that the library keeps in device memory, instead of a
workspace from the caller.

The test calls the entry point directly through the C ABI (ctypes). It runs two calls in
a row, on different logits, so the second call must reset the shared scratch the first
one left behind. Each result must match the workspace entry point: ids bit-exact, unary
logits within the suite's tolerance. The file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import parity as P
import draft_candidate_selector_gb300 as ds
from draft_candidate_selector_gb300 import _native

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _noalloc(lib, logits, K, cand, unary):
    R, S, V = logits.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream(logits.device).cuda_stream)
    return lib.dflash_topk_candidates_noalloc(
        ctypes.c_void_p(logits.data_ptr()), R, S, V, K, ctypes.c_void_p(cand.data_ptr()),
        ctypes.c_void_p(unary.data_ptr()), stream)


def test_noalloc_matches_workspace_entry_point_twice(dev):
    lib = _native.load()
    R, S, V, K = 6, 15, 50001, 32           # rows split across warps, V % 4 = 1
    rng = np.random.default_rng(21)
    for call in range(2):
        x = rng.standard_normal((R, S, V)).astype(np.float32)
        x[call, 3, ::97] = 9.0               # exact ties across the K-th place
        logits = torch.from_numpy(x).to(dev)
        cand = torch.empty((R, S, K), dtype=torch.int32, device=dev)
        unary = torch.empty((R, S, K), dtype=torch.float32, device=dev)
        st = _noalloc(lib, logits, K, cand, unary)
        assert st == _native.DFLASH_OK, lib.dflash_last_error().decode()
        ref_ids, ref_un = ds.dflash_topk_candidates(logits, K)
        torch.cuda.synchronize(dev)
        P.assert_ids_equal(cand.cpu().numpy(), ref_ids.cpu().numpy(), f"call {call} ids")
        P.assert_close(unary.cpu().numpy(), ref_un.cpu().numpy(), f"call {call} unary")


def test_noalloc_rejects_sizes_beyond_its_scratch(dev):
    lib = _native.load()
    A = ctypes.c_void_p(4096)   # aligned stand-in; the call returns before any launch
    rows = 2 ** 20              # 4 MiB of arrival counters alone: more than the scratch
    st = lib.dflash_topk_candidates_noalloc(A, rows, 1, 64, 8, A, A, None)
    assert st == _native.DFLASH_UNSUPPORTED
    assert b"scratch" in lib.dflash_last_error()
