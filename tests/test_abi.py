"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every function
include/dflash.h declares, and rejects bad arguments before any CUDA call."""

import ctypes
import os
import shutil
import subprocess

import pytest
import torch

from draft_candidate_selector_gb300 import _native

P = ctypes.c_void_p
A = P(4096)     # a non-null, 16-byte aligned stand-in pointer (never dereferenced)
MIS = P(4100)   # misaligned


@pytest.fixture(scope="module")
def lib():
    return _native.load()


def test_header_symbols_exported(lib):
    names = _native.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/dflash.h but not exported"
    assert set(names) == set(_native.SIGNATURES), "binding signatures out of sync with header"


def test_status_strings(lib):
    for code, name in [(0, "DFLASH_OK"), (1, "DFLASH_INVALID_ARGUMENT"),
                       (2, "DFLASH_UNSUPPORTED"), (3, "DFLASH_WORKSPACE_TOO_SMALL"),
                       (4, "DFLASH_CUDA_ERROR"), (5, "DFLASH_NO_DEVICE"),
                       (99, "DFLASH_UNKNOWN_STATUS")]:
        assert lib.dflash_status_string(code).decode() == name
    assert lib.dflash_version().decode().count(".") == 2


def _topk(lib, R=2, S=3, V=100, K=4, logits=A, ids=A, un=A, ws=A, wsb=1 << 20, cap=0.0,
          scale=1.0):
    return lib.dflash_topk_candidates(logits, R, S, V, K, cap, scale, ids, un, ws, wsb, None)


def test_topk_argument_checks(lib):
    assert _topk(lib, R=0) == _native.DFLASH_INVALID_ARGUMENT
    assert _topk(lib, V=0) == _native.DFLASH_INVALID_ARGUMENT
    assert _topk(lib, K=0) == _native.DFLASH_INVALID_ARGUMENT
    assert _topk(lib, K=101, V=100) == _native.DFLASH_INVALID_ARGUMENT
    assert _topk(lib, K=33) == _native.DFLASH_UNSUPPORTED
    assert _topk(lib, logits=P(None)) == _native.DFLASH_INVALID_ARGUMENT
    assert _topk(lib, ids=P(4098)) == _native.DFLASH_INVALID_ARGUMENT     # 2-byte offset
    assert _topk(lib, logits=P(4098)) == _native.DFLASH_INVALID_ARGUMENT   # 2-byte offset
    assert b"aligned" in lib.dflash_last_error()
    assert _topk(lib, ws=P(None)) == _native.DFLASH_INVALID_ARGUMENT
    assert _topk(lib, cap=-1.0) == _native.DFLASH_INVALID_ARGUMENT
    assert _topk(lib, cap=float("inf")) == _native.DFLASH_INVALID_ARGUMENT
    assert _topk(lib, scale=0.0) == _native.DFLASH_INVALID_ARGUMENT
    assert _topk(lib, scale=float("nan")) == _native.DFLASH_INVALID_ARGUMENT


def test_projection_argument_checks(lib):
    f = lib.dflash_hidden_projection
    assert f(A, A, 2, 3, 60, 16, A, None) == _native.DFLASH_UNSUPPORTED      # H % 8
    assert f(A, A, 2, 3, 64, 12, A, None) == _native.DFLASH_UNSUPPORTED      # rank % 8
    assert f(A, A, 2, 3, 64, 264, A, None) == _native.DFLASH_UNSUPPORTED     # rank > 256
    assert f(A, A, 0, 3, 64, 16, A, None) == _native.DFLASH_INVALID_ARGUMENT
    assert f(P(None), A, 2, 3, 64, 16, A, None) == _native.DFLASH_INVALID_ARGUMENT
    assert f(A, A, 2, 3, 64, 16, MIS, None) == _native.DFLASH_INVALID_ARGUMENT


def test_edges_argument_checks(lib):
    f = lib.dflash_candidate_edges
    args = [A] * 6
    assert f(*args, 2, 3, 0, 100, 16, A, None) == _native.DFLASH_INVALID_ARGUMENT
    assert f(*args, 2, 3, 40, 100, 16, A, None) == _native.DFLASH_UNSUPPORTED
    assert f(*args, 2, 3, 8, 4, 16, A, None) == _native.DFLASH_INVALID_ARGUMENT   # K > V
    assert f(*args, 2, 3, 8, 100, 20, A, None) == _native.DFLASH_UNSUPPORTED      # rank % 8
    assert f(A, A, A, A, A, P(None), 2, 3, 8, 100, 16, A, None) == _native.DFLASH_INVALID_ARGUMENT


def test_selector_argument_checks(lib):
    f = lib.dflash_selector
    good = dict(R=2, S=3, K=4, V=100, H=64, rank=16)

    def call(**kw):
        d = {**good, **kw}
        ptrs = kw.pop("ptrs", [A] * 6)
        return f(*ptrs, d["R"], d["S"], d["K"], d["V"], d["H"], d["rank"], d.get("cap", 0.0),
                 d.get("scale", 1.0), A, A, A, A, A, 1 << 20, None)

    assert call(K=33) == _native.DFLASH_UNSUPPORTED
    assert call(H=12) == _native.DFLASH_UNSUPPORTED
    assert call(V=2, K=4) == _native.DFLASH_INVALID_ARGUMENT
    assert call(ptrs=[A, A, A, A, MIS, A]) == _native.DFLASH_INVALID_ARGUMENT
    assert call(scale=-2.0) == _native.DFLASH_INVALID_ARGUMENT


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks behaviour without a GPU")
def test_no_device_is_reported(lib):
    assert _topk(lib) == _native.DFLASH_NO_DEVICE
    assert lib.dflash_topk_workspace_bytes(2, 3, 100, 4) == 0
    flags = ctypes.c_uint32(0)
    assert lib.dflash_device_status(ctypes.byref(flags), 0) == _native.DFLASH_NO_DEVICE
    assert lib.dflash_trace_begin(4) == _native.DFLASH_NO_DEVICE


def test_python_errors_map_to_exceptions(lib):
    with pytest.raises(ValueError):
        _native.check(_native.DFLASH_INVALID_ARGUMENT)
    with pytest.raises(NotImplementedError):
        _native.check(_native.DFLASH_UNSUPPORTED)
    with pytest.raises(_native.DflashError):
        _native.check(_native.DFLASH_CUDA_ERROR)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No fallback: without the compiled library the binding raises instead of computing."""
    monkeypatch.setattr(_native, "_lib", None)
    monkeypatch.setattr(_native._build, "LIBRARY", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _native.load(build_if_needed=False)


def test_trace_end_without_begin(lib):
    n = ctypes.c_int(7)
    assert lib.dflash_trace_end(None, 0, ctypes.byref(n)) == _native.DFLASH_INVALID_ARGUMENT
    assert lib.dflash_trace_begin(0) == _native.DFLASH_INVALID_ARGUMENT


def test_lmhead_argument_checks(lib):
    f = lib.dflash_lmhead_topk
    assert f(A, A, 2, 3, 60, 1000, 8, 0.0, 1.0, A, A, A, 1 << 20, None) == _native.DFLASH_UNSUPPORTED
    assert f(A, A, 2, 3, 64, 1000, 40, 0.0, 1.0, A, A, A, 1 << 20, None) == _native.DFLASH_UNSUPPORTED
    assert f(A, A, 2, 3, 64, 4, 8, 0.0, 1.0, A, A, A, 1 << 20, None) == _native.DFLASH_INVALID_ARGUMENT
    assert f(A, MIS, 2, 3, 64, 1000, 8, 0.0, 1.0, A, A, A, 1 << 20, None) == _native.DFLASH_INVALID_ARGUMENT
    assert f(A, A, 2, 3, 64, 1000, 8, 0.0, -1.0, A, A, A, 1 << 20, None) == _native.DFLASH_INVALID_ARGUMENT


def test_selector_lmhead_argument_checks(lib):
    f = lib.dflash_selector_lmhead

    def call(R=2, S=3, K=4, V=100, H=64, rank=16, cap=0.0, scale=1.0, ptrs=None, ws=1 << 20):
        ptrs = ptrs or [A] * 6
        return f(*ptrs, R, S, K, V, H, rank, cap, scale, A, A, A, A, A, ws, None)

    assert call(K=33) == _native.DFLASH_UNSUPPORTED
    assert call(H=12) == _native.DFLASH_UNSUPPORTED
    assert call(rank=20) == _native.DFLASH_UNSUPPORTED
    assert call(V=2, K=4) == _native.DFLASH_INVALID_ARGUMENT
    assert call(R=0) == _native.DFLASH_INVALID_ARGUMENT
    assert call(ptrs=[A, MIS, A, A, A, A]) == _native.DFLASH_INVALID_ARGUMENT
    assert call(ptrs=[A, A, A, A, A, P(None)]) == _native.DFLASH_INVALID_ARGUMENT
    assert call(scale=-2.0) == _native.DFLASH_INVALID_ARGUMENT
    assert call(cap=float("nan")) == _native.DFLASH_INVALID_ARGUMENT


def test_selector_forward_argument_checks(lib):
    f = lib.dflash_selector_forward

    def call(R=2, S=3, K=4, V=100, H=64, rank=16, ptrs=None):
        ptrs = ptrs or [A] * 7
        return f(*ptrs, R, S, K, V, H, rank, A, A, None)

    if not torch.cuda.is_available():
        assert call() == _native.DFLASH_NO_DEVICE    # valid arguments reach the device check
    assert call(K=33) == _native.DFLASH_UNSUPPORTED
    assert call(K=8, V=4) == _native.DFLASH_INVALID_ARGUMENT
    assert call(H=12) == _native.DFLASH_UNSUPPORTED
    assert call(rank=264) == _native.DFLASH_UNSUPPORTED
    assert call(S=0) == _native.DFLASH_INVALID_ARGUMENT
    assert call(ptrs=[A, A, MIS, A, A, A, A]) == _native.DFLASH_INVALID_ARGUMENT
    assert call(ptrs=[A, A, A, P(None), A, A, A]) == _native.DFLASH_INVALID_ARGUMENT


def test_best_path_argument_checks(lib):
    f = lib.dflash_best_path
    assert f(A, A, 0, 3, 4, A, A, A, None) == _native.DFLASH_INVALID_ARGUMENT
    assert f(A, A, 2, 3, 0, A, A, A, None) == _native.DFLASH_INVALID_ARGUMENT
    assert f(A, A, 2, 3, 33, A, A, A, None) == _native.DFLASH_UNSUPPORTED
    assert f(A, A, 2, 257, 4, A, A, A, None) == _native.DFLASH_UNSUPPORTED
    assert f(P(4098), A, 2, 3, 4, A, A, A, None) == _native.DFLASH_INVALID_ARGUMENT  # 2-byte
    assert f(A, A, 2, 3, 4, A, P(None), A, None) == _native.DFLASH_INVALID_ARGUMENT
    if not torch.cuda.is_available():
        assert f(A, A, 2, 3, 4, A, A, A, None) == _native.DFLASH_NO_DEVICE


def test_anchors_need_only_natural_alignment(lib):
    """anchors is read one id at a time: 4-byte alignment passes the checks, 2-byte does not."""
    f = lib.dflash_candidate_edges
    ok4, bad2 = P(4096 + 4), P(4096 + 2)
    expect_ok = _native.DFLASH_NO_DEVICE if not torch.cuda.is_available() else None
    st = f(A, A, A, A, A, ok4, 2, 3, 4, 100, 16, A, None)
    assert st != _native.DFLASH_INVALID_ARGUMENT or b"anchors" not in lib.dflash_last_error()
    if expect_ok is not None:
        assert st == expect_ok
    assert f(A, A, A, A, A, bad2, 2, 3, 4, 100, 16, A, None) == _native.DFLASH_INVALID_ARGUMENT
    assert b"anchors" in lib.dflash_last_error()


def test_candidate_selector_module_host_checks():
    """The module-style holder keeps the page's names and refuses non-bf16 weights."""
    import draft_candidate_selector_gb300 as ds
    sel = ds.CandidateSelector(64, 100, 16, 4, device="cpu")
    assert sel.predecessor_codebook.shape == (100, 16)
    assert sel.successor_codebook.shape == (100, 16)
    assert sel.hidden_projection_weight.shape == (16, 64)
    assert sel.predecessor_codebook.dtype == torch.bfloat16
    with pytest.raises(NotImplementedError):
        ds.CandidateSelector(64, 100, 16, 4, device="cpu", params_dtype=torch.float16)


_C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "dflash.h"

int main(void) {
    int32_t ids[4];
    float unary[4], logits[8] = {0};
    dflash_status s;
    if (strcmp(dflash_status_string(DFLASH_INVALID_ARGUMENT), "DFLASH_INVALID_ARGUMENT") != 0)
        return 2;
    if (dflash_version() == NULL) return 3;
    /* R = 0 is refused by the argument checks, before any CUDA call. */
    s = dflash_topk_candidates(logits, 0, 1, 8, 4, 0.0f, 1.0f, ids, unary, NULL, 0, NULL);
    if (s != DFLASH_INVALID_ARGUMENT) return 4;
    if (strlen(dflash_last_error()) == 0) return 5;
    printf("%s\n", dflash_version());
    return 0;
}
"""


def test_header_is_plain_c_and_links(lib, tmp_path):
    """include/dflash.h is a C99 header: a C program compiles against it with warnings as
    errors, links the library, and gets the documented answers (no GPU needed)."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "abi.c"
    src.write_text(_C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(_native._build.LIBRARY)
    include = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", include,
                    str(src), "-L", libdir, "-ldflash_gb300", f"-Wl,-rpath,{libdir}", "-o",
                    str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.strip() == lib.dflash_version().decode()
