"""GPU parity: the sm_103a kernels, called through the C ABI, against the CPU oracle on
the same seeded inputs.

Every workload is compared in full, the large ones (qwen_zipf, gemma_softcap, gemma_large)
included: they run at full size, in the launch configuration the benchmark times, and every
row, request and edge score is compared with the oracle's. The oracle's top-k and
projection of a workload are computed once and reused by the tests that need them. Besides,
a check that needs no oracle runs on the device over every row of the large workloads:
exactly K - 1 logits beat the K-th candidate in the candidate order. Edge cases cover ragged
sizes (V, H and rank not multiples of the tile sizes), exact ties, signed zeros, infinities,
NaNs, sorted rows, K = 1, K = V, K = 32, step 0 only, and bad ids.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import parity as P
import draft_candidate_selector_gb300 as ds
from draft_candidate_selector_gb300 import _native
from draft_candidate_selector_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SMALL = ["tiny", "small_ties"]
LARGE = ["qwen_zipf", "gemma_softcap", "gemma_large"]
# Several tiles and warps, with every size ragged: V % 4 = 1, H % 64 = 8, rank % 16 = 8.
RAGGED = wl.custom_workload(3, 7, 16, 50001, 328, 40)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    ds.dflash_device_status(clear=True)
    return d


_CACHE: dict = {}


def host_inputs(name):
    """Seeded inputs, keeping one large workload in memory at a time."""
    key = name if isinstance(name, str) else name.name
    if key not in _CACHE:
        if key in LARGE:
            for k in [k for k in _CACHE if k in LARGE]:
                del _CACHE[k]
        _CACHE[key] = wl.make_inputs(name, seed=0)
    return _CACHE[key]


def _status_clean():
    assert ds.dflash_device_status(clear=True) == 0


_ORACLE: dict = {}


def oracle_topk_of(name):
    """The oracle's top-k of a workload's logits (every row), computed once."""
    inp = host_inputs(name)
    key = ("topk", inp.workload.name)
    if key not in _ORACLE:
        _ORACLE[key] = oracle.topk(inp.logits, inp.workload.K)
    return _ORACLE[key]


def oracle_h_of(name):
    """The oracle's projection of a workload's hidden states (every row), computed once."""
    inp = host_inputs(name)
    key = ("h", inp.workload.name)
    if key not in _ORACLE:
        _ORACLE[key] = oracle.projection(P.bits(inp.hidden), P.bits(inp.w_proj))
    return _ORACLE[key]


def assert_rank_of_kth(x: torch.Tensor, ids: torch.Tensor, K: int, what: str) -> None:
    """On the device, for every row: exactly K - 1 logits come before the K-th candidate in
    the candidate order (logit descending, then id ascending; -0 == +0). With distinct ids
    in descending order this says the candidates are the row's top K, ties included. It
    needs no oracle. Rows go in chunks so the temporaries stay near 1 GB."""
    V = x.shape[-1]
    x2, i2 = x.reshape(-1, V), ids.reshape(-1, K)
    col = torch.arange(V, device=x.device, dtype=torch.int64)[None, :]
    step = max(1, (1 << 28) // V)
    for r0 in range(0, x2.shape[0], step):
        xs = x2[r0:r0 + step]
        kid = i2[r0:r0 + step, K - 1].long()[:, None]
        kv = torch.gather(xs, 1, kid)
        before = ((xs > kv) | ((xs == kv) & (col < kid))).sum(dim=1)
        bad = torch.nonzero(before != K - 1)
        if bad.numel():
            r = int(bad[0, 0]) + r0
            raise AssertionError(f"{what}: row {r} has {int(before[r - r0])} logits before its "
                                 f"K-th candidate, not {K - 1}")


# ----------------------------------------------------------------------------- top-k

@pytest.mark.parametrize("name", SMALL + ["ragged"])
def test_topk_small_full(dev, name):
    inp = host_inputs(RAGGED if name == "ragged" else name)
    w = inp.workload
    x = torch.from_numpy(inp.logits).to(dev)
    ids, un = ds.dflash_topk_candidates(x, w.K)
    ref_ids, ref_un = oracle.topk(inp.logits, w.K)
    P.assert_ids_equal(ids.cpu().numpy(), ref_ids, f"{name} ids")
    P.assert_close(un.cpu().numpy(), ref_un, f"{name} unary")
    _status_clean()


@pytest.mark.parametrize("name", LARGE)
def test_topk_large_full(dev, name):
    """Every row of the large workloads against the oracle: ids bit-exact, unary within
    tolerance. Then, on the device, properties that need no oracle: distinct ids in range,
    unary equal to the logit at the id, non-increasing unary, and the rank of the K-th
    candidate."""
    inp = host_inputs(name)
    w = inp.workload
    x = torch.from_numpy(inp.logits).to(dev)
    ids, un = ds.dflash_topk_candidates(x, w.K)
    ref_ids, ref_un = oracle_topk_of(name)
    P.assert_ids_equal(ids.cpu().numpy(), ref_ids, f"{name} ids")
    P.assert_close(un.cpu().numpy(), ref_un, f"{name} unary")
    ids_all = ids.reshape(w.rows, w.K)
    assert int(ids_all.min()) >= 0 and int(ids_all.max()) < w.V
    srt = torch.sort(ids_all, dim=1).values
    assert bool((srt[:, 1:] != srt[:, :-1]).all())
    gathered = torch.gather(x.reshape(w.rows, w.V), 1, ids_all.long())
    assert torch.equal(gathered, un.reshape(w.rows, w.K))
    assert bool((un[..., 1:] <= un[..., :-1]).all())
    assert_rank_of_kth(x, ids, w.K, f"{name} rank of the K-th candidate")
    del x
    _status_clean()


@pytest.mark.parametrize("R,S,V,K", [
    (3000, 1, 25003, 32),     # many rows per warp span; spans end mid-row at odd places
    (4, 1, 20000003, 8),      # each row spread over hundreds of warps
])
def test_topk_large_odd_shapes(dev, R, S, V, K):
    """Problems above 256 MB with odd shapes: thousands of short rows (V = 25003, many rows per
    warp and spans ending mid-row at odd places), and a few rows of 20 million logits, each
    spread over hundreds of warps whose partial lists the last to finish merges. Every row
    against the oracle, plus the rank check on the device."""
    rng = np.random.default_rng(R + V)
    x = (rng.standard_normal((R, S, V), dtype=np.float32) * 5).astype(np.float32)
    x.reshape(-1)[rng.choice(x.size, 1000, replace=False)] = 12.0     # ties near the top
    assert x.nbytes >= 256 << 20
    xt = torch.from_numpy(x).to(dev)
    ids, un = ds.dflash_topk_candidates(xt, K)
    ref_ids, ref_un = oracle.topk(x, K)
    P.assert_ids_equal(ids.cpu().numpy(), ref_ids, f"R={R} V={V} ids")
    P.assert_close(un.cpu().numpy(), ref_un, f"R={R} V={V} unary")
    assert_rank_of_kth(xt, ids, K, f"R={R} V={V} rank of the K-th candidate")
    _status_clean()


def _topk_case(dev, x: np.ndarray, K: int, what: str):
    xt = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev)
    ids, un = ds.dflash_topk_candidates(xt, K)
    ref_ids, ref_un = oracle.topk(x, K)
    P.assert_ids_equal(ids.cpu().numpy(), ref_ids, what)
    P.assert_close(un.cpu().numpy(), ref_un, what)


@pytest.mark.parametrize("V", [1, 2, 3, 4, 5, 31, 32, 33, 127, 129, 4095, 4097, 65537])
def test_topk_ragged_vocab(dev, V):
    rng = np.random.default_rng(V)
    x = rng.integers(-3, 4, size=(2, 3, V)).astype(np.float32)      # heavy ties
    x[x == 0] = np.where(rng.random(int((x == 0).sum())) < 0.5, -0.0, 0.0)
    for K in sorted({1, min(V, 7), min(V, 32)}):
        _topk_case(dev, x, K, f"V={V} K={K}")


def test_topk_special_values(dev):
    V = 9000
    rng = np.random.default_rng(7)
    x = rng.standard_normal((4, 5, V)).astype(np.float32)
    x[0, 0, ::7] = np.inf
    x[0, 1, ::5] = -np.inf
    x[0, 1, 1::5] = np.nan
    x[0, 2, 3::11] = np.copysign(np.float32(np.nan), np.float32(-1))
    x[0, 3, :] = -np.inf                       # the whole row at -inf: ties on ids
    x[0, 4, :] = np.copysign(np.float32(np.nan), np.float32(-1))
    x[1, 0, :] = 0.0
    x[1, 0, ::2] = -0.0                        # signed zeros only
    x[1, 1, :] = np.arange(V, dtype=np.float32)          # ascending: every element enters
    x[1, 2, :] = -np.arange(V, dtype=np.float32)         # descending
    x[1, 3, :] = 1e-45                         # subnormals
    x[2] = np.float32(1.5)                     # all equal
    for K in (1, 8, 32):
        _topk_case(dev, x, K, f"special K={K}")


def test_topk_many_small_rows(dev):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((50, 40, 33)).astype(np.float32)   # 2000 rows, V % 4 = 1
    _topk_case(dev, x, 32, "V=33 K=32")
    y = rng.standard_normal((7, 13, 4099)).astype(np.float32)
    _topk_case(dev, y, 17, "V=4099 K=17")


def test_topk_k_equals_v(dev):
    rng = np.random.default_rng(4)
    x = rng.integers(-2, 3, size=(3, 4, 32)).astype(np.float32)
    _topk_case(dev, x, 32, "K = V = 32")


def test_topk_reuses_workspace(dev):
    """Two calls in a row with one workspace: the arrival counters start from zero again."""
    inp = host_inputs(RAGGED)
    w = inp.workload
    x = torch.from_numpy(inp.logits).to(dev)
    nb = ds.dflash_topk_workspace_bytes(w.R, w.S, w.V, w.K)
    ws = torch.full((nb,), 0xAB, dtype=torch.uint8, device=dev)   # garbage on entry
    ref_ids, _ = oracle.topk(inp.logits, w.K)
    for _ in range(3):
        ids, _ = ds.dflash_topk_candidates(x, w.K, workspace=ws)
        P.assert_ids_equal(ids.cpu().numpy(), ref_ids, "reused workspace")


# ----------------------------------------------------------------------------- projection

def _projection_case(dev, rows, H, rank, seed, what):
    g = torch.Generator().manual_seed(seed)
    hid = torch.randn(1, rows, H, generator=g).to(torch.bfloat16)
    w = (torch.randn(rank, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    h = ds.dflash_hidden_projection(hid.to(dev), w.to(dev))
    P.assert_projection(P.bits(h), P.bits(hid), P.bits(w), what)


@pytest.mark.parametrize("rows,H,rank", [
    (1, 8, 8), (129, 72, 24), (300, 1000, 256), (256, 64, 128), (17, 4096, 40),
    (1000, 5376, 256), (385, 3840, 128), (64, 2048, 136), (130, 520, 248),
    # 256-wide N tiles run on CTA pairs (256-row tiles over two CTAs): a single row (the odd
    # CTA's rows all out of range), a tail tile of one row, one K block, a K split.
    (1, 64, 256), (257, 520, 256), (7680, 64, 256), (640, 2048, 256),
])
def test_projection_shapes(dev, rows, H, rank):
    _projection_case(dev, rows, H, rank, rows + H + rank, f"rows={rows} H={H} rank={rank}")
    _status_clean()


@pytest.mark.parametrize("name", SMALL + ["ragged"] + LARGE)
def test_projection_workloads(dev, name):
    inp = host_inputs(RAGGED if name == "ragged" else name)
    w = inp.workload
    h = ds.dflash_hidden_projection(inp.hidden.to(dev), inp.w_proj.to(dev))
    P.assert_projection(P.bits(h), P.bits(inp.hidden), P.bits(inp.w_proj), f"{name} h")
    _status_clean()


def test_projection_closed_forms(dev):
    rows, H = 200, 256
    g = torch.Generator().manual_seed(5)
    hid = torch.randn(2, rows // 2, H, generator=g).to(torch.bfloat16).to(dev)
    zero = torch.zeros(64, H, dtype=torch.bfloat16, device=dev)
    assert torch.equal(ds.dflash_hidden_projection(hid, zero),
                       torch.zeros(2, rows // 2, 64, dtype=torch.bfloat16, device=dev))
    eye = torch.eye(H, dtype=torch.bfloat16, device=dev)       # rank = H = 256
    assert torch.equal(ds.dflash_hidden_projection(hid, eye), hid)


# ----------------------------------------------------------------------------- edges

def _edge_inputs_from_oracle(name):
    """Candidates, unary and h from the ORACLE, so the edge kernel is tested alone."""
    ids, un = oracle_topk_of(name)
    return ids, un, oracle_h_of(name), host_inputs(name).anchors


def _run_edges(dev, inp, ids, un, h, anchors):
    h_t = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev)
    return ds.dflash_candidate_edges(
        inp.pred_cb.to(dev), inp.succ_cb.to(dev), torch.from_numpy(ids).to(dev),
        torch.from_numpy(un).to(dev), h_t, torch.from_numpy(anchors).to(dev))


@pytest.mark.parametrize("name", SMALL + ["ragged"] + LARGE)
def test_edges_workloads(dev, name):
    key = RAGGED if name == "ragged" else name
    inp = host_inputs(key)
    ids, un, h, anchors = _edge_inputs_from_oracle(key)
    e = _run_edges(dev, inp, ids, un, h, anchors)
    ref = oracle.edges(P.bits(inp.pred_cb), P.bits(inp.succ_cb), ids, un, h, anchors)
    P.assert_close(e.cpu().numpy(), ref, f"{name} edges")
    _status_clean()


@pytest.mark.parametrize("R,S,K,V,rank", [
    (2, 1, 4, 100, 16),      # step 0 only: every row from the anchor
    (3, 5, 1, 50, 8),        # K = 1
    (2, 4, 32, 64, 8),       # K = 32 with the smallest rank
    (1, 3, 32, 40000, 256),  # K = 32, largest rank
    (4, 6, 5, 77, 24),       # K not a power of two
])
def test_edges_shapes(dev, R, S, K, V, rank):
    rng = np.random.default_rng(R * 1000 + K)
    g = torch.Generator().manual_seed(K + rank)
    pred = (torch.randn(V, rank, generator=g) / rank ** 0.5).to(torch.bfloat16)
    succ = (torch.randn(V, rank, generator=g) / rank ** 0.5).to(torch.bfloat16)
    ids = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(S)])
                    for _ in range(R)]).astype(np.int32)
    un = rng.standard_normal((R, S, K)).astype(np.float32)
    h = P.bits(torch.randn(R, S, rank, generator=g).to(torch.bfloat16))
    anchors = rng.integers(0, V, R).astype(np.int32)
    e = ds.dflash_candidate_edges(
        pred.to(dev), succ.to(dev), torch.from_numpy(ids).to(dev), torch.from_numpy(un).to(dev),
        torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev),
        torch.from_numpy(anchors).to(dev))
    ref = oracle.edges(P.bits(pred), P.bits(succ), ids, un, h, anchors)
    P.assert_close(e.cpu().numpy(), ref, f"edges R={R} S={S} K={K} V={V} rank={rank}")
    # Structure that holds at any size: every predecessor row at step 0 is identical.
    e0 = e[:, 0]
    assert torch.equal(e0, e0[:, :1, :].expand_as(e0))
    # The output only needs 4-byte alignment: written at an address that is not 8-byte
    # aligned (one value at a time rather than in pairs), the scores are the same bits.
    buf = torch.full((R * S * K * K + 1,), float("nan"), dtype=torch.float32, device=dev)
    e_odd = buf[1:].view(R, S, K, K)
    ds.dflash_candidate_edges(
        pred.to(dev), succ.to(dev), torch.from_numpy(ids).to(dev), torch.from_numpy(un).to(dev),
        torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev),
        torch.from_numpy(anchors).to(dev), edges=e_odd)
    assert torch.equal(e_odd.view(torch.int32), e.view(torch.int32))
    _status_clean()


def test_edges_subnormal_codebook_entries(dev):
    """Products are taken as in fp32, subnormal bf16 inputs included: pred entries of 2^-130
    (subnormal), h = 2^100 and succ = 2^20 give 2^-10 per term and exactly 16 * 2^-10 = 2^-6
    per score over rank 16. Flushing the subnormal inputs would give 0."""
    R, S, K, V, rank = 1, 2, 2, 4, 16
    sub, big_h, big_s = np.uint16(0x0008), np.uint16(0x7180), np.uint16(0x4980)
    assert float(oracle.bits_to_float(np.array([sub]))[0]) == 2.0 ** -130
    assert float(oracle.bits_to_float(np.array([big_h]))[0]) == 2.0 ** 100
    assert float(oracle.bits_to_float(np.array([big_s]))[0]) == 2.0 ** 20
    pred = np.full((V, rank), sub, dtype=np.uint16)
    succ = np.full((V, rank), big_s, dtype=np.uint16)
    ids = np.array([[[0, 1], [2, 3]]], dtype=np.int32)
    un = np.zeros((R, S, K), dtype=np.float32)
    h = np.full((R, S, rank), big_h, dtype=np.uint16)
    anchors = np.array([3], dtype=np.int32)
    as_bf16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    e = ds.dflash_candidate_edges(as_bf16(pred), as_bf16(succ), torch.from_numpy(ids).to(dev),
                                  torch.from_numpy(un).to(dev), as_bf16(h),
                                  torch.from_numpy(anchors).to(dev))
    ref = oracle.edges(pred, succ, ids, un, h, anchors)
    assert np.all(ref == 2.0 ** -6)
    assert np.array_equal(e.cpu().numpy(), ref.astype(np.float32))
    _status_clean()


def test_edges_bad_ids_are_reported_not_followed(dev):
    """An anchor or candidate id outside [0, V) gives NaN scores and sets the status bit."""
    R, S, K, V, rank = 2, 3, 4, 50, 16
    rng = np.random.default_rng(9)
    g = torch.Generator().manual_seed(9)
    pred = torch.randn(V, rank, generator=g).to(torch.bfloat16)
    succ = torch.randn(V, rank, generator=g).to(torch.bfloat16)
    ids = rng.integers(0, V, (R, S, K)).astype(np.int32)
    ids[1, 2, 3] = V + 5          # bad candidate: column 3 of request 1, step 2
    un = rng.standard_normal((R, S, K)).astype(np.float32)
    h = P.bits(torch.randn(R, S, rank, generator=g).to(torch.bfloat16))
    anchors = np.array([-1, 7], dtype=np.int32)   # bad anchor for request 0
    e = ds.dflash_candidate_edges(
        pred.to(dev), succ.to(dev), torch.from_numpy(ids).to(dev), torch.from_numpy(un).to(dev),
        torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev),
        torch.from_numpy(anchors).to(dev))
    status = ds.dflash_device_status(clear=True)
    assert status & ds.DEVICE_BAD_ID
    ref = oracle.edges(P.bits(pred), P.bits(succ), ids, un, h, anchors, allow_bad_ids=True)
    P.assert_close(e.cpu().numpy(), ref, "edges with bad ids")


@pytest.mark.parametrize("R,S,K,V,rank", [
    (400, 15, 23, 5000, 40),      # padded contraction (40 -> 48), ragged K
    (160, 15, 32, 262144, 256),   # the largest layout
])
def test_edges_many_waves_with_bad_ids(dev, R, S, K, V, rank):
    """Thousands of (r, p) tiles, several waves of CTAs per SM, with bad ids sprinkled in:
    every score equals the oracle's, bad rows and columns are NaN, and the status bit is
    set."""
    rng = np.random.default_rng(R + K + rank)
    g = torch.Generator().manual_seed(R + rank)
    pred = (torch.randn(V, rank, generator=g) / rank ** 0.5).to(torch.bfloat16)
    succ = (torch.randn(V, rank, generator=g) / rank ** 0.5).to(torch.bfloat16)
    ids = rng.integers(0, V, (R, S, K)).astype(np.int32)
    bad = rng.choice(R * S * K, 7, replace=False)
    ids.reshape(-1)[bad[:4]] = V + rng.integers(0, 100, 4)
    ids.reshape(-1)[bad[4:]] = -1 - rng.integers(0, 100, 3)
    un = rng.standard_normal((R, S, K)).astype(np.float32)
    h = P.bits(torch.randn(R, S, rank, generator=g).to(torch.bfloat16))
    anchors = rng.integers(0, V, R).astype(np.int32)
    anchors[R // 2] = V                            # one bad anchor
    ds.dflash_device_status(clear=True)
    e = ds.dflash_candidate_edges(
        pred.to(dev), succ.to(dev), torch.from_numpy(ids).to(dev), torch.from_numpy(un).to(dev),
        torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev),
        torch.from_numpy(anchors).to(dev))
    assert ds.dflash_device_status(clear=True) & ds.DEVICE_BAD_ID
    ref = oracle.edges(P.bits(pred), P.bits(succ), ids, un, h, anchors, allow_bad_ids=True)
    P.assert_close(e.cpu().numpy(), ref, f"edges, many waves, K={K} rank={rank}")


# ----------------------------------------------------------------------------- fused selector

def _selector_check(dev, inp: wl.Inputs, what: str):
    """The fused call on a whole workload against the oracle's own fused selector (every
    request, row and edge score)."""
    w = inp.workload
    d = P.to_device(inp, dev)
    ids, un, h, e = ds.dflash_selector(d["logits"], d["hidden"], d["w_proj"], d["pred_cb"],
                                       d["succ_cb"], d["anchors"], w.K)
    r_ids, r_un, r_h, r_e = oracle.selector(inp.logits, P.bits(inp.hidden), P.bits(inp.w_proj),
                                            P.bits(inp.pred_cb), P.bits(inp.succ_cb),
                                            inp.anchors, w.K)
    P.assert_ids_equal(ids.cpu().numpy(), r_ids, f"{what} ids")
    P.assert_close(un.cpu().numpy(), r_un, f"{what} unary")
    P.assert_projection(P.bits(h), P.bits(inp.hidden), P.bits(inp.w_proj), f"{what} h")
    P.assert_close(e.cpu().numpy(), r_e, f"{what} edges")
    del d
    _status_clean()


@pytest.mark.parametrize("name", SMALL + ["ragged"])
def test_selector_small_full(dev, name):
    _selector_check(dev, host_inputs(RAGGED if name == "ragged" else name), name)


@pytest.mark.parametrize("name", LARGE)
def test_selector_large_full(dev, name):
    _selector_check(dev, host_inputs(name), name)


def test_selector_trace(dev):
    """Traced calls time each stage, and give the same bits as untraced ones: a traced call
    runs the projection first and the kernels one after another, while an untraced call at
    this size launches the projection after the top-k."""
    inp = host_inputs("small_ties")
    w = inp.workload
    d = P.to_device(inp, dev)
    args = (d["logits"], d["hidden"], d["w_proj"], d["pred_cb"], d["succ_cb"], d["anchors"], w.K)
    untraced = [x.clone() for x in ds.dflash_selector(*args)]
    ds.dflash_trace_begin(3)
    outs = []
    for _ in range(4):   # the fourth call is beyond the trace capacity and not traced
        outs.append([x.clone() for x in ds.dflash_selector(*args)])
    stages = ds.dflash_trace_end(8)
    assert len(stages) == 3
    assert all(t >= 0 for row in stages for t in row) and all(row[1] > 0 for row in stages)
    bits = {torch.bfloat16: torch.int16, torch.float32: torch.int32, torch.int32: torch.int32}
    for o in outs:
        for a, b in zip(o, untraced):
            assert torch.equal(a.view(bits[a.dtype]), b.view(bits[b.dtype]))
    _status_clean()


def test_selector_cuda_graph_replay(dev):
    """The fused call captured once in a CUDA graph (a memset node and three kernels), then
    replayed on fresh inputs copied into the same buffers, matches the oracle each time."""
    w = wl.WORKLOADS["small_ties"]
    first = wl.make_inputs(w, seed=0)
    d = P.to_device(first, dev)
    cand = torch.empty((w.R, w.S, w.K), dtype=torch.int32, device=dev)
    unary = torch.empty((w.R, w.S, w.K), dtype=torch.float32, device=dev)
    h = torch.empty((w.R, w.S, w.rank), dtype=torch.bfloat16, device=dev)
    edges = torch.empty((w.R, w.S, w.K, w.K), dtype=torch.float32, device=dev)
    ws = torch.empty(ds.dflash_selector_workspace_bytes(w.R, w.S, w.V, w.K), dtype=torch.uint8,
                     device=dev)

    def call():
        ds.dflash_selector(d["logits"], d["hidden"], d["w_proj"], d["pred_cb"], d["succ_cb"],
                           d["anchors"], w.K, cand, unary, h, edges, ws)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        call()                       # eager warm-up on a side stream, as torch advises
    torch.cuda.current_stream(dev).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for seed in (1, 2):
        inp = wl.make_inputs(w, seed=seed)
        d["logits"].copy_(torch.from_numpy(inp.logits))
        d["hidden"].copy_(inp.hidden)
        d["anchors"].copy_(torch.from_numpy(inp.anchors))
        graph.replay()
        torch.cuda.synchronize(dev)
        r_ids, r_un, r_h, r_e = oracle.selector(
            inp.logits, P.bits(inp.hidden), P.bits(first.w_proj), P.bits(first.pred_cb),
            P.bits(first.succ_cb), inp.anchors, w.K)
        P.assert_ids_equal(cand.cpu().numpy(), r_ids, f"graph replay {seed} ids")
        P.assert_projection(P.bits(h), P.bits(inp.hidden), P.bits(first.w_proj),
                            f"graph replay {seed} h")
        P.assert_close(edges.cpu().numpy(), r_e, f"graph replay {seed} edges")
    _status_clean()


# ----------------------------------------------------------------------------- logits processor

@pytest.mark.parametrize("cap,scale", [(30.0, 1.0), (10.0, 0.5), (0.0, 2.0), (1.0, 1.0)])
def test_topk_logits_processor(dev, cap, scale):
    """Soft cap and output multiplier on the reported unary values; ids from raw logits."""
    inp = host_inputs("small_ties")
    w = inp.workload
    x = inp.logits * np.float32(8.0)      # large logits, so tanh saturates in places
    ids, un = ds.dflash_topk_candidates(torch.from_numpy(x).to(dev), w.K, softcap=cap,
                                        scale=scale)
    ref_ids, ref_un = oracle.topk(x, w.K, softcap=cap, scale=scale)
    P.assert_ids_equal(ids.cpu().numpy(), ref_ids, f"cap={cap} scale={scale} ids")
    P.assert_close(un.cpu().numpy(), ref_un, f"cap={cap} scale={scale} unary")


def test_topk_logits_processor_saturation_keeps_raw_order(dev):
    x = np.array([[[20.0, 30.0, -5.0, 25.0]]], dtype=np.float32)
    ids, un = ds.dflash_topk_candidates(torch.from_numpy(x).to(dev), 3, softcap=1.0, scale=1.0)
    assert ids.cpu().numpy().tolist() == [[[1, 3, 0]]]
    assert un.cpu().numpy().tolist() == [[[1.0, 1.0, 1.0]]]


@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_selector_logits_processor(dev, name):
    inp = host_inputs(RAGGED if name == "ragged" else name)
    w = inp.workload
    d = P.to_device(inp, dev)
    ids, un, h, e = ds.dflash_selector(d["logits"], d["hidden"], d["w_proj"], d["pred_cb"],
                                       d["succ_cb"], d["anchors"], w.K, softcap=30.0, scale=1.5)
    r_ids, r_un, r_h, r_e = oracle.selector(inp.logits, P.bits(inp.hidden), P.bits(inp.w_proj),
                                            P.bits(inp.pred_cb), P.bits(inp.succ_cb),
                                            inp.anchors, w.K, softcap=30.0, scale=1.5)
    P.assert_ids_equal(ids.cpu().numpy(), r_ids, f"{name} ids")
    P.assert_close(un.cpu().numpy(), r_un, f"{name} processed unary")
    P.assert_projection(P.bits(h), P.bits(inp.hidden), P.bits(inp.w_proj), f"{name} h")
    P.assert_close(e.cpu().numpy(), r_e, f"{name} edges")
    _status_clean()


@pytest.mark.parametrize("name", SMALL + ["ragged"])
def test_selector_forward(dev, name):
    """The selector's forward pass on given candidates. Fed the fused selector's candidates it
    reproduces its h and edges bit for bit; fed arbitrary candidates (repeats included) its
    h and edges match the oracle."""
    inp = host_inputs(RAGGED if name == "ragged" else name)
    w = inp.workload
    d = P.to_device(inp, dev)
    ids, un, h, e = ds.dflash_selector(d["logits"], d["hidden"], d["w_proj"], d["pred_cb"],
                                       d["succ_cb"], d["anchors"], w.K)
    h2, e2 = ds.dflash_selector_forward(ids, un, d["hidden"], d["anchors"], d["w_proj"],
                                        d["pred_cb"], d["succ_cb"])
    torch.cuda.synchronize(dev)
    assert np.array_equal(P.bits(h2), P.bits(h))
    assert np.array_equal(e2.cpu().numpy().view(np.uint32), e.cpu().numpy().view(np.uint32))

    rng = np.random.default_rng(17)
    cand = rng.integers(0, w.V, size=(w.R, w.S, w.K)).astype(np.int32)
    cand[:, :, -1] = cand[:, :, 0]                    # a repeated candidate in every row
    unary = rng.standard_normal((w.R, w.S, w.K)).astype(np.float32)
    h3, e3 = ds.dflash_selector_forward(torch.from_numpy(cand).to(dev),
                                        torch.from_numpy(unary).to(dev), d["hidden"],
                                        d["anchors"], d["w_proj"], d["pred_cb"], d["succ_cb"])
    P.assert_projection(P.bits(h3), P.bits(inp.hidden), P.bits(inp.w_proj), f"{name} forward h")
    ref = oracle.edges(P.bits(inp.pred_cb), P.bits(inp.succ_cb), cand, unary, P.bits(h3),
                       inp.anchors)
    P.assert_close(e3.cpu().numpy(), ref, f"{name} forward edges")
    _status_clean()


@pytest.mark.parametrize("name", LARGE)
def test_selector_forward_full_size(dev, name):
    """The forward pass at full size in the launch configuration `bench.py --forward` times
    (gemma_large: the projection on 30 CTA pairs split over K in two, the edges launched as its
    programmatic dependent), on the workload's inputs and seeded candidates with a repeat in
    every row: every entry of h and every edge score against the oracle."""
    inp = host_inputs(name)
    w = inp.workload
    d = P.to_device(inp, dev)
    rng = np.random.default_rng(23)
    cand = rng.integers(0, w.V, size=(w.R, w.S, w.K)).astype(np.int32)
    cand[:, :, -1] = cand[:, :, 0]
    unary = rng.standard_normal((w.R, w.S, w.K)).astype(np.float32)
    h, e = ds.dflash_selector_forward(torch.from_numpy(cand).to(dev),
                                      torch.from_numpy(unary).to(dev), d["hidden"],
                                      d["anchors"], d["w_proj"], d["pred_cb"], d["succ_cb"])
    torch.cuda.synchronize(dev)
    P.assert_projection(P.bits(h), P.bits(inp.hidden), P.bits(inp.w_proj), f"{name} forward h")
    ref = oracle.edges(P.bits(inp.pred_cb), P.bits(inp.succ_cb), cand, unary, P.bits(h),
                       inp.anchors)
    P.assert_close(e.cpu().numpy(), ref, f"{name} forward edges")
    del d
    _status_clean()


@pytest.mark.parametrize("R,S,K,V,H,rank", [(4, 15, 32, 50000, 5376, 256), (3, 7, 13, 40000, 520, 256)])
def test_selector_forward_rank_256(dev, R, S, K, V, H, rank):
    """The forward pass at a rank of 256, where the projection runs on CTA pairs with a K
    split (the fused selector's build takes another plan there): h and the edge scores
    against the oracle, with repeated candidates and an odd K."""
    g = torch.Generator().manual_seed(R * 1000 + K)
    hidden = torch.randn(R, S, H, generator=g).to(torch.bfloat16)
    w_proj = (torch.randn(rank, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    pred_cb = (torch.randn(V, rank, generator=g) / rank ** 0.5).to(torch.bfloat16)
    succ_cb = (torch.randn(V, rank, generator=g) / rank ** 0.5).to(torch.bfloat16)
    rng = np.random.default_rng(R + K)
    cand = rng.integers(0, V, size=(R, S, K)).astype(np.int32)
    cand[:, :, -1] = cand[:, :, 0]
    unary = rng.standard_normal((R, S, K)).astype(np.float32)
    anchors = rng.integers(0, V, size=(R,)).astype(np.int32)
    h, e = ds.dflash_selector_forward(torch.from_numpy(cand).to(dev), torch.from_numpy(unary).to(dev),
                                      hidden.to(dev), torch.from_numpy(anchors).to(dev),
                                      w_proj.to(dev), pred_cb.to(dev), succ_cb.to(dev))
    torch.cuda.synchronize(dev)
    P.assert_projection(P.bits(h), P.bits(hidden), P.bits(w_proj), f"rank 256 forward h R={R} K={K}")
    ref = oracle.edges(P.bits(pred_cb), P.bits(succ_cb), cand, unary, P.bits(h), anchors)
    P.assert_close(e.cpu().numpy(), ref, f"rank 256 forward edges R={R} K={K}")
    _status_clean()


@pytest.mark.parametrize("name", SMALL + ["ragged"] + LARGE)
def test_best_path(dev, name):
    """The best path through the fused selector's edge scores equals the oracle's (same fp32
    decisions in the same order): path, tokens and score bit for bit, every request."""
    w = wl.WORKLOADS[name] if name != "ragged" else RAGGED
    if name in LARGE:
        # Edge scores shaped like the workload's, without the (large) logits: the path only
        # reads E and the candidates.
        rng = np.random.default_rng(31)
        e = rng.standard_normal((w.R, w.S, w.K, w.K)).astype(np.float32)
        cand = rng.integers(0, w.V, size=(w.R, w.S, w.K)).astype(np.int32)
        E = torch.from_numpy(e).to(dev)
        ids = torch.from_numpy(cand).to(dev)
    else:
        inp = host_inputs(RAGGED if name == "ragged" else name)
        d = P.to_device(inp, dev)
        ids, _, _, E = ds.dflash_selector(d["logits"], d["hidden"], d["w_proj"], d["pred_cb"],
                                          d["succ_cb"], d["anchors"], w.K)
    path, tokens, score = ds.dflash_best_path(E, ids)
    ref_path, ref_tokens, ref_score = oracle.best_path(E.cpu().numpy(), ids.cpu().numpy())
    P.assert_ids_equal(path.cpu().numpy(), ref_path, f"{name} path")
    P.assert_ids_equal(tokens.cpu().numpy(), ref_tokens, f"{name} tokens")
    assert np.array_equal(score.cpu().numpy().view(np.uint32), ref_score.view(np.uint32))
    _status_clean()


def test_best_path_ties_and_edge_shapes(dev):
    """Exact ties everywhere (integer scores), K = 1, odd K and K = 32, S = 1 and the maximum
    S, and NaNs and infinities: every choice must match the oracle's scan exactly."""
    rng = np.random.default_rng(32)
    for (R, S, K) in [(5, 7, 4), (3, 1, 8), (4, 9, 1), (2, 256, 32), (9, 15, 32), (6, 11, 7),
                      (8, 15, 32)]:
        e = rng.integers(-2, 3, size=(R, S, K, K)).astype(np.float32)      # many ties
        if K == 32 and S == 15 and R == 8:
            # NaNs (as bad candidate ids give) and infinities, at predecessor 0 and elsewhere
            e[rng.random(e.shape) < 0.05] = np.nan
            e[rng.random(e.shape) < 0.02] = np.inf
            e[rng.random(e.shape) < 0.02] = -np.inf
            e[0, 3, 0, :] = np.nan
        cand = rng.integers(0, 1 << 20, size=(R, S, K)).astype(np.int32)
        path, tokens, score = ds.dflash_best_path(torch.from_numpy(e).to(dev),
                                                  torch.from_numpy(cand).to(dev))
        rp, rt, rs = oracle.best_path(e, cand)
        P.assert_ids_equal(path.cpu().numpy(), rp, f"path R={R} S={S} K={K}")
        P.assert_ids_equal(tokens.cpu().numpy(), rt, f"tokens R={R} S={S} K={K}")
        # Equal values; a NaN score matches a NaN (its payload is the adder's, not the data's)
        assert np.array_equal(score.cpu().numpy(), rs, equal_nan=True)
    _status_clean()


def test_odd_k_request_slices(dev):
    """With K odd, request slices of the candidate ids, unary values, edge scores and the
    best path's outputs start off 16-byte boundaries. Those arrays need only 4-byte alignment:
    the fused selector writing into slices, the forward pass reading them and the best path
    staging them equal calls on whole, aligned arrays."""
    w = wl.custom_workload(5, 3, 7, 3001, 64, 16)
    d = P.to_device(wl.make_inputs(w, seed=0), dev)
    ids, un, h, e = ds.dflash_selector(d["logits"], d["hidden"], d["w_proj"], d["pred_cb"],
                                       d["succ_cb"], d["anchors"], w.K)
    a, b = 1, 4                                   # requests 1..3
    s_ids, s_un, s_h, s_e = (torch.empty_like(x) for x in (ids, un, h, e))
    ds.dflash_selector(d["logits"][a:b], d["hidden"][a:b], d["w_proj"], d["pred_cb"],
                       d["succ_cb"], d["anchors"][a:b], w.K, s_ids[a:b], s_un[a:b], s_h[a:b],
                       s_e[a:b])
    assert s_ids[a:b].data_ptr() % 16 != 0 and s_e[a:b].data_ptr() % 16 != 0
    assert d["logits"][a:b].data_ptr() % 16 != 0
    assert torch.equal(s_ids[a:b], ids[a:b])
    assert torch.equal(s_un[a:b].view(torch.int32), un[a:b].view(torch.int32))
    assert torch.equal(s_e[a:b].view(torch.int32), e[a:b].view(torch.int32))
    _, f_e = ds.dflash_selector_forward(ids[a:b], un[a:b], d["hidden"][a:b], d["anchors"][a:b],
                                        d["w_proj"], d["pred_cb"], d["succ_cb"])
    assert torch.equal(f_e.view(torch.int32), e[a:b].view(torch.int32))
    path = torch.zeros((w.R, w.S), dtype=torch.int32, device=dev)
    tokens = torch.zeros_like(path)
    score = torch.zeros((w.R,), dtype=torch.float32, device=dev)
    ds.dflash_best_path(e[a:b], ids[a:b], path[a:b], tokens[a:b], score[a:b])
    rp, rt, rs = oracle.best_path(e[a:b].cpu().numpy(), ids[a:b].cpu().numpy())
    P.assert_ids_equal(path[a:b].cpu().numpy(), rp, "best path on a slice")
    P.assert_ids_equal(tokens[a:b].cpu().numpy(), rt, "best path tokens on a slice")
    assert np.array_equal(score[a:b].cpu().numpy().view(np.uint32), rs.view(np.uint32))
    # K even with the edge scores off a 16-byte boundary: the path stages with 4-byte copies
    rng = np.random.default_rng(9)
    flat = rng.standard_normal(4 * 5 * 8 * 8 + 2).astype(np.float32)
    big = torch.from_numpy(flat).to(dev)
    e8 = big[2:].view(4, 5, 8, 8)
    c8 = torch.from_numpy(rng.integers(0, 100, (4, 5, 8)).astype(np.int32)).to(dev)
    assert e8.data_ptr() % 16 == 8
    p8, t8, s8 = ds.dflash_best_path(e8, c8)
    rp8, rt8, rs8 = oracle.best_path(e8.cpu().numpy(), c8.cpu().numpy())
    P.assert_ids_equal(p8.cpu().numpy(), rp8, "best path, offset base")
    P.assert_ids_equal(t8.cpu().numpy(), rt8, "best path tokens, offset base")
    assert np.array_equal(s8.cpu().numpy().view(np.uint32), rs8.view(np.uint32))
    _status_clean()


# ----------------------------------------------------------------------------- candidate head from the LM head

def _bf16(t):
    return t.to(torch.bfloat16)


@pytest.mark.parametrize("rows,H,V,K", [
    (7, 64, 300, 4),          # one row tile, two vocabulary tiles
    (130, 520, 8000, 8),      # ragged rows, K and V; 32 vocabulary splits of one tile each
    (300, 256, 3000, 32),     # K = 32
    (2560, 64, 20000, 16),    # on 152 SMs: CTA pairs, 10 units of 256 rows x 7 splits
    (50, 64, 200, 20),        # one vocabulary tile: no split, no merge; K between list sizes
    (40, 128, 1500, 12),      # K between list sizes, ragged last chunk of 32 columns
    # On 152 SMs: 40 row tiles x 3 splits plus 30 helper CTAs (4 row tiles' tails each)
    (5000, 64, 6000, 8),
    # On 152 SMs: 100 row tiles x 1 split plus 50 helpers (2 tails each): two lists per row
    (12700, 64, 2100, 32),
    # Single CTAs, 9 row tiles x 16 splits (pairs would pad the rows by a sixth)
    (1100, 64, 20000, 16),
    # CTA pairs, 5 row units x 15 splits; the odd CTA of the last pair holds padding only
    (1152, 96, 9000, 32),
    # CTA pairs, 4 row units x 19 splits, the last unit a quarter padding; K = 8
    (960, 128, 11000, 8),
])
def test_lmhead_topk_valid(dev, rows, H, V, K):
    g = torch.Generator().manual_seed(rows + V)
    hid = _bf16(torch.randn(1, rows, H, generator=g))
    w = _bf16(torch.randn(V, H, generator=g) / H ** 0.5)
    ids, un = ds.dflash_lmhead_topk(hid.to(dev), w.to(dev), K)
    same = P.assert_lmhead_valid(ids.cpu().numpy(), un.cpu().numpy(), P.bits(hid), P.bits(w), K,
                                 f"rows={rows} H={H} V={V} K={K}")
    assert same > 0.9, f"only {same:.2f} of rows match the exact order"
    _status_clean()


def _lmhead_full_size(dev, name):
    w = wl.WORKLOADS[name]
    hid = wl._bf16_normal(0, wl._TAG_HIDDEN, (w.R, w.S, w.H), 1.0)
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    lm = (torch.randn((w.V, w.H), generator=g, device=dev) / w.H ** 0.5).to(torch.bfloat16)
    ids, un = ds.dflash_lmhead_topk(hid.to(dev), lm, w.K, softcap=w.softcap)
    return w, hid, lm, ids, un


@pytest.mark.parametrize("name", ["qwen_zipf", "gemma_softcap", "gemma_large"])
def test_lmhead_topk_full_size_sampled(dev, name):
    """At the full sizes the benchmark times, in the launch configuration it times (on 152 SMs:
    qwen_zipf 4 CTA pairs of 256 rows x 19 splits, the last unit a quarter padding;
    gemma_softcap 15 pairs x 5 splits, with the soft cap; gemma_large 60 single CTAs x 2
    splits plus 30 helper CTAs), sampled rows against the exact logits of the oracle."""
    w, hid, lm, ids, un = _lmhead_full_size(dev, name)
    last = w.rows - 1
    rows = P.sample_rows(w.rows, 4, seed=11, extra=[127, 128, 255, 256, last - 128, last - 1])
    ids = ids.cpu().numpy().reshape(-1, w.K)[rows]
    un = un.cpu().numpy().reshape(-1, w.K)[rows]
    hb = P.bits(hid).reshape(-1, w.H)[rows]
    same = P.assert_lmhead_valid(ids, un, hb, P.bits(lm), w.K, f"{name} sampled rows",
                                 softcap=w.softcap)
    assert same >= 0.5, f"only {same:.2f} of the sampled rows match the exact order"
    _status_clean()


@pytest.mark.parametrize("name", ["qwen_zipf", "gemma_softcap", "gemma_large"])
def test_lmhead_topk_full_size_every_row(dev, name):
    """Every row at full size, against plain fp32 logits on the device (torch's GEMM of the
    same bf16 inputs): ids valid and distinct, no clear winner left out, values ordered and
    within the fp32 summation bound of the reference."""
    w, hid, lm, ids, un = _lmhead_full_size(dev, name)
    P.assert_lmhead_valid_every_row(ids, un, hid.to(dev), lm, w.K, f"{name} every row",
                                    softcap=w.softcap)
    _status_clean()


@pytest.mark.parametrize("rows", [200, 1024])
def test_lmhead_topk_one_hot_exact(dev, rows):
    """One-hot hidden states make every logit an exact LM-head entry: no rounding at all, so
    the ids must equal the oracle's, ties (planted in the LM head) included. 1024 rows run on
    CTA pairs (4 row units of 256 x 19 vocabulary splits on 152 SMs)."""
    H, V, K = 128, 5000, 16
    rng = np.random.default_rng(5)
    hot = rng.integers(0, H, rows)
    x = np.zeros((1, rows, H), dtype=np.float32)
    x[0, np.arange(rows), hot] = rng.choice([1.0, -1.0, 0.5, 2.0], rows)
    w = rng.integers(-6, 7, size=(V, H)).astype(np.float32) / 4   # many exact ties
    xb, wb = P.float_bits(x), P.float_bits(w)
    ids, un = ds.dflash_lmhead_topk(torch.from_numpy(x).to(torch.bfloat16).to(dev),
                                    torch.from_numpy(w).to(torch.bfloat16).to(dev), K)
    ref_ids, ref_un = oracle.lmhead_topk(xb.reshape(rows, H), wb, K)
    P.assert_ids_equal(ids.cpu().numpy().reshape(rows, K), ref_ids, "one-hot ids")
    P.assert_close(un.cpu().numpy().reshape(rows, K), ref_un, "one-hot unary")
    _status_clean()


def test_lmhead_topk_fuzz_shapes(dev):
    """Seeded random shapes, most of them in the CTA-pair regime on 152 SMs (rows a multiple
    of 256 or close below one, no helper CTAs): ragged vocabularies (the odd CTA's half of the
    last vocabulary tile out of range), hidden sizes that are not a multiple of the 64-wide K
    block, K from 1 to 32, with and without the logits processor. Every row is checked
    against plain fp32 logits on the device."""
    rng = np.random.default_rng(2024)
    for case in range(8):
        rows = int(rng.choice([512, 1000, 1024, 1536, 1800, 2048, 700, 256]))
        V = int(rng.integers(300, 12000))
        H = int(rng.integers(1, 80)) * 8
        K = int(rng.integers(1, 33))
        cap, scale = [(0.0, 1.0), (20.0, 0.75)][case % 2]
        g = torch.Generator().manual_seed(case)
        hid = _bf16(torch.randn(1, rows, H, generator=g)).to(dev)
        w = _bf16(torch.randn(V, H, generator=g) / H ** 0.5).to(dev)
        ids, un = ds.dflash_lmhead_topk(hid, w, K, softcap=cap, scale=scale)
        P.assert_lmhead_valid_every_row(ids, un, hid, w, K,
                                        f"rows={rows} H={H} V={V} K={K} cap={cap}",
                                        softcap=cap, scale=scale)
    _status_clean()


def test_lmhead_topk_logits_processor(dev):
    g = torch.Generator().manual_seed(3)
    rows, H, V, K = 64, 96, 2000, 8
    hid = _bf16(torch.randn(1, rows, H, generator=g) * 4)
    w = _bf16(torch.randn(V, H, generator=g))
    ids, un = ds.dflash_lmhead_topk(hid.to(dev), w.to(dev), K, softcap=5.0, scale=0.5)
    P.assert_lmhead_valid(ids.cpu().numpy(), un.cpu().numpy(), P.bits(hid), P.bits(w), K,
                          "lm head with soft cap", softcap=5.0, scale=0.5)


def test_lmhead_odd_k_request_slices(dev):
    """With K odd, request slices of the candidate ids, unary values and edge scores start off
    16-byte boundaries (4-byte alignment is all they need). The LM-head top-k and the draft
    step from the LM head, writing into such slices, equal the calls on whole arrays bit for
    bit: each output's arithmetic does not depend on where its row sits in a tile."""
    R, S, K, V, H, rank = 5, 3, 7, 3001, 128, 16
    g = torch.Generator().manual_seed(77)
    hid = _bf16(torch.randn(R, S, H, generator=g)).to(dev)
    lm = _bf16(torch.randn(V, H, generator=g) / H ** 0.5).to(dev)
    wp = _bf16(torch.randn(rank, H, generator=g) / H ** 0.5).to(dev)
    pc = _bf16(torch.randn(V, rank, generator=g) / rank ** 0.5).to(dev)
    sc = _bf16(torch.randn(V, rank, generator=g) / rank ** 0.5).to(dev)
    anchors = torch.randint(0, V, (R,), generator=g, dtype=torch.int32).to(dev)
    a, b = 1, 4
    ids, un = ds.dflash_lmhead_topk(hid, lm, K)
    s_ids, s_un = torch.zeros_like(ids), torch.zeros_like(un)
    ds.dflash_lmhead_topk(hid[a:b], lm, K, s_ids[a:b], s_un[a:b])
    torch.cuda.synchronize(dev)
    assert s_ids[a:b].data_ptr() % 16 != 0
    assert torch.equal(s_ids[a:b], ids[a:b])
    assert torch.equal(s_un[a:b].view(torch.int32), un[a:b].view(torch.int32))
    f_ids, f_un, f_h, f_e = ds.dflash_selector_lmhead(hid, lm, wp, pc, sc, anchors, K)
    o_ids, o_un = torch.zeros_like(f_ids), torch.zeros_like(f_un)
    o_h, o_e = torch.zeros_like(f_h), torch.zeros_like(f_e)
    ds.dflash_selector_lmhead(hid[a:b], lm, wp, pc, sc, anchors[a:b], K, o_ids[a:b], o_un[a:b],
                              o_h[a:b], o_e[a:b])
    torch.cuda.synchronize(dev)
    assert o_e[a:b].data_ptr() % 16 != 0
    assert torch.equal(o_ids[a:b], f_ids[a:b])
    assert torch.equal(o_un[a:b].view(torch.int32), f_un[a:b].view(torch.int32))
    assert torch.equal(o_h[a:b].view(torch.int16), f_h[a:b].view(torch.int16))
    assert torch.equal(o_e[a:b].view(torch.int32), f_e[a:b].view(torch.int32))
    _status_clean()


@pytest.mark.parametrize("R,S,K,V,H,rank,cap,scale", [
    (3, 7, 8, 5000, 256, 64, 0.0, 1.0),        # 21 rows, 20 vocabulary splits
    (40, 15, 32, 6000, 128, 128, 30.0, 1.5),   # 600 rows in 5 row tiles, K = 32, processed
    (64, 16, 16, 7000, 192, 64, 30.0, 1.0),    # 1024 rows on CTA pairs (152 SMs), soft cap
])
def test_selector_lmhead(dev, R, S, K, V, H, rank, cap, scale):
    """The draft step from the LM head: its candidates are those of dflash_lmhead_topk (same
    kernel, bit for bit) and valid against the exact logits; h and the edge scores of the
    returned candidates match the oracle."""
    g = torch.Generator().manual_seed(R * V + K)
    hid = _bf16(torch.randn(R, S, H, generator=g))
    lm = _bf16(torch.randn(V, H, generator=g) / H ** 0.5)
    wp = _bf16(torch.randn(rank, H, generator=g) / H ** 0.5)
    pc = _bf16(torch.randn(V, rank, generator=g) / rank ** 0.5)
    sc = _bf16(torch.randn(V, rank, generator=g) / rank ** 0.5)
    anchors = torch.randint(0, V, (R,), generator=g, dtype=torch.int32)
    d = [x.to(dev) for x in (hid, lm, wp, pc, sc, anchors)]
    ids, un, h, e = ds.dflash_selector_lmhead(*d, K, softcap=cap, scale=scale)
    ids2, un2 = ds.dflash_lmhead_topk(d[0], d[1], K, softcap=cap, scale=scale)
    torch.cuda.synchronize(dev)
    ids_np, un_np = ids.cpu().numpy(), un.cpu().numpy()
    P.assert_ids_equal(ids_np, ids2.cpu().numpy(), "ids against dflash_lmhead_topk")
    assert np.array_equal(un_np.view(np.uint32), un2.cpu().numpy().view(np.uint32))
    P.assert_lmhead_valid(ids_np, un_np, P.bits(hid), P.bits(lm), K, "selector from the LM head",
                          softcap=cap, scale=scale)
    P.assert_projection(P.bits(h), P.bits(hid), P.bits(wp), "selector from the LM head: h")
    ref_e = oracle.edges(P.bits(pc), P.bits(sc), ids_np, un_np, P.bits(h), anchors.numpy())
    P.assert_close(e.cpu().numpy(), ref_e, "selector from the LM head: edges")
    _status_clean()


@pytest.mark.parametrize("name", ["qwen_zipf", "gemma_softcap"])
def test_selector_lmhead_full_size(dev, name):
    """The draft step from the LM head at full size (on 152 SMs its LM-head top-k runs on CTA
    pairs at both shapes), with the workload's hidden states, projection and codebooks and a
    seeded synthetic LM head: its candidates are those of dflash_lmhead_topk bit for bit and
    valid on every row against fp32 logits; h and every edge score match the oracle on those
    candidates."""
    inp = host_inputs(name)
    w = inp.workload
    d = P.to_device(inp, dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    lm = (torch.randn((w.V, w.H), generator=g, device=dev) / w.H ** 0.5).to(torch.bfloat16)
    ids, un, h, e = ds.dflash_selector_lmhead(d["hidden"], lm, d["w_proj"], d["pred_cb"],
                                              d["succ_cb"], d["anchors"], w.K, softcap=w.softcap)
    ids2, un2 = ds.dflash_lmhead_topk(d["hidden"], lm, w.K, softcap=w.softcap)
    torch.cuda.synchronize(dev)
    assert torch.equal(ids, ids2)
    assert torch.equal(un.view(torch.int32), un2.view(torch.int32))
    P.assert_lmhead_valid_every_row(ids, un, d["hidden"], lm, w.K, f"{name} draft step",
                                    softcap=w.softcap)
    P.assert_projection(P.bits(h), P.bits(inp.hidden), P.bits(inp.w_proj), f"{name} h")
    ref_e = oracle.edges(P.bits(inp.pred_cb), P.bits(inp.succ_cb), ids.cpu().numpy(),
                         un.cpu().numpy(), P.bits(h), inp.anchors)
    P.assert_close(e.cpu().numpy(), ref_e, f"{name} edges")
    del d, lm
    _status_clean()


def test_wait_timeout_is_reported_and_the_context_survives(dev):
    """The failure path of the bounded waits, without a fault: a wait on an mbarrier that
    nothing arrives on, then an edge CTA's wait in the fused selector's ready queue for a tile
    nothing pushes, each give up after about a second and set the timeout bit; afterwards the
    same context still runs the top-k and the fused selector (ready queue included)
    correctly."""
    import time
    lib = _native.load()
    ds.dflash_device_status(clear=True)
    t0 = time.perf_counter()
    _native.check(lib.dflash_selftest_wait_timeout())
    dt = time.perf_counter() - t0
    assert ds.dflash_device_status(clear=True) & _native.DEVICE_TIMEOUT
    assert 1.5 < dt < 60.0, dt
    x = np.random.default_rng(3).standard_normal((2, 3, 5000)).astype(np.float32)
    _topk_case(dev, x, 8, "top-k after a timeout")
    _selector_check(dev, host_inputs("small_ties"), "fused selector after a timeout")
    _status_clean()


@pytest.mark.parametrize("entry", ["selector_lmhead", "selector_forward"])
def test_draft_step_cuda_graph_replay(dev, entry):
    """The draft step captured once in a CUDA graph and replayed on fresh inputs copied into
    the captured buffers gives, bit for bit, what eager calls give."""
    R, S, K, V, H, rank = 6, 7, 16, 5000, 256, 64
    g = torch.Generator().manual_seed(77)
    lm = _bf16(torch.randn(V, H, generator=g) / H ** 0.5).to(dev)
    wp = _bf16(torch.randn(rank, H, generator=g) / H ** 0.5).to(dev)
    pc = _bf16(torch.randn(V, rank, generator=g) / rank ** 0.5).to(dev)
    sc = _bf16(torch.randn(V, rank, generator=g) / rank ** 0.5).to(dev)
    hid = torch.empty((R, S, H), dtype=torch.bfloat16, device=dev)
    anchors = torch.empty((R,), dtype=torch.int32, device=dev)
    cand = torch.empty((R, S, K), dtype=torch.int32, device=dev)
    unary = torch.empty((R, S, K), dtype=torch.float32, device=dev)
    h = torch.empty((R, S, rank), dtype=torch.bfloat16, device=dev)
    edges = torch.empty((R, S, K, K), dtype=torch.float32, device=dev)
    ws = torch.empty(ds.dflash_selector_lmhead_workspace_bytes(R, S, V, K), dtype=torch.uint8,
                     device=dev)

    def fresh(seed):
        gg = torch.Generator().manual_seed(seed)
        hid.copy_(_bf16(torch.randn(R, S, H, generator=gg)))
        anchors.copy_(torch.randint(0, V, (R,), generator=gg, dtype=torch.int32))
        cand.copy_(torch.randint(0, V, (R, S, K), generator=gg, dtype=torch.int32))
        unary.copy_(torch.randn(R, S, K, generator=gg))

    def call():
        if entry == "selector_lmhead":
            ds.dflash_selector_lmhead(hid, lm, wp, pc, sc, anchors, K, cand, unary, h, edges, ws)
        else:
            ds.dflash_selector_forward(cand, unary, hid, anchors, wp, pc, sc, h, edges)

    fresh(0)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        call()                                       # eager warm-up on a side stream
    torch.cuda.current_stream(dev).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for seed in (1, 2):
        fresh(seed)
        graph.replay()
        torch.cuda.synchronize(dev)
        got = [x.clone() for x in (cand, unary, h, edges)]
        fresh(seed)
        call()
        torch.cuda.synchronize(dev)
        for a, b in zip(got, (cand, unary, h, edges)):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"{entry} replay {seed}"
    _status_clean()


@pytest.mark.parametrize("name", ["small_ties", "ragged"])
def test_selector_request_chunks_equal_one_call(dev, name):
    """The end-to-end benchmark runs the fused selector on request chunks. Every kernel's
    per-row arithmetic is independent of how many rows a call holds, so chunked calls must
    give exactly the results of one call."""
    inp = host_inputs(RAGGED if name == "ragged" else name)
    w = inp.workload
    d = P.to_device(inp, dev)
    whole = ds.dflash_selector(d["logits"], d["hidden"], d["w_proj"], d["pred_cb"],
                               d["succ_cb"], d["anchors"], w.K)
    cuts = [0, 1, w.R // 2, w.R] if w.R > 2 else [0, 1, w.R]
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        if a == b:
            continue
        # Views: the logits and anchors need only 4-byte alignment; hidden (H % 8 == 0) stays
        # 16-byte aligned under any request slice.
        parts.append(ds.dflash_selector(d["logits"][a:b], d["hidden"][a:b], d["w_proj"],
                                        d["pred_cb"], d["succ_cb"], d["anchors"][a:b], w.K))
    torch.cuda.synchronize(dev)
    for i, name_i in enumerate(["ids", "unary", "h", "edges"]):
        got = torch.cat([pt[i] for pt in parts], dim=0)
        assert torch.equal(got.view(torch.uint8), whole[i].view(torch.uint8)), name_i
    _status_clean()


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_topk_logits_off_16_byte_boundary(dev, offset):
    """Logits that start 4, 8 or 12 bytes past a 16-byte boundary (a slice of requests out of
    a larger array): the top-k must find the boundaries itself and give the oracle's result,
    alone and inside the fused selector."""
    rng = np.random.default_rng(40 + offset)
    for (R, S, V, K) in [(3, 5, 1001, 8), (2, 3, 70003, 32), (4, 2, 17, 5)]:
        x = (rng.standard_normal((R, S, V)) * 3).astype(np.float32)
        x[0, 0, ::7] = 2.0                                    # ties
        base = torch.empty(R * S * V + 8, dtype=torch.float32, device=dev)
        view = base[offset:offset + R * S * V].view(R, S, V)
        view.copy_(torch.from_numpy(x))
        assert view.data_ptr() % 16 == 4 * offset
        ids, un = ds.dflash_topk_candidates(view, K)
        ref_ids, ref_un = oracle.topk(x, K)
        P.assert_ids_equal(ids.cpu().numpy(), ref_ids, f"offset {offset} R={R} V={V}")
        P.assert_close(un.cpu().numpy(), ref_un, f"offset {offset} R={R} V={V}")
    inp = host_inputs("small_ties")
    w = inp.workload
    d = P.to_device(inp, dev)
    base = torch.empty(d["logits"].numel() + 8, dtype=torch.float32, device=dev)
    view = base[offset:offset + d["logits"].numel()].view(d["logits"].shape)
    view.copy_(d["logits"])
    got = ds.dflash_selector(view, d["hidden"], d["w_proj"], d["pred_cb"], d["succ_cb"],
                             d["anchors"], w.K)
    want = ds.dflash_selector(d["logits"], d["hidden"], d["w_proj"], d["pred_cb"], d["succ_cb"],
                              d["anchors"], w.K)
    torch.cuda.synchronize(dev)
    for a, b in zip(got, want):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    _status_clean()


def test_candidate_selector_module(dev):
    """The module-style holder runs the same calls: forward equals dflash_selector_forward,
    select equals dflash_selector, both bit for bit."""
    inp = host_inputs("small_ties")
    w = inp.workload
    d = P.to_device(inp, dev)
    sel = ds.CandidateSelector(w.H, w.V, w.rank, w.K, device=dev)
    sel.predecessor_codebook.copy_(d["pred_cb"])
    sel.successor_codebook.copy_(d["succ_cb"])
    sel.hidden_projection_weight.copy_(d["w_proj"])
    ids, un, edges = sel.select(d["logits"], d["hidden"], d["anchors"])
    r_ids, r_un, _, r_e = ds.dflash_selector(d["logits"], d["hidden"], d["w_proj"], d["pred_cb"],
                                             d["succ_cb"], d["anchors"], w.K)
    e2 = sel(ids, un, d["hidden"], d["anchors"])
    torch.cuda.synchronize(dev)
    assert torch.equal(ids, r_ids) and torch.equal(un.view(torch.int32), r_un.view(torch.int32))
    assert torch.equal(edges.view(torch.int32), r_e.view(torch.int32))
    assert torch.equal(e2.view(torch.int32), r_e.view(torch.int32))
    path, tokens, _ = sel.best_path(edges, ids)
    ref_path, ref_tokens, _ = oracle.best_path(edges.cpu().numpy(), ids.cpu().numpy())
    P.assert_ids_equal(tokens.cpu().numpy(), ref_tokens, "module best path tokens")
    lm = (torch.randn((w.V, w.H), device=dev) / w.H ** 0.5).to(torch.bfloat16)
    c_ids, c_un = sel.compute_candidates(d["hidden"], lm)
    l_ids, l_un, l_e = sel.select_from_lm_head(d["hidden"], lm, d["anchors"])
    torch.cuda.synchronize(dev)
    assert torch.equal(c_ids, l_ids) and torch.equal(c_un.view(torch.int32), l_un.view(torch.int32))
    assert l_e.shape == (w.R, w.S, w.K, w.K)
    _status_clean()


# ----------------------------------------------------------------------------- robustness

def test_topk_fuzz_shapes(dev):
    """Seeded random shapes (rows, V, K) against the oracle: spans, row splits and ragged
    heads and tails land in many different places."""
    rng = np.random.default_rng(2024)
    for trial in range(24):
        V = int(rng.choice([int(rng.integers(1, 200)), int(rng.integers(200, 70000))]))
        K = int(rng.integers(1, min(32, V) + 1))
        R, S = int(rng.integers(1, 6)), int(rng.integers(1, 9))
        scale = float(rng.choice([0.5, 3.0, 40.0]))
        x = (rng.standard_normal((R, S, V)) * scale).astype(np.float32)
        if trial % 3 == 0:
            x = np.round(x)                               # ties
        _topk_case(dev, x, K, f"fuzz {trial}: R={R} S={S} V={V} K={K}")


def test_selector_concurrent_streams(dev):
    """Two host threads call the fused selector at once on two streams. The shared side
    stream of the projection must not mix their work: each result equals a lone call's."""
    import threading
    inp = [wl.make_inputs(RAGGED, seed=s) for s in (0, 1)]
    w = RAGGED
    d = [P.to_device(i, dev) for i in inp]
    ref = [ds.dflash_selector(x["logits"], x["hidden"], x["w_proj"], x["pred_cb"], x["succ_cb"],
                              x["anchors"], w.K) for x in d]
    torch.cuda.synchronize(dev)
    out = [None, None]
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]

    def run(i):
        torch.cuda.set_device(dev)
        with torch.cuda.stream(streams[i]):
            for _ in range(20):
                out[i] = ds.dflash_selector(d[i]["logits"], d[i]["hidden"], d[i]["w_proj"],
                                            d[i]["pred_cb"], d[i]["succ_cb"], d[i]["anchors"],
                                            w.K, stream=streams[i])
        streams[i].synchronize()

    th = [threading.Thread(target=run, args=(i,)) for i in (0, 1)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    for i in (0, 1):
        for a, b in zip(out[i], ref[i]):
            assert torch.equal(a, b), f"thread {i}: a result differs from the lone call"
    _status_clean()
