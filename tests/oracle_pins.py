"""Pins for the CPU oracle: checks against facts the oracle's own code does not supply.

Each check takes an oracle handle, so tests/test_oracle_mutants.py can run the same
checks against deliberately broken builds. The facts are of four kinds:
  * hand-derived golden cases (tests/golden/*.txt, each citing its passage);
  * brute force on tiny inputs (all K-subsets);
  * closed forms and invariants (zero codebooks, rank-1, p = 0 rows identical, ...);
  * special cases that reduce to a library routine (stable argsort when K = V, numpy
    fp64 matmul / einsum, torch's float32 -> bf16 rounding).
The order used for top-k is the selector's candidate order: logit descending, then token
id ascending, with -0 == +0, NaN (sign clear) above +inf and NaN (sign set) below -inf.
"""

from __future__ import annotations

import itertools
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------- helpers

def _parse_float(tok: str) -> np.float32:
    t = tok.strip().lower()
    if t in ("nan", "+nan"):
        return np.float32(np.nan)
    if t == "-nan":
        return np.copysign(np.float32(np.nan), np.float32(-1.0))
    return np.float32(float(t))


def _golden_lines(name: str):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def _sort_key(v: float, i: int):
    """A tuple that Python orders the way the candidate order does (smaller = first)."""
    if math.isnan(v):
        cls = 0 if math.copysign(1.0, v) > 0 else 2
        return (cls, 0.0, i)
    return (1, -float(v) + 0.0, i)   # + 0.0 folds -0 into +0


def bits_to_float(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def float_to_bf16_bits_exact(x: np.ndarray) -> np.ndarray:
    """bf16 bits of float32 values that are already exactly bf16 (checked)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value is not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def _bf16_neighbours(bits: int):
    """The bf16 values just below and just above a finite bf16 (by bit pattern)."""
    f = float(bits_to_float(np.array([bits]))[0])
    if f == 0.0:
        tiny = float(bits_to_float(np.array([1]))[0])
        return -tiny, tiny
    up = bits + 1 if f > 0 else bits - 1
    dn = bits - 1 if f > 0 else bits + 1
    return (float(bits_to_float(np.array([dn & 0xFFFF]))[0]),
            float(bits_to_float(np.array([up & 0xFFFF]))[0]))


def check_nearest_bf16(x: float, bits: int) -> None:
    """bits must be the bf16 nearest to x, and on a tie the one with an even mantissa."""
    y = float(bits_to_float(np.array([bits]))[0])
    lo, hi = _bf16_neighbours(bits)
    d = abs(y - x)
    assert d <= abs(lo - x) and d <= abs(hi - x), (x, hex(bits), y, lo, hi)
    if d == abs(lo - x) or d == abs(hi - x):
        assert bits % 2 == 0, ("tie not rounded to even", x, hex(bits))


# ----------------------------------------------------------------------------- top-k

def pin_topk_golden(orc) -> None:
    for line in _golden_lines("topk_order.txt"):
        k_s, logits_s, ids_s = [p.strip() for p in line.split(";")]
        K = int(k_s)
        x = np.array([_parse_float(t) for t in logits_s.split()], dtype=np.float32)
        want = [int(t) for t in ids_s.split()]
        ids, unary = orc.topk(x[None, :], K)
        assert ids[0].tolist() == want, (line, ids[0].tolist())
        got = unary[0]
        ref = x[want]
        assert np.array_equal(got, ref, equal_nan=True), (line, got, ref)


def _brute_force_topk(x: np.ndarray, K: int) -> list[int]:
    """Among all K-subsets, the one whose every member precedes every non-member; then
    its members in pairwise-precedence order."""
    V = len(x)
    keys = [_sort_key(float(x[i]), i) for i in range(V)]
    winners = []
    for sub in itertools.combinations(range(V), K):
        inside = set(sub)
        if all(keys[a] < keys[b] for a in sub for b in range(V) if b not in inside):
            winners.append(sub)
    assert len(winners) == 1
    members = list(winners[0])
    # order: a member's position = the number of members that precede it
    pos = {m: sum(keys[o] < keys[m] for o in members) for m in members}
    return [m for m, _ in sorted(pos.items(), key=lambda t: t[1])]


def pin_topk_bruteforce(orc, trials: int = 300, seed: int = 1) -> None:
    rng = np.random.default_rng(seed)
    pool = np.array([-1.0, -0.0, 0.0, 0.5, 1.0, 2.0, np.inf, -np.inf], dtype=np.float32)
    for _ in range(trials):
        V = int(rng.integers(1, 8))
        K = int(rng.integers(1, V + 1))
        x = pool[rng.integers(0, len(pool), size=V)].copy()
        if rng.random() < 0.2:
            x[rng.integers(0, V)] = np.float32(np.nan)
        if rng.random() < 0.2:
            x[rng.integers(0, V)] = np.copysign(np.float32(np.nan), np.float32(-1))
        ids, _ = orc.topk(x[None, :], K)
        assert ids[0].tolist() == _brute_force_topk(x, K), (x.tolist(), K, ids[0].tolist())


def pin_topk_stable_sort(orc, seed: int = 2) -> None:
    """K = V: the candidate order is a stable descending sort, numpy's argsort(kind=stable)."""
    rng = np.random.default_rng(seed)
    for V in (1, 2, 7, 64, 1000):
        x = rng.integers(-4, 5, size=(3, V)).astype(np.float32)   # many ties
        x[x == 0] = np.where(rng.random((x == 0).sum()) < 0.5, -0.0, 0.0)
        ids, unary = orc.topk(x, V)
        for r in range(3):
            want = np.argsort(-x[r], kind="stable")
            assert np.array_equal(ids[r], want), (V, r)
            assert np.array_equal(unary[r], x[r][want])


def pin_topk_invariants(orc, seed: int = 3) -> None:
    """Random rows with heavy ties: the output is K distinct ids in [0, V), unary equals
    the logits at those ids, the K are in order, and every other id comes after the K-th."""
    rng = np.random.default_rng(seed)
    for V, K in ((5000, 32), (4099, 17), (33, 32), (40, 1)):
        x = np.round(rng.standard_normal((4, V)) * 4).astype(np.float32) / 4
        ids, unary = orc.topk(x, K)
        for r in range(4):
            sel = ids[r].tolist()
            assert len(set(sel)) == K and all(0 <= i < V for i in sel)
            assert np.array_equal(unary[r], x[r][sel])
            keys = [_sort_key(float(x[r][i]), i) for i in sel]
            assert keys == sorted(keys)
            kth = keys[-1]
            rest = np.setdiff1d(np.arange(V), sel)
            assert all(_sort_key(float(x[r][i]), int(i)) > kth for i in rest)


def pin_topk_logits_processor_golden(orc) -> None:
    for line in _golden_lines("logits_processor.txt"):
        head, logits_s, ids_s, un_s = [p.strip() for p in line.split(";")]
        cap, scale, K = head.split()
        x = np.array([_parse_float(t) for t in logits_s.split()], dtype=np.float32)
        ids, unary = orc.topk(x[None, :], int(K), softcap=float(cap), scale=float(scale))
        assert ids[0].tolist() == [int(t) for t in ids_s.split()], (line, ids[0].tolist())
        want = np.array([float(t) for t in un_s.split()], dtype=np.float32)
        assert np.allclose(unary[0], want, rtol=1e-6, atol=0), (line, unary[0], want)


def pin_topk_logits_processor_vs_numpy(orc, seed: int = 13) -> None:
    """Against numpy's tanh: unary = float32(scale * cap * tanh(x / cap)), ids unchanged."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((6, 3000)) * 40).astype(np.float32)
    ids_raw, un_raw = orc.topk(x, 16)
    for cap, scale in ((30.0, 1.0), (10.0, 0.25), (0.0, 2.0), (50.0, 3.0)):
        ids, un = orc.topk(x, 16, softcap=cap, scale=scale)
        assert np.array_equal(ids, ids_raw)
        v = un_raw.astype(np.float64)
        want = (cap * np.tanh(v / cap) if cap > 0 else v) * scale
        assert np.allclose(un, want.astype(np.float32), rtol=2e-7, atol=1e-30)


# ----------------------------------------------------------------------------- bf16 rounding

def pin_bf16_round_cases(orc) -> None:
    cases = [   # a list, not a dict: 0.0 and -0.0 are equal keys
        (1.0, 0x3F80), (-1.0, 0xBF80), (0.0, 0x0000), (-0.0, 0x8000),
        (1 + 2**-8, 0x3F80),                # tie -> even (down)
        (1 + 3 * 2**-8, 0x3F82),            # tie -> even (up)
        (1 + 2**-8 + 2**-30, 0x3F81),       # just above the tie: one rounding, not two
        (1 + 2**-8 - 2**-40, 0x3F80),       # just below the tie
        (-(1 + 2**-8 + 2**-30), 0xBF81),
        (2.0**-133, 0x0001),                # smallest bf16 subnormal
        (2.0**-134, 0x0000),                # half of it: tie -> even (zero)
        (1.5 * 2.0**-133, 0x0002),          # tie between 1 and 2 subnormal steps -> even
        (2.0**-126, 0x0080),                # smallest normal
        (3.3895313892515355e38, 0x7F7F),    # largest finite bf16
        (3.40e38, 0x7F80),                  # rounds past the largest finite value -> inf
        (math.inf, 0x7F80), (-math.inf, 0xFF80),
    ]
    for x, want in cases:
        got = orc.bf16_round(x)
        assert got == want, (x, hex(got), hex(want))
    assert (orc.bf16_round(math.nan) & 0x7FFF) > 0x7F80


def pin_bf16_round_vs_torch(orc, seed: int = 4) -> None:
    """For float32 inputs, one rounding to bf16 is what torch's float32 -> bf16 cast does."""
    rng = np.random.default_rng(seed)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(1000) * 1e-39).astype(np.float32),     # subnormals
        rng.integers(0, 2**31, size=2000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.bf16_round(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, want)


def pin_bf16_round_nearest(orc, seed: int = 5) -> None:
    """For doubles with more bits than binary32 holds: the result is a nearest bf16, and
    an even one on ties."""
    rng = np.random.default_rng(seed)
    xs = rng.standard_normal(3000) * np.exp2(rng.integers(-20, 20, size=3000))
    for x in xs:
        check_nearest_bf16(float(x), orc.bf16_round(float(x)))


# ----------------------------------------------------------------------------- projection

def pin_projection_golden(orc) -> None:
    for line in _golden_lines("projection_worked.txt"):
        dims, w_s, x_s, h_s, bits_s = [p.strip() for p in line.split(";")]
        rank, H = (int(t) for t in dims.split())
        w = np.array([float(t) for t in w_s.split()], dtype=np.float32).reshape(rank, H)
        x = np.array([float(t) for t in x_s.split()], dtype=np.float32).reshape(1, H)
        h = orc.projection(float_to_bf16_bits_exact(x), float_to_bf16_bits_exact(w))
        want_bits = [int(t, 16) for t in bits_s.split()]
        want_vals = [float(t) for t in h_s.split()]
        assert h[0].tolist() == want_bits, (line, [hex(b) for b in h[0]])
        assert bits_to_float(h[0]).tolist() == want_vals


def pin_projection_closed_forms(orc, seed: int = 6) -> None:
    rng = np.random.default_rng(seed)
    H, rank, rows = 48, 16, 5
    x = float_to_bf16_bits_exact(
        torch.randn(rows, H, generator=torch.Generator().manual_seed(seed))
        .to(torch.bfloat16).float().numpy())
    # W = 0 -> h = 0
    h = orc.projection(x, np.zeros((rank, H), dtype=np.uint16))
    assert np.all(bits_to_float(h) == 0)
    # W = I (rank = H) -> h = hidden exactly
    eye = float_to_bf16_bits_exact(np.eye(H, dtype=np.float32))
    assert np.array_equal(orc.projection(x, eye), x)
    # one-hot rows: h_j = hidden[perm[j]] * scale_j, with power-of-two scales (exact)
    perm = rng.permutation(H)[:rank]
    scale = np.exp2(rng.integers(-3, 4, size=rank)).astype(np.float32)
    w = np.zeros((rank, H), dtype=np.float32)
    w[np.arange(rank), perm] = scale
    h = orc.projection(x, float_to_bf16_bits_exact(w))
    want = bits_to_float(x)[:, perm] * scale[None, :]
    assert np.array_equal(bits_to_float(h), want)


def pin_projection_vs_numpy(orc, seed: int = 7) -> None:
    """Against numpy's fp64 matmul: h is the nearest bf16 to W.hidden (ties to even)."""
    g = torch.Generator().manual_seed(seed)
    rows, H, rank = 6, 200, 24
    xb = torch.randn(rows, H, generator=g).to(torch.bfloat16)
    wb = (torch.randn(rank, H, generator=g) / math.sqrt(H)).to(torch.bfloat16)
    xbits = xb.view(torch.int16).numpy().view(np.uint16)
    wbits = wb.view(torch.int16).numpy().view(np.uint16)
    h, exact = orc.projection(xbits, wbits, want_exact=True)
    ref = xb.double().numpy() @ wb.double().numpy().T
    assert np.allclose(exact, ref, rtol=0, atol=1e-12)
    for r in range(rows):
        for j in range(rank):
            check_nearest_bf16(float(ref[r, j]), int(h[r, j]))


# ----------------------------------------------------------------------------- edges

def _read_edges_fixture():
    kv = {}
    for line in _golden_lines("edges_worked.txt"):
        key, *vals = line.split()
        kv[key] = [float(v) for v in vals]
    V, rank = int(kv["V"][0]), int(kv["rank"][0])
    R, S, K = int(kv["R"][0]), int(kv["S"][0]), int(kv["K"][0])
    f = lambda k, shape: np.array(kv[k], dtype=np.float32).reshape(shape)  # noqa: E731
    return dict(
        pred=float_to_bf16_bits_exact(f("pred_cb", (V, rank))),
        succ=float_to_bf16_bits_exact(f("succ_cb", (V, rank))),
        anchors=np.array(kv["anchors"], dtype=np.int32),
        cand=np.array(kv["cand"], dtype=np.int32).reshape(R, S, K),
        unary=f("unary", (R, S, K)),
        h=float_to_bf16_bits_exact(f("h", (R, S, rank))),
        edges=f("edges", (R, S, K, K)),
    )


def pin_edges_golden(orc) -> None:
    d = _read_edges_fixture()
    e = orc.edges(d["pred"], d["succ"], d["cand"], d["unary"], d["h"], d["anchors"])
    assert np.array_equal(e, d["edges"]), (e, d["edges"])


def _random_edge_inputs(seed, R=3, S=5, K=6, V=50, rank=16, distinct_pred=True):
    g = torch.Generator().manual_seed(seed)
    bf = lambda *s: (torch.randn(*s, generator=g) / 4).to(torch.bfloat16)  # noqa: E731
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    rng = np.random.default_rng(seed)
    cand = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(S)])
                     for _ in range(R)]).astype(np.int32)
    return dict(
        pred=bits(bf(V, rank)), succ=bits(bf(V, rank)), cand=cand,
        unary=rng.standard_normal((R, S, K)).astype(np.float32),
        h=bits(bf(R, S, rank)), anchors=rng.integers(0, V, R).astype(np.int32))


def pin_edges_zero_codebooks(orc, seed: int = 8) -> None:
    d = _random_edge_inputs(seed)
    z = np.zeros_like(d["pred"])
    for pred, succ in ((z, d["succ"]), (d["pred"], z), (z, z)):
        e = orc.edges(pred, succ, d["cand"], d["unary"], d["h"], d["anchors"])
        want = np.broadcast_to(d["unary"][:, :, None, :], e.shape)
        assert np.array_equal(e, want)
    e = orc.edges(d["pred"], d["succ"], d["cand"], d["unary"], np.zeros_like(d["h"]),
                  d["anchors"])
    assert np.array_equal(e, np.broadcast_to(d["unary"][:, :, None, :], e.shape))


def pin_edges_rank1(orc, seed: int = 9) -> None:
    """rank = 1 closed form: E[r,p,q,c] = unary[r,p,c] + a[pid] * h[r,p] * b[cid]."""
    d = _random_edge_inputs(seed, rank=1)
    a = bits_to_float(d["pred"])[:, 0].astype(np.float64)
    b = bits_to_float(d["succ"])[:, 0].astype(np.float64)
    h = bits_to_float(d["h"])[..., 0].astype(np.float64)
    e = orc.edges(d["pred"], d["succ"], d["cand"], d["unary"], d["h"], d["anchors"])
    R, S, K = d["cand"].shape
    for r in range(R):
        for p in range(S):
            for q in range(K):
                pid = d["anchors"][r] if p == 0 else d["cand"][r, p - 1, q]
                for c in range(K):
                    want = np.float32(d["unary"][r, p, c] + a[pid] * h[r, p] * b[d["cand"][r, p, c]])
                    assert e[r, p, q, c] == want


def pin_edges_subnormal_products(orc) -> None:
    """Closed form with subnormal codebook entries: pred = 2^-130 (a bf16 subnormal), h = 2^100,
    succ = 2^20, so every term is 2^-10 and every score is rank * 2^-10 exactly. A flush of
    subnormal inputs, or a product taken in a format without them, gives 0 instead."""
    R, S, K, V, rank = 2, 3, 2, 4, 16
    pred = np.full((V, rank), 0x0008, dtype=np.uint16)       # 8 * 2^-133
    succ = np.full((V, rank), 0x4980, dtype=np.uint16)       # exponent 147: 2^20
    h = np.full((R, S, rank), 0x7180, dtype=np.uint16)       # exponent 227: 2^100
    assert bits_to_float(pred)[0, 0] == np.float32(2.0 ** -130)
    cand = np.array([[[0, 1], [2, 3], [1, 2]], [[3, 2], [1, 0], [0, 3]]], dtype=np.int32)
    e = orc.edges(pred, succ, cand, np.zeros((R, S, K), np.float32), h,
                  np.array([1, 2], dtype=np.int32))
    assert np.all(e == np.float32(rank * 2.0 ** -10)), e


def pin_edges_structure(orc, seed: int = 10) -> None:
    """At p = 0 every predecessor row is the same (the anchor). For p > 0, row q depends
    only on cand[r, p-1, q]: equal predecessors give equal rows, and changing the
    candidates at p-1 changes nothing at p+1."""
    d = _random_edge_inputs(seed)
    e = orc.edges(d["pred"], d["succ"], d["cand"], d["unary"], d["h"], d["anchors"])
    assert np.all(e[:, 0] == e[:, 0, :1, :])
    cand2 = d["cand"].copy()
    cand2[:, 1, 1] = cand2[:, 1, 0]          # duplicate the predecessor of q=1 at p=2
    e2 = orc.edges(d["pred"], d["succ"], cand2, d["unary"], d["h"], d["anchors"])
    assert np.array_equal(e2[:, 2, 1], e2[:, 2, 0])
    assert np.array_equal(e2[:, 3:], e[:, 3:])
    assert np.array_equal(e2[:, :1], e[:, :1])


def pin_edges_vs_einsum(orc, seed: int = 11) -> None:
    """Against numpy's fp64 einsum of the definition, on independent random codebooks."""
    d = _random_edge_inputs(seed, R=4, S=6, K=5, V=40, rank=24)
    P = bits_to_float(d["pred"]).astype(np.float64)
    Sb = bits_to_float(d["succ"]).astype(np.float64)
    h = bits_to_float(d["h"]).astype(np.float64)
    prev = np.concatenate([np.repeat(d["anchors"][:, None, None], d["cand"].shape[2], axis=2),
                           d["cand"][:, :-1]], axis=1)            # [R, S, K] predecessor ids
    G = P[prev] * h[:, :, None, :]                              # [R, S, q, rank]
    want = np.einsum("rsqj,rscj->rsqc", G, Sb[d["cand"]]) + d["unary"][:, :, None, :]
    e = orc.edges(d["pred"], d["succ"], d["cand"], d["unary"], d["h"], d["anchors"])
    assert np.allclose(e, want.astype(np.float32), rtol=1e-6, atol=1e-6)


def pin_selector_composes(orc, seed: int = 12) -> None:
    """The all-in-one call equals top-k, then projection, then edges."""
    rng = np.random.default_rng(seed)
    R, S, K, V, H, rank = 2, 3, 4, 300, 32, 8
    g = torch.Generator().manual_seed(seed)
    bits = lambda t: t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)  # noqa
    logits = rng.standard_normal((R, S, V)).astype(np.float32)
    hid, w = bits(torch.randn(R, S, H, generator=g)), bits(torch.randn(rank, H, generator=g) / 6)
    a, b = bits(torch.randn(V, rank, generator=g) / 3), bits(torch.randn(V, rank, generator=g) / 3)
    anc = rng.integers(0, V, R).astype(np.int32)
    ids, un, h, e = orc.selector(logits, hid, w, a, b, anc, K, softcap=3.0, scale=0.5)
    ids2, un2 = orc.topk(logits, K, softcap=3.0, scale=0.5)
    h2 = orc.projection(hid, w)
    e2 = orc.edges(a, b, ids2, un2, h2, anc)
    assert np.array_equal(ids, ids2) and np.array_equal(un, un2)
    assert np.array_equal(h, h2) and np.array_equal(e, e2)


def pin_lmhead_topk_vs_numpy(orc, seed: int = 14) -> None:
    """Against numpy: fp64 matmul of the bf16 values, then a stable sort by (-logit, id)."""
    g = torch.Generator().manual_seed(seed)
    rows, H, V, K = 5, 72, 300, 7
    x = torch.randn(rows, H, generator=g).to(torch.bfloat16)
    w = (torch.randn(V, H, generator=g) / 8).to(torch.bfloat16)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    ids, un, logits = orc.lmhead_topk(bits(x), bits(w), K, softcap=4.0, scale=0.5,
                                      want_logits=True)
    ref = x.double().numpy() @ w.double().numpy().T
    assert np.allclose(logits, ref, rtol=0, atol=1e-12)
    for r in range(rows):
        want = np.argsort(-ref[r], kind="stable")[:K]
        assert ids[r].tolist() == want.tolist()
        v = ref[r][want].astype(np.float32).astype(np.float64)
        assert np.allclose(un[r], (4.0 * np.tanh(v / 4.0) * 0.5).astype(np.float32), rtol=2e-7)


def pin_lmhead_topk_one_hot(orc) -> None:
    """A one-hot hidden state picks one column of the LM head: logits = lm_head[:, i]."""
    H, V, K = 16, 40, 5
    w = np.arange(V * H, dtype=np.float32).reshape(V, H) % 7 - 3.0       # ties on purpose
    x = np.zeros((1, H), dtype=np.float32)
    x[0, 3] = 1.0
    ids, un = orc.lmhead_topk(float_to_bf16_bits_exact(x), float_to_bf16_bits_exact(w), K)
    col = w[:, 3]
    want = sorted(range(V), key=lambda v: (-col[v], v))[:K]
    assert ids[0].tolist() == want and np.array_equal(un[0], col[want])


def pin_best_path_golden(orc) -> None:
    """The hand-worked case of tests/golden/best_path_worked.txt, ties included."""
    K = S = 0
    entries, cands = [], []
    for line in _golden_lines("best_path_worked.txt"):
        tok = line.split()
        if tok[0] == "K":
            K = int(tok[1])
        elif tok[0] == "S":
            S = int(tok[1])
        elif tok[0] == "E":
            entries.append((int(tok[1]), int(tok[2]), int(tok[3]), float(tok[4])))
        elif tok[0] == "cand":
            cands.append((int(tok[1]), int(tok[2]), int(tok[3])))
        elif tok[0] == "path":
            want_path = [int(x) for x in tok[1:]]
        elif tok[0] == "tokens":
            want_tokens = [int(x) for x in tok[1:]]
        elif tok[0] == "score":
            want_score = float(tok[1])
    E = np.zeros((1, S, K, K), dtype=np.float32)
    for p_, q, c, v in entries:
        E[0, p_, q, c] = v
    cand = np.zeros((1, S, K), dtype=np.int32)
    for p_, c, i in cands:
        cand[0, p_, c] = i
    path, tokens, score = orc.best_path(E, cand)
    assert path[0].tolist() == want_path, path
    assert tokens[0].tolist() == want_tokens, tokens
    assert float(score[0]) == want_score, score


def _path_sum(E: np.ndarray, path) -> float:
    """Exact sum of a path's scores (p = 0 uses predecessor row 0)."""
    s = float(E[0, 0, path[0]])
    for p_ in range(1, len(path)):
        s += float(E[p_, path[p_ - 1], path[p_]])
    return s


def pin_best_path_bruteforce(orc, trials: int = 60, seed: int = 15) -> None:
    """Against every path on tiny lattices. Scores lie on a 1/8 grid in [-4, 4], so every
    fp32 sum is exact: the oracle's score must equal the best path sum, and so must the sum
    of the path it returns."""
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        S = int(rng.integers(1, 6))
        K = int(rng.integers(1, 5))
        R = 2
        E = (rng.integers(-32, 33, size=(R, S, K, K)) / 8.0).astype(np.float32)
        cand = rng.integers(0, 1000, size=(R, S, K)).astype(np.int32)
        path, tokens, score = orc.best_path(E, cand)
        for r in range(R):
            best = max(_path_sum(E[r], pth) for pth in itertools.product(range(K), repeat=S))
            assert float(score[r]) == best
            assert _path_sum(E[r], path[r].tolist()) == best
            assert tokens[r].tolist() == [int(cand[r, p_, path[r, p_]]) for p_ in range(S)]


def pin_best_path_independent_steps(orc, seed: int = 16) -> None:
    """With no pairwise term (E[p,q,c] = u[p,c] for every q, as zero codebooks give), the best
    path takes each step's best candidate, the first one on ties, and the score is the fp32
    sum of those, left to right."""
    rng = np.random.default_rng(seed)
    R, S, K = 4, 6, 8
    u = np.round(rng.standard_normal((R, S, K)) * 4).astype(np.float32)   # ties on purpose
    E = np.repeat(u[:, :, None, :], K, axis=2)
    cand = np.arange(R * S * K, dtype=np.int32).reshape(R, S, K)
    path, tokens, score = orc.best_path(E, cand)
    for r in range(R):
        want = [int(np.argmax(u[r, p_])) for p_ in range(S)]          # first maximum
        assert path[r].tolist() == want
        acc = np.float32(0)
        for p_ in range(S):
            acc = np.float32(acc + u[r, p_, want[p_]]) if p_ else u[r, 0, want[0]]
        assert score[r] == acc


def pin_best_path_single_candidate(orc) -> None:
    """K = 1: the only path; its score is the fp32 sum of E[p,0,0], left to right."""
    E = np.array([[[[0.5]], [[-2.25]], [[1e-3]]]], dtype=np.float32)
    cand = np.array([[[7], [8], [9]]], dtype=np.int32)
    path, tokens, score = orc.best_path(E, cand)
    assert path[0].tolist() == [0, 0, 0] and tokens[0].tolist() == [7, 8, 9]
    assert score[0] == np.float32(np.float32(np.float32(0.5) + np.float32(-2.25)) + np.float32(1e-3))


ALL_PINS = [
    pin_topk_golden, pin_topk_bruteforce, pin_topk_stable_sort, pin_topk_invariants,
    pin_topk_logits_processor_golden, pin_topk_logits_processor_vs_numpy,
    pin_bf16_round_cases, pin_bf16_round_vs_torch, pin_bf16_round_nearest,
    pin_projection_golden, pin_projection_closed_forms, pin_projection_vs_numpy,
    pin_edges_golden, pin_edges_zero_codebooks, pin_edges_rank1, pin_edges_subnormal_products,
    pin_edges_structure, pin_edges_vs_einsum, pin_selector_composes, pin_lmhead_topk_vs_numpy,
    pin_lmhead_topk_one_hot, pin_best_path_golden, pin_best_path_bruteforce,
    pin_best_path_independent_steps, pin_best_path_single_candidate,
]
