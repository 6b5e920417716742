"""The every-row LM-head checker used at full size on the GPU, run here on the CPU: it
accepts the exact top-k of small cases (with and without the soft cap) and rejects each
planted mistake: a clear winner swapped out, a unary value moved, the order reversed, an id
repeated."""
import pytest
import torch

import parity as P

ROWS, H, V, K = 300, 96, 5000, 8


@pytest.fixture(scope="module")
def case():
    g = torch.Generator().manual_seed(0)
    hid = torch.randn(ROWS, H, generator=g).to(torch.bfloat16)
    lm = (torch.randn(V, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    f = hid.double() @ lm.double().t()
    vals, order = torch.sort(f, dim=1, descending=True, stable=True)
    return hid, lm, order, order[:, :K].int(), vals[:, :K].float()


def test_exact_top_k_passes(case):
    hid, lm, _, ids, un = case
    P.assert_lmhead_valid_every_row(ids, un, hid, lm, K, "exact")
    cap = 3.0
    P.assert_lmhead_valid_every_row(ids, cap * torch.tanh(un / cap), hid, lm, K, "capped",
                                    softcap=cap)


def _planted(case, kind):
    _, _, order, ids, un = case
    if kind == "winner swapped out":
        bad = ids.clone()
        bad[5, 0] = int(order[5, K + 50])
        return bad, un
    if kind == "unary moved":
        u = un.clone()
        u[7, 3] += 0.5
        return ids, u
    if kind == "order reversed":
        return ids.flip(1), un.flip(1)
    return torch.cat([ids[:, :1], ids[:, :-1]], 1), un       # an id repeated


@pytest.mark.parametrize("kind", ["winner swapped out", "unary moved", "order reversed",
                                  "id repeated"])
def test_planted_mistake_is_caught(case, kind):
    hid, lm = case[0], case[1]
    ids, un = _planted(case, kind)
    with pytest.raises(AssertionError):
        P.assert_lmhead_valid_every_row(ids, un, hid, lm, K, kind)
