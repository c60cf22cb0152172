"""Pins for the oracle's router (softmax top-k gate ahead of the expert path).

The pages take routes as given and return the routing-weight gradient
("grad-route", fw-ai/DeepGEMM PR #9, Correctness coverage); the router read here
is softmax over all experts, the k largest probabilities (ties to the lower expert
id), weights renormalised to sum 1.  Each test pins the oracle to something other
than itself: torch float64 softmax/top-k and autograd, a closed form derived by
hand, finite differences, and hand-made ties.
"""
from __future__ import annotations

import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def _inputs(T=7, H=24, E=12, seed=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g, dtype=torch.float64)
    Wr = torch.randn(E, H, generator=g, dtype=torch.float64) / H ** 0.5
    return x, Wr


def _torch_router(x, Wr, k):
    l = x @ Wr.t()
    p = torch.softmax(l, dim=-1)
    top = torch.topk(p, k, dim=-1)
    w = top.values / top.values.sum(-1, keepdim=True)
    return l, top.indices, w


@pytest.mark.parametrize("k", [1, 3, 12])
def test_forward_matches_torch_softmax_topk(k):
    x, Wr = _inputs(seed=k)
    l_ref, ids_ref, w_ref = _torch_router(x, Wr, k)
    l, ids, w = oracle.router_forward(x, Wr, k, prec="f64")
    assert torch.equal(ids.long(), ids_ref)
    assert torch.allclose(l, l_ref, rtol=0, atol=1e-12)
    assert torch.allclose(w, w_ref, rtol=0, atol=1e-12)


def test_forward_f32_matches_f64():
    x, Wr = _inputs(T=16, H=64, E=32, seed=3)
    l64, ids64, w64 = oracle.router_forward(x, Wr, 4, prec="f64")
    l32, ids32, w32 = oracle.router_forward(x.float(), Wr.float(), 4, prec="f32")
    assert torch.equal(ids64, ids32)
    assert (w32.double() - w64).abs().max() < 1e-6
    assert (l32.double() - l64).abs().max() < 1e-5


def test_ties_go_to_the_lower_expert_id():
    # Rows 1, 4 and 6 of Wr are equal and give the largest logit; row 2 is second.
    H, E = 8, 8
    x = torch.ones(1, H, dtype=torch.float64)
    Wr = torch.zeros(E, H, dtype=torch.float64)
    for e in (1, 4, 6):
        Wr[e] = 0.5
    Wr[2] = 0.25
    _, ids, w = oracle.router_forward(x, Wr, 4, prec="f64")
    assert ids.tolist() == [[1, 4, 6, 2]]
    # three equal weights e^4 and one e^2, renormalised
    a, b = torch.exp(torch.tensor(4.0, dtype=torch.float64)), torch.exp(torch.tensor(2.0, dtype=torch.float64))
    want = torch.tensor([a, a, a, b]) / (3 * a + b)
    assert torch.allclose(w[0], want, rtol=0, atol=1e-15)


def test_invariants():
    x, Wr = _inputs(T=20, H=32, E=16, seed=5)
    l, ids, w = oracle.router_forward(x, Wr, 5, prec="f64")
    assert torch.allclose(w.sum(-1), torch.ones(20, dtype=torch.float64), atol=1e-14)
    assert (w[:, :-1] >= w[:, 1:]).all()
    for row in ids.tolist():
        assert len(set(row)) == 5
    # every selected logit is at least every unselected one
    for t in range(20):
        sel = set(ids[t].tolist())
        lo = min(l[t, e] for e in sel)
        hi = max((l[t, e] for e in range(16) if e not in sel), default=-1e30)
        assert lo >= hi


@pytest.mark.parametrize("k", [1, 2, 5])
def test_backward_matches_torch_autograd(k):
    x, Wr = _inputs(T=9, H=20, E=10, seed=10 + k)
    g = torch.Generator().manual_seed(99)
    dw = torch.randn(9, k, generator=g, dtype=torch.float64)
    xa = x.clone().requires_grad_(True)
    Wa = Wr.clone().requires_grad_(True)
    l = xa @ Wa.t()
    l.retain_grad()
    p = torch.softmax(l, dim=-1)
    ids = torch.topk(p.detach(), k, dim=-1).indices
    sel = torch.gather(p, 1, ids)
    w = sel / sel.sum(-1, keepdim=True)
    (w * dw).sum().backward()
    dl, dWr, dx = oracle.router_backward(x, Wr, ids.to(torch.int32), dw, prec="f64")
    assert torch.allclose(dl, l.grad, rtol=0, atol=1e-13)
    assert torch.allclose(dWr, Wa.grad, rtol=0, atol=1e-12)
    assert torch.allclose(dx, xa.grad, rtol=0, atol=1e-12)


def test_backward_closed_form():
    # With w the softmax of the selected logits only, dl_m = w_m (dw_m - <w, dw>) on
    # the selected experts and 0 elsewhere (the full-softmax normaliser cancels).
    x, Wr = _inputs(T=6, H=16, E=9, seed=21)
    k = 4
    _, ids, w = oracle.router_forward(x, Wr, k, prec="f64")
    dw = torch.randn(6, k, generator=torch.Generator().manual_seed(4), dtype=torch.float64)
    dl, _, _ = oracle.router_backward(x, Wr, ids, dw, prec="f64")
    want = torch.zeros(6, 9, dtype=torch.float64)
    for t in range(6):
        s = float((w[t] * dw[t]).sum())
        for j in range(k):
            want[t, int(ids[t, j])] = float(w[t, j]) * (float(dw[t, j]) - s)
    assert torch.allclose(dl, want, rtol=0, atol=1e-14)
    assert dl.sum(-1).abs().max() < 1e-14  # logit shifts leave the weights unchanged


def test_backward_finite_differences():
    x, Wr = _inputs(T=5, H=12, E=8, seed=31)
    k = 3
    _, ids0, _ = oracle.router_forward(x, Wr, k, prec="f64")
    dw = torch.randn(5, k, generator=torch.Generator().manual_seed(7), dtype=torch.float64)
    _, dWr, dx = oracle.router_backward(x, Wr, ids0, dw, prec="f64")
    g = torch.Generator().manual_seed(8)
    vx, vW = torch.randn(x.shape, generator=g, dtype=torch.float64), torch.randn(Wr.shape, generator=g,
                                                                                 dtype=torch.float64)
    eps = 1e-6

    def loss(xx, WW):
        _, ids, w = oracle.router_forward(xx, WW, k, prec="f64")
        assert torch.equal(ids, ids0)  # no selection change inside the step
        return float((w * dw).sum())

    fd = (loss(x + eps * vx, Wr + eps * vW) - loss(x - eps * vx, Wr - eps * vW)) / (2 * eps)
    an = float((dx * vx).sum() + (dWr * vW).sum())
    assert abs(fd - an) <= 1e-7 * max(1.0, abs(an))


def test_invalid_slots_are_skipped():
    x, Wr = _inputs(T=3, H=8, E=6, seed=41)
    _, ids, _ = oracle.router_forward(x, Wr, 3, prec="f64")
    dw = torch.randn(3, 3, generator=torch.Generator().manual_seed(1), dtype=torch.float64)
    dl_all, _, _ = oracle.router_backward(x, Wr, ids, dw, prec="f64")
    ids2 = ids.clone()
    ids2[1, 2] = -1
    dl, _, _ = oracle.router_backward(x, Wr, ids2, dw, prec="f64")
    assert torch.equal(dl[0], dl_all[0]) and torch.equal(dl[2], dl_all[2])
    # token 1 behaves as a top-2 router on its first two slots
    ids3 = ids[1:2, :2].clone()
    dl3, _, _ = oracle.router_backward(x[1:2], Wr, ids3, dw[1:2, :2], prec="f64")
    assert torch.allclose(dl[1], dl3[0], rtol=0, atol=1e-15)
