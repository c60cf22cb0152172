"""GPU parity of the routing step (softmax top-k router and its backward) against
the oracle's router.

The pages take the routes as inputs and return their weight gradient
("grad-route", fw-ai/DeepGEMM PR #9, Correctness coverage); the router read here is
softmax over all experts, top-k (ties to the lower id), weights renormalised to 1.
Bars: expert ids equal to the oracle's except where the oracle's own logits tie to
within fp32 accumulation noise (then the choice must still be a valid top-k);
logits and weights to fp32 accuracy; dlogits, dW_r and grad-x within relative L2
5e-3 and cosine 0.9999 (the path's BF16 gate; dlogits is rounded to bf16 as the
tensor-core operand of both backward contractions).
"""
import pytest
import torch

import moe_expert_ffn_top_gb300 as m
import oracle
from synth import make_router_inputs

from gpu_common import assert_close, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_ffn_top_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield


def _dims(T, H, E, k):
    return m.make_dims(T, H, 256, E, k, 16)


def _gpu_forward(inp, T, H, E, k, logits=True):
    d = _dims(T, H, E, k)
    sc = m.router_scratch(d)
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), device="cuda")
    lg = torch.full((T, E), float("nan"), device="cuda") if logits else None
    m.moe_lora_router_forward(d, inp["x"], inp["Wr"], ids, w, lg, sc)
    torch.cuda.synchronize()
    assert m.moe_lora_router_get_error(sc) == 0
    return d, sc, ids, w, lg


def _check_selection(ids_g, w_g, l_g, l_ref, ids_ref, w_ref, tie_tol):
    """ids equal to the oracle's, except on near-ties of the oracle's logits, where
    the GPU's choice must be a valid top-k in the oracle's order (within tie_tol).
    Weights of agreeing tokens: w_j is the softmax of the selected logits, so
    |dw_j| <= 2 max_e |dl_e| w_j for logit differences dl (fp32 accumulation order),
    plus fp32 rounding of the exponentials and sums."""
    T, k = ids_ref.shape
    same = (ids_g.cpu() == ids_ref).all(dim=1)
    for t in torch.nonzero(~same).flatten().tolist():
        g, r = ids_g[t].cpu().long(), ids_ref[t].long()
        assert len(set(g.tolist())) == k and int(g.min()) >= 0
        for j in range(k):  # slot by slot, the logits agree to within the tie tolerance
            assert abs(float(l_ref[t, g[j]] - l_ref[t, r[j]])) <= tie_tol, (t, g.tolist(), r.tolist())
    assert int((~same).sum()) <= max(2, T // 200), int((~same).sum())
    if same.any():
        dlog = (l_g.cpu().double() - l_ref.double()).abs().max(dim=1).values[same].unsqueeze(1)
        wr = w_ref[same].double()
        err = (w_g.cpu()[same].double() - wr).abs()
        assert (err <= 2 * dlog * wr + 1e-6 * wr + 1e-7).all(), float((err / (2 * dlog * wr + 1e-6 * wr + 1e-7)).max())
    return same


@pytest.mark.parametrize("T,H,E,k", [(300, 512, 16, 2), (1000, 1024, 128, 8), (517, 4096, 256, 6),
                                     (4096, 4096, 256, 6), (129, 256, 32, 32), (200, 576, 64, 4)])
def test_router_forward_matches_oracle(T, H, E, k):
    inp = make_router_inputs(T, H, E, k, seed=T + E, device="cuda")
    _, _, ids, w, lg = _gpu_forward(inp, T, H, E, k)
    l_ref, ids_ref, w_ref = oracle.router_forward(inp["x"].cpu(), inp["Wr"].cpu(), k, prec="f32")
    assert rel_l2(lg, l_ref) <= 1e-5
    tie_tol = 1e-5 * float(l_ref.abs().max()) + 1e-6
    _check_selection(ids, w, lg, l_ref, ids_ref, w_ref, tie_tol)
    assert torch.allclose(w.sum(1).cpu(), torch.ones(T), atol=1e-6)


def test_router_ties_go_to_the_lower_id():
    T, H, E, k = 130, 256, 32, 5
    inp = make_router_inputs(T, H, E, k, seed=3, device="cuda")
    Wr = inp["Wr"].clone()
    big = Wr[3] * 4  # exact in bf16
    for e in (3, 17, 30):  # three equal, large rows: equal logits on both sides
        Wr[e] = big
    inp["Wr"] = Wr
    _, _, ids, w, lg = _gpu_forward(inp, T, H, E, k)
    l_ref, ids_ref, w_ref = oracle.router_forward(inp["x"].cpu(), Wr.cpu(), k, prec="f32")
    lgc = lg.cpu()
    assert torch.equal(lgc[:, 3], lgc[:, 17]) and torch.equal(lgc[:, 3], lgc[:, 30])
    seen = 0
    for t in range(T):
        row = ids[t].tolist()
        for a, b in ((3, 17), (17, 30)):  # a tied pair is taken lower id first, back to back
            if a in row and row.index(a) < k - 1:
                assert row[row.index(a) + 1] == b, row
                seen += 1
    assert seen > T // 4
    _check_selection(ids, w, lg, l_ref, ids_ref, w_ref, 1e-5 * float(l_ref.abs().max()) + 1e-6)


@pytest.mark.parametrize("T,H,E,k", [(300, 512, 16, 2), (1000, 1024, 128, 8), (4096, 4096, 256, 6),
                                     (200, 576, 64, 4), (150, 64, 16, 2)])
def test_router_backward_matches_oracle(T, H, E, k):
    inp = make_router_inputs(T, H, E, k, seed=11 * T + E, device="cuda")
    d, sc, ids, w, _ = _gpu_forward(inp, T, H, E, k, logits=False)
    dl = torch.full((T, E), float("nan"), device="cuda")
    dWr = torch.full((E, H), float("nan"), device="cuda")
    dx = inp["dx0"].clone()
    m.moe_lora_router_backward(d, inp["x"], inp["Wr"], ids, w, inp["dw"], dl, dWr, dx, sc)
    torch.cuda.synchronize()
    assert m.moe_lora_router_get_error(sc) == 0
    # the oracle differentiates its own forward for the GPU's selection
    dl_ref, dWr_ref, dx_ref = oracle.router_backward(inp["x"].cpu(), inp["Wr"].cpu(), ids.cpu(),
                                                     inp["dw"].cpu(), prec="f32")
    assert rel_l2(dl, dl_ref) <= 1e-4
    assert_close("dWr", dWr, dWr_ref)
    want = inp["dx0"].cpu().double() + dx_ref.double()
    assert_close("dx (accumulated)", dx, want)
    # the router's part alone
    dx2 = torch.zeros_like(dx)
    m.moe_lora_router_backward(d, inp["x"], inp["Wr"], ids, w, inp["dw"], None, dWr, dx2, sc)
    torch.cuda.synchronize()
    assert_close("dx (router part)", dx2, dx_ref)


def test_router_production_size_sampled():
    """65,536 tokens, H4096, E256, top-6: every token's selection and weights from the
    GPU; the oracle checks 192 sampled tokens' logits, ids, weights, dlogits and grad-x
    rows; dW_r is checked as dl^T x (fp64) for the bf16 dlogits the kernels used
    (the oracle's dW_r is compared at 4,096 tokens in the backward test)."""
    T, H, E, k = 65536, 4096, 256, 6
    inp = make_router_inputs(T, H, E, k, seed=2026, device="cuda")
    d, sc, ids, w, lg = _gpu_forward(inp, T, H, E, k)
    dl = torch.empty(T, E, device="cuda")
    dWr = torch.empty(E, H, device="cuda")
    dx = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    m.moe_lora_router_backward(d, inp["x"], inp["Wr"], ids, w, inp["dw"], dl, dWr, dx, sc)
    torch.cuda.synchronize()
    assert m.moe_lora_router_get_error(sc) == 0
    # every token: distinct ids, weights descending and summing to 1
    assert (ids >= 0).all() and (ids < E).all()
    srt = torch.sort(ids.long(), dim=1).values
    assert (srt[:, 1:] != srt[:, :-1]).all()
    assert (w[:, :-1] >= w[:, 1:]).all()
    assert (w.sum(1) - 1).abs().max().item() <= 1e-6
    g = torch.Generator().manual_seed(5)
    tok = torch.cat([torch.tensor([0, 1, T - 1]), torch.randperm(T - 2, generator=g)[:189] + 1])
    xs = inp["x"][tok.cuda()].cpu()
    l_ref, ids_ref, w_ref = oracle.router_forward(xs, inp["Wr"].cpu(), k, prec="f32")
    assert rel_l2(lg[tok.cuda()], l_ref) <= 1e-5
    _check_selection(ids[tok.cuda()], w[tok.cuda()], lg[tok.cuda()], l_ref, ids_ref, w_ref,
                     1e-5 * float(l_ref.abs().max()) + 1e-6)
    ids_s = ids[tok.cuda()].cpu()
    dl_ref, _, dx_ref = oracle.router_backward(xs, inp["Wr"].cpu(), ids_s, inp["dw"][tok.cuda()].cpu(),
                                               prec="f32")
    assert rel_l2(dl[tok.cuda()], dl_ref) <= 1e-4
    assert_close("dx rows", dx[tok.cuda()], dx_ref)
    # dW_r = dl^T x for the dl the kernels used (bf16 operand), fp64 on the host
    ref = dl.to(torch.bfloat16).double().t() @ inp["x"].double()
    assert_close("dWr", dWr, ref)


def test_router_empty_batch():
    d = _dims(0, 512, 16, 2)
    sc = m.router_scratch(d)
    e = torch.empty(0, device="cuda")
    ids = torch.empty(0, 2, dtype=torch.int32, device="cuda")
    w = torch.empty(0, 2, device="cuda")
    Wr = torch.randn(16, 512, device="cuda").to(torch.bfloat16)
    x = torch.empty(0, 512, dtype=torch.bfloat16, device="cuda")
    m.moe_lora_router_forward(d, x, Wr, ids, w, None, sc)
    dWr = torch.full((16, 512), float("nan"), device="cuda")
    dx = torch.empty(0, 512, dtype=torch.bfloat16, device="cuda")
    m.moe_lora_router_backward(d, x, Wr, ids, w, e.view(0, 2), None, dWr, dx, sc)
    torch.cuda.synchronize()
    assert m.moe_lora_router_get_error(sc) == 0
    assert (dWr == 0).all()


def test_router_deterministic():
    T, H, E, k = 40000, 1024, 64, 4
    inp = make_router_inputs(T, H, E, k, seed=9, device="cuda")
    outs = []
    for _ in range(2):
        d, sc, ids, w, lg = _gpu_forward(inp, T, H, E, k)
        dWr = torch.empty(E, H, device="cuda")
        dx = inp["dx0"].clone()
        m.moe_lora_router_backward(d, inp["x"], inp["Wr"], ids, w, inp["dw"], None, dWr, dx, sc)
        torch.cuda.synchronize()
        outs.append((ids.cpu(), w.cpu(), lg.cpu(), dWr.cpu(), dx.cpu()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def _run_router(inp, T, H, E, k, A, offs, x, Wr, dw, dx0):
    d = m.make_dims(T, H, 256, E, k, 16, A)
    sc = m.router_scratch(d)
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), device="cuda")
    lg = torch.full((T, E), float("nan"), device="cuda")
    m.moe_lora_router_forward(d, x, Wr, ids, w, lg, sc, adapter_offsets=offs)
    dl = torch.full((T, E), float("nan"), device="cuda")
    dWr = torch.full((A, E, H), float("nan"), device="cuda")
    dx = dx0.clone()
    m.moe_lora_router_backward(d, x, Wr, ids, w, dw, dl, dWr, dx, sc, adapter_offsets=offs)
    torch.cuda.synchronize()
    assert m.moe_lora_router_get_error(sc) == 0
    return ids, w, lg, dl, dWr, dx


@pytest.mark.parametrize("H,E,k,offs", [
    (2048, 128, 8, [1024 * a for a in range(17)]),       # 16 adapters x 1,024 tokens (the multi-adapter pass)
    (1024, 64, 4, [0, 256, 256, 896, 1000]),             # an empty adapter and a ragged last one
    (1024, 64, 4, [0, 32768, 40000]),                    # adapter 0's dW_r is split over token slices
])
def test_router_multi_adapter_equals_standalone(H, E, k, offs):
    """One router per adapter (OpenPipe/ART PR #1139, Behavior): the fused pass over
    all adapters equals every adapter's standalone run bit for bit, and matches the
    oracle's router with that adapter's W_r."""
    A, T = len(offs) - 1, offs[-1]
    inp = make_router_inputs(T, H, E, k, seed=31 + A, device="cuda", A=A)
    ids, w, lg, dl, dWr, dx = _run_router(inp, T, H, E, k, A, offs, inp["x"], inp["Wr"], inp["dw"], inp["dx0"])
    for a in range(A):
        t0, t1 = offs[a], offs[a + 1]
        if t1 == t0:
            assert (dWr[a] == 0).all(), a
            continue
        s_ids, s_w, s_lg, s_dl, s_dWr, s_dx = _run_router(
            inp, t1 - t0, H, E, k, 1, None, inp["x"][t0:t1].contiguous(), inp["Wr"][a].contiguous(),
            inp["dw"][t0:t1].contiguous(), inp["dx0"][t0:t1].contiguous())
        for name, fused, alone in (("ids", ids[t0:t1], s_ids), ("w", w[t0:t1], s_w), ("logits", lg[t0:t1], s_lg),
                                   ("dlogits", dl[t0:t1], s_dl), ("dWr", dWr[a], s_dWr[0]),
                                   ("dx", dx[t0:t1], s_dx)):
            assert torch.equal(fused, alone), (a, name)
    for a in (0, A - 1):  # the oracle, with each adapter's own router weights
        t0, t1 = offs[a], min(offs[a + 1], offs[a] + 512)
        if t1 == t0:
            continue
        xs = inp["x"][t0:t1].cpu()
        l_ref, ids_ref, w_ref = oracle.router_forward(xs, inp["Wr"][a].cpu(), k, prec="f32")
        assert rel_l2(lg[t0:t1], l_ref) <= 1e-5
        _check_selection(ids[t0:t1], w[t0:t1], lg[t0:t1], l_ref, ids_ref, w_ref,
                         1e-5 * float(l_ref.abs().max()) + 1e-6)
        dl_ref, _, dx_ref = oracle.router_backward(xs, inp["Wr"][a].cpu(), ids[t0:t1].cpu(), inp["dw"][t0:t1].cpu(),
                                                   prec="f32")
        assert rel_l2(dl[t0:t1], dl_ref) <= 1e-4
        assert_close("dx rows", dx[t0:t1], inp["dx0"][t0:t1].cpu().double() + dx_ref.double())
    # dW_r[a] = dl^T x over adapter a's tokens, for the bf16 dlogits the kernels used
    for a in range(A):
        t0, t1 = offs[a], offs[a + 1]
        if t1 > t0:
            ref = dl[t0:t1].to(torch.bfloat16).double().t() @ inp["x"][t0:t1].double()
            assert_close(f"dWr[{a}]", dWr[a], ref)
