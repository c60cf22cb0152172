"""Pins for the CPU oracle, independent of the oracle itself (CPU only).

Each test ties the oracle to something it does not compute itself:
  * the dense special case: side-LoRA is a low-rank update of the frozen weight,
    so with rounding off every route equals a dense SwiGLU FFN with merged weights
    W1+sB1A1, W3+sB3A3, W2+sB2A2; torch float64 (matmul + autograd) gives the
    forward and every gradient the oracle returns;
  * central finite differences of the oracle's own forward for its backward;
  * the zero-scale identity (the pages: zero adapter scale reproduces the plain MoE
    bitwise, "feat(mega): add fused shared side-LoRA kernels", Correctness coverage);
  * brute-force sorting for the routing plan;
  * the OCP MX decode table for MXFP4 (tests/golden/e2m1_ue8m0.txt);
  * torch's own bf16 conversion for the rounding helper;
  * each adapter of a multi-adapter batch equal to its standalone run (OpenPipe/ART
    PR #1139, Validation: fused and serial runs bitwise equal).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from synth import Shape, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ADAPTER_GRADS = ("dA1", "dA3", "dB1", "dB3", "dA2", "dB2")


def _f64(inp):
    out = {}
    for n, v in inp.items():
        if isinstance(v, torch.Tensor) and v.is_floating_point():
            out[n] = v.double()
        else:
            out[n] = v
    return out


def _tiny(T=5, H=16, I=8, E=3, k=2, r=2, A=1, scale=0.7, seed=0, mask=0.0, act="swiglu", clamp=0.0):
    shp = Shape(T=T, H=H, I=I, E=E, k=k, r=r, A=A, scale=scale, mask_frac=mask, act=act, clamp=clamp)
    inp = _f64(make_inputs(shp, seed=seed))
    # make the side path large enough to matter in the comparisons
    g = torch.Generator().manual_seed(100 + seed)
    for n in ("B1", "B3", "B2"):
        inp[n] = torch.randn(inp[n].shape, generator=g, dtype=torch.float64) * 0.3
    return shp, inp


def _merged_reference(inp, shp, scale):
    """Dense-FFN formulation with merged LoRA weights, float64, torch autograd."""
    T, E, k, A = shp.T, shp.E, shp.k, shp.A
    leaves = {n: inp[n].clone().double().requires_grad_(True)
              for n in ("x", "topk_w", "A1", "A3", "B1", "B3", "A2", "B2")}
    W1, W3, W2 = inp["W1"].double(), inp["W3"].double(), inp["W2"].double()
    ids = inp["topk_ids"].long()
    offs = inp["adapter_offsets"]
    adapter = torch.zeros(T, dtype=torch.long)
    for a in range(A):
        adapter[int(offs[a]):int(offs[a + 1])] = a
    y = torch.zeros(T, shp.H, dtype=torch.float64)
    outs = []
    for t in range(T):
        a = int(adapter[t])
        acc = torch.zeros(shp.H, dtype=torch.float64)
        for j in range(k):
            e = int(ids[t, j])
            if e < 0:
                continue
            W1m = W1[e] + scale * leaves["B1"][a, e] @ leaves["A1"][a]
            W3m = W3[e] + scale * leaves["B3"][a, e] @ leaves["A3"][a]
            W2m = W2[e] + scale * leaves["B2"][a] @ leaves["A2"][a, e]
            xt = leaves["x"][t]
            g, u = W1m @ xt, W3m @ xt
            if shp.clamp > 0:
                g, u = g.clamp(-shp.clamp, shp.clamp), u.clamp(-shp.clamp, shp.clamp)
            act = torch.nn.functional.gelu(g) if shp.act == "geglu" else torch.nn.functional.silu(g)
            h = act * u
            acc = acc + leaves["topk_w"][t, j] * (W2m @ h)
        outs.append(acc)
    y = torch.stack(outs)
    loss = (y * inp["dy"].double()).sum()
    loss.backward()
    return y.detach(), {n: v.grad for n, v in leaves.items()}


def _rel(a, b):
    a, b = a.double(), b.double()
    den = b.norm().item()
    return (a - b).norm().item() / (den if den > 0 else 1.0)


@pytest.mark.parametrize("act,clamp", [("swiglu", 0.0), ("geglu", 0.0), ("swiglu", 0.3), ("geglu", 0.3)])
@pytest.mark.parametrize("scale", [0.7, 0.0])
@pytest.mark.parametrize("A,mask", [(1, 0.0), (1, 0.3), (2, 0.2)])
def test_dense_merged_weight_autograd(scale, A, mask, act, clamp):
    """torch.nn.functional.silu / gelu (exact erf form) and torch.clamp give the
    activation variants; the clamp value 0.3 is small enough to bind on these inputs."""
    shp, inp = _tiny(T=6, A=A, mask=mask, scale=scale, seed=1, act=act, clamp=clamp)
    y_ref, g_ref = _merged_reference(inp, shp, scale)
    y = oracle.forward(inp, shp, prec="f64", scale=scale, round_bf16=False)
    assert _rel(y, y_ref) < 1e-12
    g = oracle.backward(inp, shp, prec="f64", scale=scale, round_bf16=False)
    assert _rel(g["dx"], g_ref["x"]) < 1e-12
    dw_ref = g_ref["topk_w"] * (inp["topk_ids"] >= 0)
    assert _rel(g["dw"], dw_ref) < 1e-12
    for n in ADAPTER_GRADS:
        ref = g_ref[n[1:]]
        if scale == 0.0:
            assert g[n].abs().max().item() == 0.0 and ref.abs().max().item() == 0.0
        else:
            assert _rel(g[n], ref) < 1e-11, n


@pytest.mark.parametrize("act,clamp", [("swiglu", 0.0), ("geglu", 0.3)])
def test_finite_differences(act, clamp):
    """Central differences of the FP64 oracle forward against its backward, for
    every differentiable input (x, routing weights, six adapters)."""
    shp, inp = _tiny(T=4, seed=2, act=act, clamp=clamp)
    g = oracle.backward(inp, shp, prec="f64", round_bf16=False)
    gen = torch.Generator().manual_seed(7)
    names = {"x": "dx", "topk_w": "dw", "A1": "dA1", "A3": "dA3", "B1": "dB1",
             "B3": "dB3", "A2": "dA2", "B2": "dB2"}
    dy = inp["dy"].double()

    def loss(mod):
        return (oracle.forward(mod, shp, prec="f64", round_bf16=False) * dy).sum().item()

    for n, gn in names.items():
        for _ in range(2):
            v = torch.randn(inp[n].shape, generator=gen, dtype=torch.float64)
            if n == "topk_w":
                v = v * (inp["topk_ids"] >= 0)
            eps = 1e-6 * max(1.0, inp[n].abs().max().item())
            lp = loss({**inp, n: inp[n] + eps * v})
            lm = loss({**inp, n: inp[n] - eps * v})
            fd = (lp - lm) / (2 * eps)
            an = (g[gn].reshape(v.shape) * v).sum().item()
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (n, fd, an)


@pytest.mark.parametrize("A,mask,act,clamp", [(1, 0.0, "swiglu", 0.0), (2, 0.25, "geglu", 0.3)])
def test_adjoint_in_the_linear_factors(A, mask, act, clamp):
    """The output is linear in the routing weights w, in A2 and in B2 (each enters once,
    after the activation), so for any direction v the change y(theta + v) - y(theta)
    is exactly the Jacobian applied to v, and <dy, y(theta + v) - y(theta)> must equal
    <grad theta, v> -- an adjoint test with no finite-difference step (FP64 oracle,
    rounding off: agreement to ~1e-12 relative).  A sign, index or transposition
    mistake in dw, dA2 or dB2 breaks it."""
    shp, inp = _tiny(T=6, H=16, I=8, E=3, k=2, r=3, A=A, mask=mask, act=act, clamp=clamp, seed=7)
    if A > 1:
        inp["adapter_offsets"] = torch.tensor([0, 3, 6], dtype=torch.int64)
    y0 = oracle.forward(inp, shp, prec="f64", round_bf16=False)
    grads = oracle.backward(inp, shp, prec="f64", round_bf16=False)
    dy = inp["dy"].double()
    g = torch.Generator().manual_seed(11)
    for name, grad_name in (("topk_w", "dw"), ("A2", "dA2"), ("B2", "dB2")):
        v = torch.randn(inp[name].shape, generator=g, dtype=torch.float64)
        moved = dict(inp)
        moved[name] = inp[name].double() + v
        y1 = oracle.forward(moved, shp, prec="f64", round_bf16=False)
        lhs = (dy * (y1 - y0)).sum().item()
        gv = grads[grad_name]
        if name == "topk_w":  # masked slots carry no gradient and move nothing
            v = torch.where(inp["topk_ids"] >= 0, v, torch.zeros_like(v))
        rhs = (gv * v).sum().item()
        assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(lhs)), (name, lhs, rhs)


def test_zero_scale_is_plain_moe_bitwise():
    """s = 0 with random adapters gives bit-for-bit the output of the same layer
    with the side path removed (adapters zero), in the rounded FP32 oracle."""
    shp = Shape(T=24, H=64, I=32, E=4, k=2, r=8, scale=0.0)
    inp = make_inputs(shp, seed=3)
    y0 = oracle.forward(inp, shp, scale=0.0)
    bare = dict(inp)
    for n in ("A1", "A3", "B1", "B3", "A2", "B2"):
        bare[n] = torch.zeros_like(inp[n])
    y_plain = oracle.forward(bare, shp, scale=1.0)
    assert torch.equal(y0, y_plain)
    g0 = oracle.backward(inp, shp, scale=0.0)
    gp = oracle.backward(bare, shp, scale=1.0)
    assert torch.equal(g0["dx"], gp["dx"])
    assert torch.equal(g0["dw"], gp["dw"])


def test_rounding_points_active_and_small():
    shp = Shape(T=16, H=64, I=32, E=4, k=2, r=8)
    inp = make_inputs(shp, seed=4)
    y32 = oracle.forward(inp, shp)
    y64 = oracle.forward(_f64(inp), shp, prec="f64", round_bf16=False)
    assert torch.equal(y32, y32.to(torch.bfloat16).float())   # outputs are bf16 values
    assert 0 < _rel(y32, y64) < 1e-2


def test_round_bf16_matches_torch():
    g = torch.Generator().manual_seed(5)
    v = torch.randn(20000, generator=g, dtype=torch.float32) * torch.exp2(torch.randint(-20, 20, (20000,)).float())
    ref = v.to(torch.bfloat16).float()
    got = torch.tensor([oracle.round_bf16(float(a)) for a in v.tolist()], dtype=torch.float32)
    assert torch.equal(got, ref)
    assert oracle.round_bf16(1 + 2 ** -8) == 1.0                 # tie -> even
    assert oracle.round_bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6     # tie -> even


def test_mxfp4_decode_table():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_ue8m0.txt")) if l.strip() and l[0] != "#"]
    for kind, code, val in rows:
        got = oracle.e2m1_value(int(code)) if kind == "e2m1" else oracle.ue8m0_value(int(code))
        want = float(val)
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (kind, code)


def _golden_dequant(packed, scales):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_ue8m0.txt")) if l.strip() and l[0] != "#"]
    table = torch.tensor([float(v) for kd, c, v in rows if kd == "e2m1"], dtype=torch.float64)
    lo = (packed & 15).long()
    hi = (packed >> 4).long()
    codes = torch.stack([lo, hi], dim=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    vals = table[codes]
    sc = torch.exp2(scales.double() - 127).repeat_interleave(32, dim=-1)
    return (vals * sc)


def test_mxfp4_base_equals_dequantized_bf16_base():
    shp = Shape(T=12, H=64, I=64, E=3, k=2, r=8, base_fmt="mxfp4")
    inp = make_inputs(shp, seed=6)
    deq = dict(inp)
    for n in ("W1", "W3", "W2"):
        w = _golden_dequant(inp[n], inp["S" + n[1]])
        assert torch.equal(w.to(torch.bfloat16).double(), w)   # exactly representable in bf16
        deq[n] = w.to(torch.bfloat16)
        del deq["S" + n[1]]
    y_q = oracle.forward(inp, shp)
    y_d = oracle.forward(deq, shp)
    assert torch.equal(y_q, y_d)
    g_q = oracle.backward(inp, shp)
    g_d = oracle.backward(deq, shp)
    for n in g_q:
        assert torch.equal(g_q[n], g_d[n]), n


def _plan_bruteforce(ids, E, offs, BM):
    T, k = ids.shape
    A = len(offs) - 1
    adapter = np.zeros(T, dtype=np.int64)
    for a in range(A):
        adapter[offs[a]:offs[a + 1]] = a
    keys = []
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            if 0 <= e < E:
                keys.append((e * A + adapter[t], t, j))  # (expert, adapter, token, slot)
    keys.sort()
    counts = np.zeros(A * E, dtype=np.int64)
    for g, _, _ in keys:
        counts[g] += 1
    padded = -(-counts // BM) * BM
    offsets = np.concatenate([[0], np.cumsum(padded)])
    row_of_route = -np.ones(T * k, dtype=np.int64)
    route_of_row = -np.ones(offsets[-1], dtype=np.int64)
    seen = np.zeros(A * E, dtype=np.int64)
    for g, t, j in keys:
        row = offsets[g] + seen[g]
        seen[g] += 1
        row_of_route[t * k + j] = row
        route_of_row[row] = t * k + j
    return counts, offsets, row_of_route, route_of_row


@pytest.mark.parametrize("T,k,E,A,BM,seed", [(37, 3, 5, 1, 8, 0), (200, 6, 16, 1, 16, 1),
                                           (64, 2, 4, 4, 8, 2), (1, 1, 3, 1, 128, 3)])
def test_plan_bruteforce(T, k, E, A, BM, seed):
    g = torch.Generator().manual_seed(seed)
    ids = torch.randint(-1, E, (T, k), generator=g, dtype=torch.int32)
    ids[ids == 1] = -1 if E > 2 else 0
    offs = torch.linspace(0, T, A + 1).round().long()
    got = oracle.plan(ids, E, offs, BM)
    c, o, ror, rrow = _plan_bruteforce(ids.numpy(), E, offs.tolist(), BM)
    assert np.array_equal(got["counts"].numpy(), c)
    assert np.array_equal(got["offsets"].numpy(), o)
    assert np.array_equal(got["row_of_route"].numpy(), ror)
    assert np.array_equal(got["route_of_row"].numpy(), rrow)
    assert got["bad"] == 0
    # invariants
    assert (np.diff(o) % BM == 0).all() and (np.diff(o) >= 0).all()
    assert int(c.sum()) == int((ids >= 0).sum())


def test_plan_drops_invalid_ids():
    ids = torch.tensor([[0, 5], [-2, 1], [2, -1]], dtype=torch.int32)
    got = oracle.plan(ids, 3, torch.tensor([0, 3]), 4)
    assert got["bad"] == 2
    assert got["row_of_route"].tolist() == [0, -1, -1, 4, 8, -1]


def test_multi_adapter_equals_standalone():
    """Each adapter's outputs and gradients in a shared pass equal its standalone
    single-adapter run bit for bit (rounded FP32 oracle)."""
    A, per = 3, 10
    shp = Shape(T=A * per, H=64, I=32, E=4, k=2, r=8, A=A)
    inp = make_inputs(shp, seed=8)
    y = oracle.forward(inp, shp)
    g = oracle.backward(inp, shp)
    for a in range(A):
        sl = slice(a * per, (a + 1) * per)
        one = Shape(T=per, H=64, I=32, E=4, k=2, r=8, A=1)
        sub = {n: inp[n][sl] for n in ("x", "dy", "topk_ids", "topk_w")}
        for n in ("W1", "W3", "W2"):
            sub[n] = inp[n]
        for n in ("A1", "A3", "B1", "B3", "A2", "B2"):
            sub[n] = inp[n][a:a + 1]
        sub["adapter_offsets"] = torch.tensor([0, per])
        ys = oracle.forward(sub, one)
        gs = oracle.backward(sub, one)
        assert torch.equal(y[sl], ys)
        assert torch.equal(g["dx"][sl], gs["dx"])
        assert torch.equal(g["dw"][sl], gs["dw"])
        for n in ADAPTER_GRADS:
            assert torch.equal(g[n][a:a + 1], gs[n]), (a, n)


def test_masked_token_and_empty_expert():
    shp = Shape(T=8, H=64, I=32, E=4, k=2, r=8)
    inp = make_inputs(shp, seed=9)
    inp["topk_ids"][3] = -1                 # token 3 fully masked
    inp["topk_w"][3] = 0
    inp["topk_ids"][inp["topk_ids"] == 2] = 1   # expert 2 empty
    y = oracle.forward(inp, shp)
    g = oracle.backward(inp, shp)
    assert y[3].abs().max() == 0 and g["dx"][3].abs().max() == 0 and g["dw"][3].abs().max() == 0
    for n in ("dB1", "dB3", "dA2"):
        assert g[n][0, 2].abs().max() == 0
    assert g["dB1"][0, 1].abs().max() > 0
