"""Pins for the oracle's native FP4 forward (CPU only).

In that forward the gate/up base products take the token's activations as MXFP8:
E4M3 elements with one shared power-of-two scale per 32 values, the OCP MX format
("FP8/FP4/FP8 forwards", "feat(mega): add fused shared side-LoRA kernels", Fresh
validation).  Each test ties the oracle to something it does not compute itself:
  * the OCP OFP8 E4M3 table (tests/golden/e4m3.txt) and the grid's structure;
  * rounding to E4M3 against brute force over the whole grid (nearest value, ties
    to the even code, saturation at 448);
  * the shared-scale rule: every block's max|v| / 2^X falls in [256, 512);
  * the identity on inputs that are already MXFP8 values, with a zero down-projection
    base (so q8 of the activation has nothing to act on): native == plain bitwise;
  * the dense special case in torch float64: base products on q8(x) and q8(h) with
    straight-through gradients, side paths on x and h, for the forward and every
    gradient the oracle returns.
"""
import math
import os

import pytest
import torch

import oracle
from synth import Shape, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ADAPTER_GRADS = ("dA1", "dA3", "dB1", "dB3", "dA2", "dB2")


def _grid():
    """Positive finite E4M3 values by code 0..126, from the format's definition:
    subnormals m/8 * 2^-6, normals (1 + m/8) * 2^(e-7), e = 1..15, S.1111.111 = NaN."""
    vals = [m / 8 * 2.0 ** -6 for m in range(8)]
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            vals.append((1 + m / 8) * 2.0 ** (e - 7))
    return vals


def test_e4m3_decode_table():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e4m3.txt")) if l.strip() and l[0] != "#"]
    assert len(rows) >= 10
    for code, val in rows:
        got, want = oracle.e4m3_value(int(code)), float(val)
        if math.isnan(want):
            assert math.isnan(got), code
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), code


def test_e4m3_grid_structure():
    grid = _grid()
    assert len(grid) == 127
    for c in range(127):
        assert oracle.e4m3_value(c) == grid[c]
        assert oracle.e4m3_value(c | 0x80) == -grid[c]
    assert all(b > a for a, b in zip(grid, grid[1:]))     # strictly increasing with the code
    assert grid[-1] == 448.0 and grid[1] == 2.0 ** -9


def _nearest_even(v, grid):
    """Brute force: the grid value nearest |v| (ties to the even code), saturated,
    with v's sign."""
    a = abs(v)
    if a >= 448.0:
        r = 448.0
    else:
        best = min(range(len(grid)), key=lambda c: (abs(grid[c] - a), c & 1))
        r = grid[best]
    return -r if math.copysign(1, v) < 0 else r


def test_e4m3_round_bruteforce():
    grid = _grid()
    g = torch.Generator().manual_seed(7)
    vals = []
    for e in range(-12, 10):
        vals += (torch.rand(40, generator=g, dtype=torch.float64) * 2.0 ** e * 2 - 2.0 ** e).tolist()
    mids = [(a + b) / 2 for a, b in zip(grid, grid[1:])]             # every tie
    vals += mids + [-m for m in mids] + grid
    vals += [448.0, 455.9, 464.0, 470.0, 480.0, 512.0, 1e6, -1e6, 2.0 ** -10, 2.0 ** -10 * 1.0001, 0.0, -0.0]
    for v in vals:
        want = _nearest_even(v, grid)
        got = oracle.e4m3_round(v)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), v


def test_mxfp8_shared_scale_rule():
    g = torch.Generator().manual_seed(8)
    grid = _grid()
    for trial in range(200):
        n = 32 if trial % 5 else 1 + trial % 31          # short last blocks too
        mag = 2.0 ** float(torch.randint(-30, 30, (1,), generator=g))
        v = torch.randn(n, generator=g, dtype=torch.float64) * mag
        v = v.to(torch.bfloat16).double()                  # activations are bf16 values
        codes, scales, deq = oracle.mxfp8_quantize(v)
        X = int(scales[0]) - 127
        amax = v.abs().max().item()
        assert 256.0 <= amax / 2.0 ** X < 512.0
        for i in range(n):
            c = int(codes[i])
            val = grid[c & 0x7F] * (-1 if c & 0x80 else 1)
            assert deq[i].item() == val * 2.0 ** X                      # code x scale, exactly
            assert deq[i].item() == _nearest_even(v[i].item() / 2.0 ** X, grid) * 2.0 ** X
    codes, scales, deq = oracle.mxfp8_quantize(torch.zeros(32, dtype=torch.float64))
    assert int(scales[0]) == 127 and int(codes.max()) == 0 and deq.abs().max().item() == 0.0


def _native(shp):
    return Shape(**{**shp.__dict__, "base_fmt": "mxfp4_native"})


def test_native_identity_on_mxfp8_values():
    """x already in MXFP8 (each block's max in [256, 448] x 2^X, all values on the
    grid x 2^X): q8(x) = x; with W2 = 0 the down base product vanishes in both modes,
    so the native forward and backward equal the plain ones bitwise (FP32 oracle,
    rounding on)."""
    shp = Shape(T=6, H=64, I=32, E=3, k=2, r=8, base_fmt="mxfp4")
    inp = make_inputs(shp, seed=9)
    inp["W2"] = torch.zeros_like(inp["W2"])            # E2M1 code 0 under any scale
    grid = torch.tensor(_grid(), dtype=torch.float64)
    g = torch.Generator().manual_seed(10)
    x = torch.zeros(shp.T, shp.H, dtype=torch.float64)
    for t in range(shp.T):
        for b in range(0, shp.H, 32):
            X = int(torch.randint(-12, -6, (1,), generator=g))
            codes = torch.randint(0, 127, (32,), generator=g)
            codes[int(torch.randint(0, 32, (1,), generator=g))] = int(torch.randint(120, 127, (1,), generator=g))
            sign = torch.where(torch.rand(32, generator=g) < 0.5, -1.0, 1.0).double()
            x[t, b:b + 32] = sign * grid[codes] * 2.0 ** X
    assert torch.equal(x.to(torch.bfloat16).double(), x)   # E4M3 values fit bf16
    inp["x"] = x.to(torch.bfloat16)
    _, _, deq = oracle.mxfp8_quantize(inp["x"].double().flatten())
    assert torch.equal(deq.view_as(x), x)
    nat = _native(shp)
    assert torch.equal(oracle.forward(inp, nat), oracle.forward(inp, shp))
    gn, gp = oracle.backward(inp, nat), oracle.backward(inp, shp)
    for n in gp:
        assert torch.equal(gn[n], gp[n]), n


def _dense_native_reference(inp, shp, scale):
    """One expert, one slot, weight w: torch float64 with the base products on q8(x)
    and q8(h) (straight-through: the gradient passes q8 unchanged) and the side
    shrinks A1 x, A3 x and A2 h on x and h themselves."""
    leaves = {n: inp[n].clone().double().requires_grad_(True)
              for n in ("x", "topk_w", "A1", "A3", "B1", "B3", "A2", "B2")}
    W1, W3, W2 = inp["W1"].double()[0], inp["W3"].double()[0], inp["W2"].double()[0]
    x = leaves["x"]
    q = torch.stack([oracle.mxfp8_quantize(x[t].detach())[2] for t in range(shp.T)])
    xq = x + (q - x).detach()
    y1 = x @ leaves["A1"][0].T
    y3 = x @ leaves["A3"][0].T
    g = xq @ W1.T + scale * y1 @ leaves["B1"][0, 0].T
    u = xq @ W3.T + scale * y3 @ leaves["B3"][0, 0].T
    h = torch.nn.functional.silu(g) * u
    hq8 = torch.stack([oracle.mxfp8_quantize(h[t].detach(), prec="f64")[2] for t in range(shp.T)])
    hq = h + (hq8 - h).detach()
    z2 = h @ leaves["A2"][0, 0].T
    o = hq @ W2.T + scale * z2 @ leaves["B2"][0].T
    y = leaves["topk_w"][:, :1] * o
    (y * inp["dy"].double()).sum().backward()
    return y.detach(), {n: v.grad for n, v in leaves.items()}, q


def test_native_dense_autograd():
    # bf16 weights: the native forward changes the activations' format, not the
    # weights' (an MXFP4 base decodes exactly, pinned elsewhere)
    shp = Shape(T=5, H=96, I=32, E=1, k=1, r=4, scale=0.7)
    inp = make_inputs(shp, seed=11)
    inp = {n: (v.double() if isinstance(v, torch.Tensor) and v.is_floating_point() else v) for n, v in inp.items()}
    g = torch.Generator().manual_seed(12)
    for n in ("B1", "B3", "B2"):
        inp[n] = torch.randn(inp[n].shape, generator=g, dtype=torch.float64) * 0.3
    nat = _native(shp)
    y_ref, g_ref, q = _dense_native_reference(inp, shp, 0.7)
    assert (q - inp["x"]).abs().max().item() > 0          # the quantisation does change x
    y = oracle.forward(inp, nat, prec="f64", round_bf16=False)
    assert (y - y_ref).norm().item() <= 1e-12 * y_ref.norm().item()
    y_plain = oracle.forward(inp, shp, prec="f64", round_bf16=False)
    assert (y_plain - y_ref).norm().item() > 1e-6 * y_ref.norm().item()
    gr = oracle.backward(inp, nat, prec="f64", round_bf16=False)
    assert (gr["dx"] - g_ref["x"]).norm().item() <= 1e-12 * g_ref["x"].norm().item()
    assert (gr["dw"] - g_ref["topk_w"]).norm().item() <= 1e-12 * g_ref["topk_w"].norm().item()
    for n in ADAPTER_GRADS:
        ref = g_ref[n[1:]]
        assert (gr[n] - ref).norm().item() <= 1e-11 * ref.norm().item(), n
