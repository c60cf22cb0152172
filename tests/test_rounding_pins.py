"""Pins of where the FP32 oracle rounds to bf16 (CPU, no GPU).

"BF16 with FP32 accumulation" is read as: every tensor-core operand is bf16 and
every accumulation fp32.  The oracle therefore rounds exactly six intermediates to
bf16 -- the shrinks y1 = A1 x and y3 = A3 x, the activation h, the A2 shrink z2,
and the outputs y and dx -- and keeps everything else (the gate and up
pre-activations g and u, each expert's down row o, the routing-weighted sum
before its final rounding, the activation gradient, dw and the adapter
gradients) in fp32.

Each case below is a one- or two-route problem whose inputs are bf16 values
chosen so that exactly the intermediate under test is, or is not, a bf16 value,
and the expected output is derived by hand in the comment next to it from that
reading (silu(z) = z / (1 + e^-z) in fp32: at z = 24, e^-24 = 3.8e-11 is below
half an fp32 ulp of 1, so silu(24) = 24 and silu'(24) = 1 exactly; at z = 16,
1 + e^-16 rounds up to 1 + 2^-23, so silu(16) = 15.9999981).
`test_every_rounding_point_is_pinned` then compiles copies of the oracle with one
rounding point removed, or one added where the reading has none, and requires
that some case fails for every such copy.
"""
import ctypes
import os
import subprocess

import pytest
import torch

import oracle
from synth import Shape

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                          "moe_lora_oracle.c")


def _bf16(v):
    t = torch.tensor(v, dtype=torch.float64)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.double(), t), f"{v} is not a bf16 value"
    return b


def _problem(x, W1, W3, W2, ids, w, *, A1=None, A3=None, B1=None, B3=None, A2=None, B2=None, r=1, dy=None):
    """Inputs for T tokens, one adapter; every tensor given as nested lists."""
    T, H = len(x), len(x[0])
    E, I = len(W1), len(W1[0])
    k = len(ids[0])
    z = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)  # noqa: E731
    inp = {
        "x": _bf16(x), "W1": _bf16(W1), "W3": _bf16(W3), "W2": _bf16(W2),
        "A1": _bf16(A1) if A1 is not None else z(1, r, H), "A3": _bf16(A3) if A3 is not None else z(1, r, H),
        "B1": _bf16(B1) if B1 is not None else z(1, E, I, r), "B3": _bf16(B3) if B3 is not None else z(1, E, I, r),
        "A2": _bf16(A2) if A2 is not None else z(1, E, r, I), "B2": _bf16(B2) if B2 is not None else z(1, H, r),
        "dy": _bf16(dy) if dy is not None else z(T, H),
        "topk_ids": torch.tensor(ids, dtype=torch.int32), "topk_w": torch.tensor(w, dtype=torch.float32),
        "adapter_offsets": torch.tensor([0, T], dtype=torch.int64),
    }
    return inp, Shape(T=T, H=H, I=I, E=E, k=k, r=r)


def _y(inp, shp):
    return oracle.forward(inp, shp).double()


# ----------------------------------------------------------------------------- cases
def case_y1_rounded():
    """y1 = rb(A1 x).  x = [1, 1]; A1 = [1, 2^-9] gives A1 x = 1 + 2^-9, which rounds to
    1 (an eighth of the bf16 step at 1), the same y1 as A1 = [1, 0].  B1 = -40 and
    W1 = 0 make g = -40 y1 = -40 in both, u = W3 x = 1, so both problems give the
    same y bit for bit.  Unrounded, g would be -40.078, where silu changes by ~7%."""
    common = dict(x=[[1, 1]], W1=[[[0, 0]]], W3=[[[1, 0]]], W2=[[[1], [0]]], ids=[[0]], w=[[1.0]],
                  B1=[[[[-40]]]])
    ya = _y(*_problem(A1=[[[1, 2 ** -9]]], **common))
    yb = _y(*_problem(A1=[[[1, 0]]], **common))
    assert ya[0, 1] == 0 and ya[0, 0] < 0
    return torch.equal(ya, yb)


def case_y3_rounded():
    """y3 = rb(A3 x).  x = [1, 1]; W1 = [24, 0] gives g = 24, silu(24) = 24.
    W3 = [1024, 1] gives W3 x = 1025 and B3 = -1024; A3 = [1, 2^-9] gives
    A3 x = 1 + 2^-9 -> y3 = 1, so u = 1025 - 1024 = 1, h = 24 and y = [24, 0]
    (W2 = [[1], [0]]).  Unrounded, u = 1025 - 1026 = -1 and y = [-24, 0]."""
    y = _y(*_problem(x=[[1, 1]], W1=[[[24, 0]]], W3=[[[1024, 1]]], W2=[[[1], [0]]], ids=[[0]], w=[[1.0]],
                     A3=[[[1, 2 ** -9]]], B3=[[[[-1024]]]]))
    return torch.equal(y, torch.tensor([[24.0, 0.0]], dtype=torch.float64))


def case_h_rounded():
    """h = rb(silu(g) u).  x = [1, 1]; both rows of W1 are [16, 0] (g = 16,
    silu = 15.9999981); W3 rows [1, 0] and [1, 2^-10] give u = [1, 1 + 2^-10].  Then
    silu(g) u = [15.9999981, 16.0156231], both of which round to 16 (the bf16 step
    at 16 is 1/8), and W2 = [[1, -1], [0, 0]] makes o = [0, 0] and y = [0, 0].
    Unrounded, o[0] = -0.015625."""
    y = _y(*_problem(x=[[1, 1]], W1=[[[16, 0], [16, 0]]], W3=[[[1, 0], [1, 2 ** -10]]],
                     W2=[[[1, -1], [0, 0]]], ids=[[0]], w=[[1.0]]))
    return torch.equal(y, torch.zeros(1, 2, dtype=torch.float64))


def case_u_not_rounded():
    """u stays fp32.  x = [1, 1]; W1 = [24, 0] (g = 24, silu = 24); W3 = [1, 3 * 2^-10]
    gives u = 1.0029296875, which is not a bf16 value (rounded, it would be 1).
    h = rb(24 * 1.0029296875) = rb(24.0703125) = 24.125 (past the midpoint 24.0625),
    so y = [24.125, 0].  With u rounded, h = 24."""
    y = _y(*_problem(x=[[1, 1]], W1=[[[24, 0]]], W3=[[[1, 3 * 2 ** -10]]], W2=[[[1], [0]]], ids=[[0]],
                     w=[[1.0]]))
    return torch.equal(y, torch.tensor([[24.125, 0.0]], dtype=torch.float64))


def case_g_not_rounded():
    """g stays fp32.  x = [1, 1]; W1 rows [-40, -2^-4] and [-40, 0] give
    g = [-40.0625, -40] (the first is not a bf16 value: the step at 40 is 1/4);
    u = [1, 1].  silu(-40.0625) = -1.60e-16 and silu(-40) = -1.70e-16 differ by 6%,
    far more than a bf16 step, so with W2 = [[1, -1], [0, 0]] y[0] is about
    +9.8e-18.  With g rounded, both gates are -40 and y = [0, 0]."""
    y = _y(*_problem(x=[[1, 1]], W1=[[[-40, -2 ** -4], [-40, 0]]], W3=[[[1, 0], [1, 0]]],
                     W2=[[[1, -1], [0, 0]]], ids=[[0]], w=[[1.0]]))
    return y[0, 1] == 0 and 5e-18 < y[0, 0].item() < 1.5e-17


def case_z2_rounded():
    """z2 = rb(A2 h).  x = [1, 1]; W1 rows [16, 0] (silu = 15.9999981), W3 rows [1, 0]:
    h = [16, 16].  A2 rows [1, 0] and [1, 2^-10] give A2 h = [16, 16.015625]; both
    round to 16.  B2 = [[1, -1], [0, 0]] and W2 = 0 make o = s B2 z2 = [0, 0], y = 0.
    Unrounded, o[0] = -0.015625."""
    y = _y(*_problem(x=[[1, 1]], W1=[[[16, 0], [16, 0]]], W3=[[[1, 0], [1, 0]]], W2=[[[0, 0], [0, 0]]],
                     ids=[[0]], w=[[1.0]], A2=[[[[1, 0], [1, 2 ** -10]]]], B2=[[[1, -1], [0, 0]]], r=2))
    return torch.equal(y, torch.zeros(1, 2, dtype=torch.float64))


def case_combine():
    """o stays fp32 and y = rb(sum_j w_j o_j).  One token, two routes (experts 0, 1),
    w = [0.5, 0.5]; H = 1, I = 2; W1 rows [16], W3 rows [1/16]: h = rb(15.9999981/16)
    = [1, 1].  W2_0 = [1, 2^-9] gives o_0 = 1 + 2^-9 (not a bf16 value), W2_1 =
    [3 * 2^-10, 0] gives o_1 = 3 * 2^-10.  The sum is 0.5 + 0.625 * 2^-8, 5/8 of the
    bf16 step above 0.5, so y = 0.5 + 2^-8 = 0.50390625.  With o rounded (o_0 = 1)
    the sum is 0.5 + 0.375 * 2^-8 and y = 0.5; without the final rounding
    y = 0.50244140625."""
    y = _y(*_problem(x=[[1]], W1=[[[16], [16]], [[16], [16]]], W3=[[[0.0625], [0.0625]], [[0.0625], [0.0625]]],
                     W2=[[[1, 2 ** -9]], [[3 * 2 ** -10, 0]]], ids=[[0, 1]], w=[[0.5, 0.5]]))
    return torch.equal(y, torch.tensor([[0.50390625]], dtype=torch.float64))


def case_backward():
    """dx = rb(...); the activation gradient, o and dw stay fp32.  One route, H = I = 1:
    x = 1, W1 = 24 (g = 24: silu = 24, silu' = 1), W3 = 1 (u = 1, h = 24),
    W2 = 1 - 2^-8, dy = 1 + 2^-7, w = 1, no adapters.
      o  = 24 (1 - 2^-8) = 23.90625 (fp32; y = rb(o) = 23.875)
      dw = <dy, o> = 1.0078125 * 23.90625 = 24.093017578125
      dA = w W2 dy = 0.99609375 * 1.0078125 = 1.003875732421875 (rounded: 1)
      dG = dA u silu'(g) = dA,  dU = dA silu(g) = 24 dA
      dx = rb(W1 dG + W3 dU) = rb(48 dA) = rb(48.18603515625) = 48.25
    With dA rounded, dx = 48; with dx unrounded, 48.186; with o rounded (23.875),
    dw = 24.0615234375; with dw rounded, 24.125."""
    inp, shp = _problem(x=[[1]], W1=[[[24]]], W3=[[[1]]], W2=[[[1 - 2 ** -8]]], ids=[[0]], w=[[1.0]],
                        dy=[[1 + 2 ** -7]])
    y = _y(inp, shp)
    g = oracle.backward(inp, shp)
    return (y.item() == 23.875 and g["dx"].double().item() == 48.25
            and g["dw"].double().item() == 24.093017578125)


CASES = [case_y1_rounded, case_y3_rounded, case_h_rounded, case_u_not_rounded, case_g_not_rounded,
         case_z2_rounded, case_combine, case_backward]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.__name__)
def test_rounding_point(case):
    assert case()


# ----------------------------------------------------------------------------- mutations
# (name, text in the oracle source, replacement): one rounding point removed, or one
# added at an intermediate the reading keeps in fp32.
MUTATIONS = [
    ("y1 unrounded", "s->y1[q] = rb(d, acc1);", "s->y1[q] = acc1;"),
    ("y3 unrounded", "s->y3[q] = rb(d, acc3);", "s->y3[q] = acc3;"),
    ("h unrounded", "s->h[i] = rb(d, act_f(d, clampv(d, s->g[i])) * clampv(d, s->u[i]));",
     "s->h[i] = act_f(d, clampv(d, s->g[i])) * clampv(d, s->u[i]);"),
    ("z2 unrounded", "s->z2[q] = rb(d, acc);", "s->z2[q] = acc;"),
    ("y unrounded", "y[n * H + c] = rb(d, acc[c]);", "y[n * H + c] = acc[c];"),
    ("dx unrounded", "dx[n * H + c] = rb(d, dxa[c]);", "dx[n * H + c] = dxa[c];"),
    ("g rounded", "s->g[i] = gb + sc * gl;", "s->g[i] = rb(d, gb + sc * gl);"),
    ("u rounded", "s->u[i] = ub + sc * ul;", "s->u[i] = rb(d, ub + sc * ul);"),
    ("o rounded", "s->o[c] = ob + sc * ol;", "s->o[c] = rb(d, ob + sc * ol);"),
    ("dA rounded", "for (int64_t i = 0; i < I; ++i) dact[i] *= wj;",
     "for (int64_t i = 0; i < I; ++i) dact[i] = rb(d, dact[i] * wj);"),
    ("dw rounded", "dw[n * k + j] = dwj;", "dw[n * k + j] = rb(d, dwj);"),
]


def _build_mutant(tmp_path, old, new):
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, old
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "mutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(so), str(path),
                    "-lm"], check=True)
    L = ctypes.CDLL(str(so))
    L.oracle_forward.restype = ctypes.c_int
    L.oracle_backward.restype = ctypes.c_int
    return L


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_every_rounding_point_is_pinned(tmp_path, monkeypatch, name, old, new):
    """An oracle with this one rounding point moved fails at least one case."""
    oracle.lib("f32")
    monkeypatch.setitem(oracle._LIBS, "f32", _build_mutant(tmp_path, old, new))
    failed = [c.__name__ for c in CASES if not _safe(c)]
    assert failed, f"no case detects: {name}"


def _safe(case):
    try:
        return case()
    except AssertionError:
        return False
