"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding, build oracle sub-problems, and the FP64 comparison metrics."""
from __future__ import annotations

from typing import Dict, Iterable, Optional

import torch

import moe_expert_ffn_top_gb300 as m
import oracle
from synth import Shape

ADAPTER_GRADS = ("dA1", "dA3", "dB1", "dB3", "dA2", "dB2")
WEIGHT_NAMES = ("W1", "W3", "W2", "A1", "A3", "B1", "B3", "A2", "B2")

# Tolerances for BF16 outputs and all gradients (FP64 metrics over whole tensors).
REL_L2_MAX = 5e-3
COSINE_MIN = 0.9999


def rel_l2(a: torch.Tensor, b: torch.Tensor) -> float:
    a, b = a.double().cpu(), b.double().cpu()
    den = b.norm().item()
    return (a - b).norm().item() / (den if den > 0 else 1.0)


def cosine(a: torch.Tensor, b: torch.Tensor) -> float:
    a, b = a.double().cpu().flatten(), b.double().cpu().flatten()
    na, nb = a.norm().item(), b.norm().item()
    if na == 0 and nb == 0:
        return 1.0
    if na == 0 or nb == 0:
        return 0.0
    return (a @ b).item() / (na * nb)


def assert_close(name: str, got: torch.Tensor, ref: torch.Tensor) -> None:
    rl, cs = rel_l2(got, ref), cosine(got, ref)
    assert torch.isfinite(got.float()).all(), f"{name}: non-finite values"
    assert rl <= REL_L2_MAX and cs >= COSINE_MIN, f"{name}: relL2={rl:.3e} cosine={cs:.7f}"


def dims_of(shp: Shape, scale: Optional[float] = None, mx_once: bool = False) -> m.Dims:
    """mx_once: an MXFP4 base decoded once per pass (base_fmt 2) instead of inside the GEMMs (1);
    base_fmt "mxfp4_native" is the native FP4 forward with the rest decoded in the GEMMs (3)
    or once per pass (4)."""
    mx = 2 if mx_once else 1
    fmt = {"mxfp4": mx, "mxfp4_native": mx + 2}.get(shp.base_fmt, 0)
    return m.make_dims(shp.T, shp.H, shp.I, shp.E, shp.k, shp.r, shp.A, shp.scale if scale is None else scale,
                       base_fmt=fmt, act=1 if shp.act == "geglu" else 0,
                       act_clamp=shp.clamp)


def run_gpu(inp: Dict[str, torch.Tensor], shp: Shape, scale: Optional[float] = None, poison: bool = False,
            backward: bool = True, ws: Optional[m.Workspaces] = None, mx_once: bool = False) -> Dict[str, torch.Tensor]:
    """Plan + forward (+ backward) on cuda:0 through the C ABI; results on the device."""
    d = dims_of(shp, scale, mx_once)
    if ws is None:
        ws = m.Workspaces.allocate(d)
    if poison:  # 0xFF bytes are bf16/fp32 NaNs: padding or stale rows must never leak
        for b in (ws.saved, ws.fwd, ws.bwd):
            b.fill_(0xFF)
    dev = {n: (v if v.is_cuda else v.cuda()) for n, v in inp.items() if n != "adapter_offsets"}
    offs = inp["adapter_offsets"].tolist() if shp.A > 1 else None
    m.moe_lora_plan(d, dev["topk_ids"], offs, ws.plan)
    y = torch.empty(shp.T, shp.H, dtype=torch.bfloat16, device="cuda")
    if poison:
        y.fill_(float("nan"))
    m.moe_lora_forward(d, ws.plan, dev["x"], dev["topk_w"], dev, y, ws.saved, ws.fwd)
    out = {"y": y, "ws": ws, "dims": d}
    if backward:
        dx = torch.empty_like(y)
        dw = torch.empty(shp.T, shp.k, dtype=torch.float32, device="cuda")
        g = m.alloc_grads(d)
        if poison:
            dx.fill_(float("nan"))
            dw.fill_(float("nan"))
            for t in g.values():
                t.fill_(float("nan"))
        m.moe_lora_backward(d, ws.plan, ws.saved, dev["x"], dev["topk_w"], dev["dy"], dev, dx, dw, g, ws.bwd)
        out.update(dx=dx, dw=dw, **g)
    torch.cuda.synchronize()
    out["err"] = m.moe_lora_get_error(d, ws.plan)
    return out


def sub_problem(inp: Dict[str, torch.Tensor], shp: Shape, tokens: Iterable[int]):
    """The sub-problem made of the listed tokens (single adapter), on the CPU, with
    the experts they touch renumbered 0..E'-1 so the oracle only needs those
    experts' weights.  Returns (inputs, shape, expert list)."""
    assert shp.A == 1
    tok = torch.as_tensor(sorted(set(int(t) for t in tokens)), dtype=torch.long)
    ids = inp["topk_ids"].cpu()[tok]
    used = sorted(set(int(e) for e in ids.flatten().tolist() if e >= 0))
    if not used:
        used = [0]
    remap = {e: i for i, e in enumerate(used)}
    new_ids = ids.clone()
    for (i, j), e in zip([(i, j) for i in range(ids.shape[0]) for j in range(ids.shape[1])], ids.flatten().tolist()):
        new_ids[i, j] = remap[e] if e >= 0 else -1
    ex = torch.as_tensor(used, dtype=torch.long)
    sub = {
        "x": inp["x"][tok.to(inp["x"].device)].cpu(),
        "dy": inp["dy"][tok.to(inp["dy"].device)].cpu(),
        "topk_w": inp["topk_w"][tok.to(inp["topk_w"].device)].cpu(),
        "topk_ids": new_ids.to(torch.int32),
        "adapter_offsets": torch.tensor([0, len(tok)], dtype=torch.int64),
    }
    exd = ex.to(inp["W1"].device)
    for n in ("W1", "W3", "W2", "S1", "S3", "S2"):
        if n in inp:
            sub[n] = inp[n][exd].cpu()
    for n in ("B1", "B3", "A2"):
        sub[n] = inp[n][:, exd].cpu()
    for n in ("A1", "A3", "B2"):
        sub[n] = inp[n].cpu()
    sshp = Shape(T=len(tok), H=shp.H, I=shp.I, E=len(used), k=shp.k, r=shp.r, A=1, scale=shp.scale,
                 base_fmt=shp.base_fmt, act=shp.act, clamp=shp.clamp)
    return sub, sshp, used, tok


def _full_check(inp, shp, out, tokens=None):
    """Compare everything the GPU returned with the oracle (all tokens if None)."""
    y_ref = oracle.forward(inp, shp, tokens=tokens)
    g_ref = oracle.backward(inp, shp, tokens=tokens)
    sel = slice(None) if tokens is None else torch.as_tensor(tokens)
    assert_close("y", out["y"].cpu()[sel], y_ref)
    assert_close("dx", out["dx"].cpu()[sel], g_ref["dx"])
    assert_close("dw", out["dw"].cpu()[sel], g_ref["dw"])
    for n in ADAPTER_GRADS:
        assert_close(n, out[n].cpu(), g_ref[n])


def _sampled_check(inp, shp, out, sample):
    """Sparse-dy parity: dy is zero outside `sample`, so every gradient only has
    contributions from the sampled tokens and the oracle can compute it exactly
    on that sub-problem; outside the sample dx and dw must be exactly zero."""
    sub, sshp, used, tok = sub_problem(inp, shp, sample)
    y_ref = oracle.forward(sub, sshp)
    g_ref = oracle.backward(sub, sshp)
    tk = tok.cuda()
    assert_close("y", out["y"][tk].cpu(), y_ref)
    assert_close("dx", out["dx"][tk].cpu(), g_ref["dx"])
    assert_close("dw", out["dw"][tk].cpu(), g_ref["dw"])
    mask = torch.ones(shp.T, dtype=torch.bool, device="cuda")
    mask[tk] = False
    assert out["dx"][mask].abs().max().item() == 0 if mask.any() else True
    assert out["dw"][mask].abs().max().item() == 0 if mask.any() else True
    ex = torch.as_tensor(used, device="cuda")
    for n in ("dA1", "dA3", "dB2"):
        assert_close(n, out[n].cpu(), g_ref[n])
    for n in ("dB1", "dB3", "dA2"):
        assert_close(n, out[n][:, ex].cpu(), g_ref[n])
        other = torch.ones(shp.E, dtype=torch.bool, device="cuda")
        other[ex] = False
        if other.any():
            assert out[n][:, other].abs().max().item() == 0, n


def _sparse_dy(inp, shp, sample):
    dy = torch.zeros_like(inp["dy"])
    idx = torch.as_tensor(sample, device=dy.device)
    dy[idx] = inp["dy"][idx]
    out = dict(inp)
    out["dy"] = dy
    return out
