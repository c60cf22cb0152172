"""Seeded synthetic inputs for the routed MoE SwiGLU expert FFN with side-LoRA.

This module is shared by the CUDA path's tests/benchmark and by the CPU oracle's
tests.  It draws random numbers, routes tokens (softmax over experts, top-k,
renormalised weights) and packs MXFP4 fixtures; it holds none of the expert-FFN
arithmetic that the oracle and the kernels compute.

Workload shapes follow the pages' fixtures:
  * "tiny": the small exact-oracle shape of "Align MegaMoE training with upgraded
    K-grouped TMA and layouts" (DeepGEMM PR #17), Validation: 256 tokens, H=512,
    I=256, E=16, top-2 (rank 16 added for the side adapters).
  * "edge": the production-width sweep of "feat(mega): add fused shared side-LoRA
    kernels" (DeepGEMM PR #9), Correctness coverage: H=4096, I=2048, 256 experts,
    top-6, rank 128, 20% masked routes, the 15 token counts listed there.
  * "prod": the matched production shape of the same PR, Matched production-shape
    performance: 65,536 tokens, H=4096, I=2048, E=256, top-6, rank 128.
  * "prod_mxfp4": the same with an MXFP4 (E2M1 + UE8M0 per 32) frozen base.
  * "prod_native": "prod_mxfp4" with the gate/up products on block-scaled FP4
    tensor cores (MXFP8 activations), the "native MXFP4" base the same PR times
    beside the dequantised one (Performance).
  * "multi": several adapters sharing one MoE layer, after OpenPipe/ART PR #1139,
    Behavior (dispatched expert rows carry adapter ids).
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Dict, Optional

import torch

EDGE_TOKEN_COUNTS = (1, 15, 16, 17, 90, 91, 176, 177, 346, 347, 688, 689, 1029, 1030, 2048)


@dataclasses.dataclass(frozen=True)
class Shape:
    T: int
    H: int
    I: int
    E: int
    k: int
    r: int
    A: int = 1            # adapters sharing the layer
    scale: float = 1.0    # side-LoRA scale s
    mask_frac: float = 0.0  # fraction of (token, slot) routes masked out
    empty_experts: tuple = ()  # experts that receive no token
    router: str = "linear"  # "linear": logits = x W_r^T ; "normal": logits ~ N(0,1)
    base_fmt: str = "bf16"  # "bf16", "mxfp4", or "mxfp4_native" (MXFP4 base, MXFP8 gate/up activations)
    act: str = "swiglu"     # "swiglu" or "geglu"
    clamp: float = 0.0      # activation clamp c on the gate/up pre-activations (0 = none)


def shape(name: str, T: Optional[int] = None) -> Shape:
    if name == "tiny":
        return Shape(T=T or 256, H=512, I=256, E=16, k=2, r=16)
    if name == "edge":
        return Shape(T=T or 2048, H=4096, I=2048, E=256, k=6, r=128, mask_frac=0.2,
                     empty_experts=(0, 127, 255))
    if name == "prod":
        return Shape(T=T or 65536, H=4096, I=2048, E=256, k=6, r=128, router="normal")
    if name == "prod_e16":
        # production widths with 16 experts and 4,096 tokens: the same ~1,536 rows
        # per expert as "prod" in a few GB of device memory (profiler captures)
        return Shape(T=T or 4096, H=4096, I=2048, E=16, k=6, r=128, router="normal")
    if name == "prod_e16_mxfp4":
        # "prod_e16" with an MXFP4 base (profiler captures of the MXFP4-decoding GEMMs)
        return Shape(T=T or 4096, H=4096, I=2048, E=16, k=6, r=128, router="normal", base_fmt="mxfp4")
    if name == "prod_mxfp4":
        return Shape(T=T or 65536, H=4096, I=2048, E=256, k=6, r=128, router="normal",
                     base_fmt="mxfp4")
    if name == "prod_e16_native":
        return Shape(T=T or 4096, H=4096, I=2048, E=16, k=6, r=128, router="normal", base_fmt="mxfp4_native")
    if name == "prod_native":
        return Shape(T=T or 65536, H=4096, I=2048, E=256, k=6, r=128, router="normal",
                     base_fmt="mxfp4_native")
    if name == "multi":
        return Shape(T=T or 16384, H=2048, I=768, E=128, k=8, r=8, A=16)
    raise KeyError(name)


def _randn(g, shp, std, device):
    return torch.randn(*shp, generator=g, device=device, dtype=torch.float32).mul_(std)


def _randn_bf16(g, shp, std, device, chunk_dim0: int = 0):
    """N(0, std^2) rounded to bf16; generated in slices along dim 0 to bound fp32 temporaries."""
    if chunk_dim0 <= 0 or shp[0] <= chunk_dim0:
        return _randn(g, shp, std, device).to(torch.bfloat16)
    out = torch.empty(*shp, dtype=torch.bfloat16, device=device)
    for s in range(0, shp[0], chunk_dim0):
        e = min(shp[0], s + chunk_dim0)
        out[s:e] = _randn(g, (e - s,) + tuple(shp[1:]), std, device).to(torch.bfloat16)
    return out


def route_topk(logits: torch.Tensor, k: int):
    """Softmax over experts, top-k by descending probability (ties -> lower expert id),
    weights renormalised to sum to 1 in fp32 and then rounded to bf16 values."""
    prob = torch.softmax(logits.float(), dim=-1)
    order = torch.sort(-prob, dim=-1, stable=True).indices[:, :k]
    w = torch.gather(prob, 1, order)
    w = w / w.sum(dim=-1, keepdim=True)
    return order.to(torch.int32), w.to(torch.bfloat16).float()


# --------------------------------------------------------------------------------------
# MXFP4 fixture quantiser: E2M1 element codes with one UE8M0 scale per 32 contiguous K.
# (Encoding of the OCP Microscaling formats: E2M1 magnitudes {0,.5,1,1.5,2,3,4,6},
#  UE8M0 byte b -> 2^(b-127).)  Round-to-nearest with ties to the even code, saturating.
# --------------------------------------------------------------------------------------
_E2M1_GRID = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def mxfp4_quantize(w: torch.Tensor, chunk: int = 1 << 22):
    """w: [..., K] (K % 32 == 0) -> (packed uint8 [..., K/2], scales uint8 [..., K/32]).
    Low nibble holds the element with the lower K index.  Large tensors are
    quantised in slices of `chunk` 32-element groups to bound temporaries."""
    K = w.shape[-1]
    groups = w.numel() // 32
    if groups > chunk:
        flat = w.reshape(-1, 32)
        parts = [_mxfp4_quantize(flat[s:s + chunk]) for s in range(0, groups, chunk)]
        packed = torch.cat([p for p, _ in parts]).reshape(*w.shape[:-1], K // 2)
        scales = torch.cat([q for _, q in parts]).reshape(*w.shape[:-1], K // 32)
        return packed.contiguous(), scales.contiguous()
    return _mxfp4_quantize(w)


def _mxfp4_quantize(w: torch.Tensor):
    K = w.shape[-1]
    assert K % 32 == 0
    lead = w.shape[:-1]
    wf = w.float().reshape(-1, K // 32, 32)
    amax = wf.abs().amax(dim=-1)
    e = torch.where(amax > 0, torch.floor(torch.log2(amax.clamp_min(1e-38))) - 2, torch.zeros_like(amax))
    e = e.clamp(-127, 127)
    scale = torch.exp2(e)
    v = (wf / scale.unsqueeze(-1)).abs().clamp(max=6.0)
    grid = _E2M1_GRID.to(v.device)
    d = (v.unsqueeze(-1) - grid).abs()                 # [..., 32, 8]
    best = d.min(dim=-1, keepdim=True).values
    cand = (d == best)
    # ties -> the even code (even mantissa bit); otherwise the unique nearest.
    codes = torch.arange(8, device=v.device)
    even_pref = cand & (codes % 2 == 0)
    pick = torch.where(even_pref.any(dim=-1, keepdim=True), even_pref, cand)
    mag = pick.float().argmax(dim=-1)                  # first candidate
    sign = (wf < 0) & (mag > 0)
    code = (mag + sign.long() * 8).to(torch.uint8).reshape(*lead, K)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).to(torch.uint8)
    sbytes = (e + 127).to(torch.uint8).reshape(*lead, K // 32)
    return packed.contiguous(), sbytes.contiguous()


def make_inputs(shp: Shape, seed: int = 0, device: str = "cpu") -> Dict[str, torch.Tensor]:
    """All tensors of one seeded problem instance (bf16 values unless noted).

    x [T,H]; topk_ids [T,k] int32 (-1 = masked route); topk_w [T,k] fp32 (bf16 values);
    W1, W3 [E,I,H]; W2 [E,H,I]; A1, A3 [A,r,H]; B1, B3 [A,E,I,r]; A2 [A,E,r,I]; B2 [A,H,r];
    dy [T,H]; adapter_offsets [A+1] int64 (tokens of adapter a are [off[a], off[a+1])).
    For an MXFP4 base, W1/W3/W2 hold packed E2M1 codes and S1/S3/S2 their UE8M0 scales.
    """
    T, H, I, E, k, r, A = shp.T, shp.H, shp.I, shp.E, shp.k, shp.r, shp.A
    g = torch.Generator(device=device).manual_seed(seed)
    out: Dict[str, torch.Tensor] = {}
    sH, sI = 1.0 / math.sqrt(H), 1.0 / math.sqrt(I)
    out["x"] = _randn_bf16(g, (T, H), 1.0, device, 8192)
    # routing (per adapter when several share the layer)
    per = T // A
    assert per * A == T
    ids, ws = [], []
    for a in range(A):
        xa = out["x"][a * per:(a + 1) * per]
        if shp.router == "normal":
            logits = _randn(g, (per, E), 1.0, device)
        else:
            Wr = _randn_bf16(g, (E, H), sH, device)
            logits = xa.float() @ Wr.float().t()
        for e in shp.empty_experts:
            logits[:, e] = -math.inf
        i_a, w_a = route_topk(logits, k)
        ids.append(i_a)
        ws.append(w_a)
    ids = torch.cat(ids, 0)
    w = torch.cat(ws, 0)
    if shp.mask_frac > 0:
        m = torch.rand(T, k, generator=g, device=device) < shp.mask_frac
        ids = torch.where(m, torch.full_like(ids, -1), ids)
        w = torch.where(m, torch.zeros_like(w), w)
    out["topk_ids"] = ids.contiguous()
    out["topk_w"] = w.contiguous()
    out["W1"] = _randn_bf16(g, (E, I, H), sH, device, 8)
    out["W3"] = _randn_bf16(g, (E, I, H), sH, device, 8)
    out["W2"] = _randn_bf16(g, (E, H, I), sI, device, 8)
    if shp.base_fmt in ("mxfp4", "mxfp4_native"):
        for n in ("W1", "W3", "W2"):
            p, s = mxfp4_quantize(out[n])
            out[n] = p
            out["S" + n[1]] = s
    out["A1"] = _randn_bf16(g, (A, r, H), sH, device)
    out["A3"] = _randn_bf16(g, (A, r, H), sH, device)
    out["B1"] = _randn_bf16(g, (A, E, I, r), 0.02, device)
    out["B3"] = _randn_bf16(g, (A, E, I, r), 0.02, device)
    out["A2"] = _randn_bf16(g, (A, E, r, I), sI, device)
    out["B2"] = _randn_bf16(g, (A, H, r), 0.02, device)
    out["dy"] = _randn_bf16(g, (T, H), 1.0, device, 8192)
    out["adapter_offsets"] = torch.arange(0, T + 1, per, dtype=torch.int64)
    return out


def make_router_inputs(T: int, H: int, E: int, k: int, seed: int = 0, device: str = "cpu",
                       A: int = 0) -> Dict[str, torch.Tensor]:
    """Inputs of the routing step: x [T,H] ~ N(0,1), W_r [E,H] ~ N(0, 1/H) (bf16 values;
    [A,E,H], one router per adapter, when A > 0); the upstream routing-weight gradient
    dw [T,k] ~ N(0,1) fp32 and a grad-x the router adds into, dx0 [T,H] ~ N(0,1) bf16."""
    g = torch.Generator(device=device).manual_seed(seed)
    return {"x": _randn_bf16(g, (T, H), 1.0, device, 8192),
            "Wr": _randn_bf16(g, (A, E, H) if A > 0 else (E, H), 1.0 / math.sqrt(H), device),
            "dw": _randn(g, (T, k), 1.0, device),
            "dx0": _randn_bf16(g, (T, H), 1.0, device, 8192)}


def sha256(t: torch.Tensor) -> str:
    """SHA-256 of a tensor's bytes (input manifests)."""
    b = t.detach().contiguous().cpu().view(torch.uint8).numpy().tobytes()
    return hashlib.sha256(b).hexdigest()
