"""CPU oracle for the routed MoE side-LoRA expert FFN (forward + backward).

TEST INFRASTRUCTURE: only the tests, the package smoke check and the benchmark's
CPU-baseline leg import this module.  The product (the CUDA library and its
binding) never does.  The arithmetic lives in ``moe_lora_oracle.c`` (plain C,
FP32 with bf16 rounding points, or FP64 for finite differences); this file only
compiles it with gcc and marshals torch CPU tensors to it through ctypes.

Parity pins: see tests/test_oracle_pins.py (dense merged-weight special case
against torch float64 autograd, central finite differences, zero-scale identity,
plan brute force, MXFP4 decode table, multi-adapter standalone equality) and
tests/test_router_pins.py (router against torch float64 softmax/top-k/autograd,
the closed-form logit gradient, finite differences, tie order).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_lora_oracle.c")
_LOCK = threading.Lock()
_LIBS: Dict[str, ctypes.CDLL] = {}

DT_BF16, DT_REAL, DT_MXFP4 = 0, 1, 2


def _so_path(prec: str) -> str:
    return os.path.join(_HERE, f"_liboracle_{prec}.so")


def build(force: bool = False) -> None:
    """Compile both precisions of the oracle (gcc, OpenMP, no FMA contraction)."""
    for prec in ("f32", "f64"):
        out = _so_path(prec)
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
            continue
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-Wall",
               "-o", out + ".tmp", _SRC, "-lm"]
        if prec == "f64":
            cmd.insert(1, "-DORACLE_DOUBLE")
        subprocess.run(cmd, check=True)
        os.replace(out + ".tmp", out)


class _OTensor(ctypes.Structure):
    _fields_ = [("p", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("dtype", ctypes.c_int32), ("pad_", ctypes.c_int32)]


class _ODims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("r", ctypes.c_int32),
                ("A", ctypes.c_int32), ("block_m", ctypes.c_int32), ("scale", ctypes.c_double),
                ("round_bf16", ctypes.c_int32), ("nthreads", ctypes.c_int32), ("act", ctypes.c_int32),
                ("act_quant", ctypes.c_int32), ("clamp", ctypes.c_double)]


_TENSOR_FIELDS = ("w", "x", "dy", "W1", "W3", "W2", "A1", "A3", "B1", "B3", "A2", "B2")


class _OInputs(ctypes.Structure):
    _fields_ = [("ids", ctypes.c_void_p), ("adapter_offsets", ctypes.c_void_p)] + \
               [(n, _OTensor) for n in _TENSOR_FIELDS]


def lib(prec: str = "f32") -> ctypes.CDLL:
    with _LOCK:
        if prec not in _LIBS:
            build()
            L = ctypes.CDLL(_so_path(prec))
            L.oracle_plan.restype = ctypes.c_int
            L.oracle_forward.restype = ctypes.c_int
            L.oracle_backward.restype = ctypes.c_int
            L.oracle_e2m1_value.restype = ctypes.c_double
            L.oracle_e4m3_value.restype = ctypes.c_double
            L.oracle_e4m3_round.restype = ctypes.c_double
            L.oracle_e4m3_round.argtypes = [ctypes.c_double]
            L.oracle_mxfp8_quantize.restype = ctypes.c_int
            L.oracle_ue8m0_value.restype = ctypes.c_double
            L.oracle_round_bf16.restype = ctypes.c_double
            L.oracle_round_bf16.argtypes = [ctypes.c_double]
            L.oracle_router_forward.restype = ctypes.c_int
            L.oracle_router_backward.restype = ctypes.c_int
            _LIBS[prec] = L
        return _LIBS[prec]


def _real_dtype(prec: str):
    return torch.float32 if prec == "f32" else torch.float64


class _Keep:
    """Holds tensors alive while a ctypes call uses their storage."""

    def __init__(self):
        self.items = []

    def __call__(self, t):
        self.items.append(t)
        return t


def _otensor(t: Optional[torch.Tensor], prec: str, keep: _Keep, scales=None) -> _OTensor:
    if t is None:
        return _OTensor(None, None, DT_REAL, 0)
    t = keep(t.detach().contiguous().cpu())
    if t.dtype == torch.bfloat16:
        return _OTensor(t.data_ptr(), None, DT_BF16, 0)
    if t.dtype == torch.uint8:
        assert scales is not None
        s = keep(scales.detach().contiguous().cpu())
        return _OTensor(t.data_ptr(), s.data_ptr(), DT_MXFP4, 0)
    t = keep(t.to(_real_dtype(prec)).contiguous())
    return _OTensor(t.data_ptr(), None, DT_REAL, 0)


def _pack(inp: dict, shp, prec: str, scale: float, round_bf16: bool, nthreads: int):
    keep = _Keep()
    d = _ODims(shp.T, shp.H, shp.I, shp.E, shp.k, shp.r, shp.A, 128, float(scale),
               1 if round_bf16 else 0, nthreads, 1 if shp.act == "geglu" else 0,
               1 if shp.base_fmt == "mxfp4_native" else 0, float(shp.clamp))
    ids = keep(inp["topk_ids"].to(torch.int32).contiguous().cpu())
    offs = keep(inp["adapter_offsets"].to(torch.int64).contiguous().cpu())
    fields = {}
    for n in _TENSOR_FIELDS:
        sc = inp.get("S" + n[1]) if n in ("W1", "W3", "W2") else None
        t = inp.get("topk_w") if n == "w" else inp.get(n)
        fields[n] = _otensor(t, prec, keep, sc)
    o = _OInputs(ids.data_ptr(), offs.data_ptr(), **fields)
    return d, o, keep


def _tok(tokens, keep):
    if tokens is None:
        return None, None
    tt = keep(torch.as_tensor(list(tokens) if not isinstance(tokens, torch.Tensor) else tokens,
                              dtype=torch.int64).contiguous())
    return tt, ctypes.c_void_p(tt.data_ptr())


def forward(inp: dict, shp, tokens: Optional[Sequence[int]] = None, prec: str = "f32",
            scale: Optional[float] = None, round_bf16: bool = True, nthreads: int = 0) -> torch.Tensor:
    """y for the listed tokens (all tokens if None): [ntok, H] in the oracle's precision."""
    L = lib(prec)
    d, o, keep = _pack(inp, shp, prec, shp.scale if scale is None else scale, round_bf16, nthreads)
    tt, tp = _tok(tokens, keep)
    ntok = shp.T if tt is None else tt.numel()
    y = torch.zeros(ntok, shp.H, dtype=_real_dtype(prec))
    rc = L.oracle_forward(ctypes.byref(d), ctypes.byref(o), tp, ctypes.c_int64(ntok),
                          ctypes.c_void_p(y.data_ptr()))
    assert rc == 0
    return y


def backward(inp: dict, shp, tokens: Optional[Sequence[int]] = None, prec: str = "f32",
             scale: Optional[float] = None, round_bf16: bool = True, nthreads: int = 0) -> Dict[str, torch.Tensor]:
    """Gradients with dy restricted to the listed tokens (all if None).

    Returns dx [ntok,H], dw [ntok,k] for the listed tokens and the adapter gradients
    dA1/dA3 [A,r,H], dB1/dB3 [A,E,I,r], dA2 [A,E,r,I], dB2 [A,H,r] summed over them."""
    L = lib(prec)
    d, o, keep = _pack(inp, shp, prec, shp.scale if scale is None else scale, round_bf16, nthreads)
    tt, tp = _tok(tokens, keep)
    ntok = shp.T if tt is None else tt.numel()
    rd = _real_dtype(prec)
    A, E, H, I, r, k = shp.A, shp.E, shp.H, shp.I, shp.r, shp.k
    out = {
        "dx": torch.zeros(ntok, H, dtype=rd), "dw": torch.zeros(ntok, k, dtype=rd),
        "dA1": torch.zeros(A, r, H, dtype=rd), "dA3": torch.zeros(A, r, H, dtype=rd),
        "dB1": torch.zeros(A, E, I, r, dtype=rd), "dB3": torch.zeros(A, E, I, r, dtype=rd),
        "dA2": torch.zeros(A, E, r, I, dtype=rd), "dB2": torch.zeros(A, H, r, dtype=rd),
    }
    ptrs = [ctypes.c_void_p(out[n].data_ptr()) for n in ("dx", "dw", "dA1", "dA3", "dB1", "dB3", "dA2", "dB2")]
    rc = L.oracle_backward(ctypes.byref(d), ctypes.byref(o), tp, ctypes.c_int64(ntok), *ptrs)
    assert rc == 0
    return out


def plan(ids: torch.Tensor, E: int, adapter_offsets: torch.Tensor, block_m: int = 128):
    """Routing plan: counts [A*E] and offsets [A*E+1] by group slot q = e*A + a,
    row_of_route [T*k], route_of_row [P]."""
    L = lib("f32")
    ids = ids.to(torch.int32).contiguous().cpu()
    T, k = ids.shape
    offs = adapter_offsets.to(torch.int64).contiguous().cpu()
    A = offs.numel() - 1
    G = A * E
    cap = T * k + G * (block_m - 1)
    counts = torch.zeros(G, dtype=torch.int32)
    offsets = torch.zeros(G + 1, dtype=torch.int32)
    ror = torch.zeros(T * k, dtype=torch.int32)
    rrow = torch.zeros(max(cap, 1), dtype=torch.int32)
    bad = L.oracle_plan(ctypes.c_int64(T), k, E, A, block_m, ctypes.c_void_p(ids.data_ptr()),
                        ctypes.c_void_p(offs.data_ptr()), ctypes.c_void_p(counts.data_ptr()),
                        ctypes.c_void_p(offsets.data_ptr()), ctypes.c_void_p(ror.data_ptr()),
                        ctypes.c_void_p(rrow.data_ptr()), ctypes.c_int64(cap))
    P = int(offsets[-1])
    return {"counts": counts, "offsets": offsets, "row_of_route": ror,
            "route_of_row": rrow[:P].clone(), "bad": bad}


def e2m1_value(code: int) -> float:
    return lib("f32").oracle_e2m1_value(ctypes.c_int(code))


def e4m3_value(code: int) -> float:
    return lib("f32").oracle_e4m3_value(ctypes.c_int(code))


def e4m3_round(v: float) -> float:
    return lib("f32").oracle_e4m3_round(v)


def mxfp8_quantize(v: torch.Tensor, prec: str = "f32"):
    """MXFP8 (E4M3 elements, one UE8M0 scale per 32 from the start) of a 1-D tensor:
    (codes uint8 [n], scale bytes uint8 [ceil(n/32)], dequantised float64 [n]).  prec:
    the oracle build whose arithmetic quantises (f32 reads the values as fp32)."""
    v = v.detach().double().contiguous().cpu().flatten()
    n = v.numel()
    codes = torch.zeros(n, dtype=torch.uint8)
    scales = torch.zeros((n + 31) // 32, dtype=torch.uint8)
    deq = torch.zeros(n, dtype=torch.float64)
    bad = lib(prec).oracle_mxfp8_quantize(ctypes.c_void_p(v.data_ptr()), ctypes.c_int64(n),
                                           ctypes.c_void_p(codes.data_ptr()), ctypes.c_void_p(scales.data_ptr()),
                                           ctypes.c_void_p(deq.data_ptr()))
    assert bad == 0
    return codes, scales, deq


def ue8m0_value(b: int) -> float:
    return lib("f32").oracle_ue8m0_value(ctypes.c_int(b))


def round_bf16(v: float) -> float:
    return lib("f32").oracle_round_bf16(v)


def _router_args(x: torch.Tensor, Wr: torch.Tensor, prec: str, keep: _Keep):
    T, H = x.shape
    E = Wr.shape[0]
    assert Wr.shape[1] == H
    return T, H, E, _otensor(x, prec, keep), _otensor(Wr, prec, keep)


def router_forward(x: torch.Tensor, Wr: torch.Tensor, k: int, prec: str = "f32", nthreads: int = 0):
    """Softmax top-k router: logits [T,E], ids [T,k] int32, w [T,k] (oracle precision)."""
    L = lib(prec)
    keep = _Keep()
    T, H, E, xo, wo = _router_args(x, Wr, prec, keep)
    rd = _real_dtype(prec)
    logits = torch.zeros(T, E, dtype=rd)
    ids = torch.zeros(T, k, dtype=torch.int32)
    w = torch.zeros(T, k, dtype=rd)
    rc = L.oracle_router_forward(ctypes.c_int64(T), H, E, k, nthreads, ctypes.byref(xo), ctypes.byref(wo),
                                 ctypes.c_void_p(logits.data_ptr()), ctypes.c_void_p(ids.data_ptr()),
                                 ctypes.c_void_p(w.data_ptr()))
    assert rc == 0
    return logits, ids, w


def router_backward(x: torch.Tensor, Wr: torch.Tensor, ids: torch.Tensor, dw: torch.Tensor, prec: str = "f32",
                    nthreads: int = 0):
    """Router backward for a fixed selection: dlogits [T,E], dWr [E,H], and the
    router's part of grad-x [T,H] (oracle precision)."""
    L = lib(prec)
    keep = _Keep()
    T, H, E, xo, wo = _router_args(x, Wr, prec, keep)
    k = ids.shape[1]
    rd = _real_dtype(prec)
    ids = keep(ids.to(torch.int32).contiguous().cpu())
    dw = keep(dw.detach().to(rd).contiguous().cpu())
    dl = torch.zeros(T, E, dtype=rd)
    dWr = torch.zeros(E, H, dtype=rd)
    dx = torch.zeros(T, H, dtype=rd)
    rc = L.oracle_router_backward(ctypes.c_int64(T), H, E, k, nthreads, ctypes.byref(xo), ctypes.byref(wo),
                                  ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(dw.data_ptr()),
                                  ctypes.c_void_p(dl.data_ptr()), ctypes.c_void_p(dWr.data_ptr()),
                                  ctypes.c_void_p(dx.data_ptr()))
    assert rc == 0
    return dl, dWr, dx
