"""GB300 (sm_103a) routed MoE SwiGLU expert FFN with rank-r side-LoRA adapters.

Thin Python binding over ``libmoelora.so`` (C ABI, ``include/moe_lora.h``).  The
functions below carry the C names and only marshal arguments: torch CUDA tensors
become device pointers, the current torch stream becomes the ``cudaStream_t``.
Every step of the path runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback, and importing a function fails loudly if the library is
missing (build it with ``moe_expert_ffn_top_gb300._build.build()``).

The method ("feat(mega): add fused shared side-LoRA kernels", DeepGEMM PR #9,
Summary): shared A1/A3/B2 side factors, expert-local B1/B3/A2, frozen W1/W2/W3;
the backward returns grad-x, router-weight gradients and the six adapter
gradients.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Dict, Optional, Sequence

import torch

from . import _build

LIB_PATH = _build.LIB

MOE_LORA_WS_PLAN, MOE_LORA_WS_SAVED, MOE_LORA_WS_FWD_SCRATCH, MOE_LORA_WS_BWD_SCRATCH = 0, 1, 2, 3
MOE_LORA_WS_ROUTER_SCRATCH = 4
MOE_LORA_DEV_BAD_ID, MOE_LORA_DEV_TIMEOUT = 1, 2


class MoeLoraError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {moe_lora_strerror(code)} (code {code})")
        self.code = code


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("r", ctypes.c_int32), ("A", ctypes.c_int32), ("block_m", ctypes.c_int32),
                ("scale", ctypes.c_float), ("act", ctypes.c_int32), ("base_fmt", ctypes.c_int32),
                ("act_clamp", ctypes.c_float)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("W1", "W3", "W2", "A1", "A3", "B1", "B3", "A2", "B2",
                                                 "S1", "S3", "S2")]


class Grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("dA1", "dA3", "dB1", "dB3", "dA2", "dB2")]


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run moe_expert_ffn_top_gb300._build.build() first")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        L.moe_lora_workspace_bytes.restype = ctypes.c_size_t
        L.moe_lora_workspace_bytes.argtypes = [ctypes.POINTER(Dims), ctypes.c_int]
        L.moe_lora_plan.restype = ctypes.c_int
        L.moe_lora_plan.argtypes = [ctypes.POINTER(Dims), P, P, P, ctypes.c_size_t, P]
        L.moe_lora_forward.restype = ctypes.c_int
        L.moe_lora_forward.argtypes = [ctypes.POINTER(Dims), P, P, P, ctypes.POINTER(Weights), P, P,
                                       ctypes.c_size_t, P, ctypes.c_size_t, P]
        L.moe_lora_backward.restype = ctypes.c_int
        L.moe_lora_backward.argtypes = [ctypes.POINTER(Dims), P, P, P, P, P, ctypes.POINTER(Weights), P, P,
                                        ctypes.POINTER(Grads), P, ctypes.c_size_t, P]
        L.moe_lora_get_error.restype = ctypes.c_int
        L.moe_lora_get_error.argtypes = [ctypes.POINTER(Dims), P, P]
        L.moe_lora_plan_noalloc.restype = ctypes.c_int
        L.moe_lora_plan_noalloc.argtypes = [ctypes.POINTER(Dims), P, P, P, ctypes.c_size_t, P]
        L.moe_lora_plan_readback.restype = ctypes.c_int
        L.moe_lora_plan_readback.argtypes = [ctypes.POINTER(Dims), P, P, P, P, P, ctypes.c_int64, P]
        L.moe_lora_strerror.restype = ctypes.c_char_p
        L.moe_lora_strerror.argtypes = [ctypes.c_int]
        L.moe_lora_gemm_selftest.restype = ctypes.c_int
        L.moe_lora_gemm_selftest.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, ctypes.c_int32, P,
                                             ctypes.c_int32, P, P]
        L.moe_lora_gemm_pair_selftest.restype = ctypes.c_int
        L.moe_lora_gemm_pair_selftest.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, ctypes.c_int32,
                                                  P, ctypes.c_int32, P, P]
        L.moe_lora_gemm_starved_selftest.restype = ctypes.c_int
        L.moe_lora_gemm_starved_selftest.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P,
                                                     ctypes.c_int32, P, ctypes.c_int32, P, ctypes.c_int32, P]
        L.moe_lora_native_selftest.restype = ctypes.c_int
        L.moe_lora_native_selftest.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, P, P, P, P,
                                               ctypes.c_int32, P]
        L.moe_lora_mxfp8_quantize.restype = ctypes.c_int
        L.moe_lora_mxfp8_quantize.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P, P, P]
        L.moe_lora_mxfp4_decode.restype = ctypes.c_int
        L.moe_lora_mxfp4_decode.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                             ctypes.c_void_p]
        L.moe_lora_profile_enable.restype = ctypes.c_int
        L.moe_lora_profile_enable.argtypes = [ctypes.c_int]
        L.moe_lora_profile_select.restype = ctypes.c_int
        L.moe_lora_profile_select.argtypes = [ctypes.c_char_p]
        L.moe_lora_profile_read.restype = ctypes.c_int
        L.moe_lora_profile_read.argtypes = [P, P, P, ctypes.c_int]
        L.moe_lora_launch_count.restype = ctypes.c_int64
        L.moe_lora_launch_count.argtypes = [ctypes.c_int]
        L.moe_lora_gemm_selftest_error.restype = ctypes.c_int
        L.moe_lora_gemm_selftest_error.argtypes = [P]
        L.moe_lora_router_forward.restype = ctypes.c_int
        L.moe_lora_router_forward.argtypes = [ctypes.POINTER(Dims), P, P, P, P, P, P, P, ctypes.c_size_t, P]
        L.moe_lora_router_backward.restype = ctypes.c_int
        L.moe_lora_router_backward.argtypes = [ctypes.POINTER(Dims), P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t,
                                               P]
        L.moe_lora_router_get_error.restype = ctypes.c_int
        L.moe_lora_router_get_error.argtypes = [P, P]
        _lib = L
    return _lib


def make_dims(T: int, H: int, I: int, E: int, k: int, r: int, A: int = 1, scale: float = 1.0,
              base_fmt: int = 0, act: int = 0, act_clamp: float = 0.0) -> Dims:
    """base_fmt: 0 = bf16 base weights; MXFP4 (packed E2M1 codes + UE8M0 scales S1/S3/S2) decoded
    inside the GEMMs (1) or once per pass into the saved workspace (2); 3 / 4 = the native FP4
    forward (gate/up base products on block-scaled FP4 tensor cores from MXFP8 activations,
    the rest as 1 / as 2; H and I multiples of 128);
    act: 0 = SwiGLU, 1 = GeGLU; act_clamp: clamp of the gate/up pre-activations (0 = none)."""
    return Dims(T, H, I, E, k, r, A, 128, float(scale), int(act), int(base_fmt), float(act_clamp))


def _ptr(t: Optional[torch.Tensor], dtype=None, name: str = "") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise MoeLoraError(rc, what)


def moe_lora_strerror(code: int) -> str:
    return lib().moe_lora_strerror(code).decode()


def moe_lora_workspace_bytes(dims: Dims, which: int) -> int:
    return int(lib().moe_lora_workspace_bytes(ctypes.byref(dims), which))


def moe_lora_plan(dims: Dims, topk_ids: torch.Tensor, adapter_offsets: Optional[Sequence[int]],
                  plan_ws: torch.Tensor, stream=None) -> None:
    offs = None
    if adapter_offsets is not None:
        vals = [int(v) for v in adapter_offsets]
        offs = (ctypes.c_int64 * len(vals))(*vals)
    rc = lib().moe_lora_plan(ctypes.byref(dims), _ptr(topk_ids, torch.int32, "topk_ids"),
                             ctypes.cast(offs, ctypes.c_void_p) if offs is not None else None,
                             _ptr(plan_ws, None, "plan_ws"), plan_ws.numel() * plan_ws.element_size(),
                             _stream(stream))
    _check(rc, "moe_lora_plan")


def moe_lora_plan_noalloc(dims: Dims, topk_ids: torch.Tensor, adapter_offsets: Optional[Sequence[int]],
                          plan_ws: torch.Tensor, plan_bytes: Optional[int] = None, stream=None) -> None:
    """The routing plan without caller-provided temporary space (see the C header):
    plan_ws only needs to hold the plan itself."""
    offs = None
    if adapter_offsets is not None:
        vals = [int(v) for v in adapter_offsets]
        offs = (ctypes.c_int64 * len(vals))(*vals)
    nbytes = plan_ws.numel() * plan_ws.element_size() if plan_bytes is None else plan_bytes
    rc = lib().moe_lora_plan_noalloc(ctypes.byref(dims), _ptr(topk_ids, torch.int32, "topk_ids"),
                                     ctypes.cast(offs, ctypes.c_void_p) if offs is not None else None,
                                     _ptr(plan_ws, None, "plan_ws"), nbytes, _stream(stream))
    _check(rc, "moe_lora_plan_noalloc")


def moe_lora_plan_readback(dims: Dims, plan_ws: torch.Tensor, stream=None) -> Dict[str, torch.Tensor]:
    """Host copies of the plan: counts, offsets, row_of_route, route_of_row."""
    G = dims.A * dims.E
    counts = torch.zeros(G, dtype=torch.int32)
    offsets = torch.zeros(G + 1, dtype=torch.int32)
    ror = torch.zeros(max(dims.T * dims.k, 1), dtype=torch.int32)
    cap = dims.T * dims.k + G * 128
    rrow = torch.zeros(max(cap, 1), dtype=torch.int32)
    rc = lib().moe_lora_plan_readback(ctypes.byref(dims), _ptr(plan_ws), counts.data_ptr(), offsets.data_ptr(),
                                      ror.data_ptr(), rrow.data_ptr(), cap, _stream(stream))
    _check(rc, "moe_lora_plan_readback")
    P = int(offsets[-1])
    return {"counts": counts, "offsets": offsets, "row_of_route": ror[:dims.T * dims.k],
            "route_of_row": rrow[:P].clone()}


def _weights(w: Dict[str, torch.Tensor], dims: Dims) -> Weights:
    mx = dims.base_fmt in (1, 2, 3, 4)
    base = [_ptr(w[n], torch.uint8 if mx else torch.bfloat16, n) for n in ("W1", "W3", "W2")]
    side = [_ptr(w[n], torch.bfloat16, n) for n in ("A1", "A3", "B1", "B3", "A2", "B2")]
    scales = [_ptr(w[n], torch.uint8, n) if mx else None for n in ("S1", "S3", "S2")]
    return Weights(*(base + side + scales))


def moe_lora_forward(dims: Dims, plan_ws: torch.Tensor, x: torch.Tensor, topk_w: torch.Tensor,
                     weights: Dict[str, torch.Tensor], y: torch.Tensor, saved: torch.Tensor,
                     scratch: torch.Tensor, stream=None) -> None:
    W = _weights(weights, dims)
    rc = lib().moe_lora_forward(ctypes.byref(dims), _ptr(plan_ws), _ptr(x, torch.bfloat16, "x"),
                                _ptr(topk_w, torch.float32, "topk_w"), ctypes.byref(W),
                                _ptr(y, torch.bfloat16, "y"), _ptr(saved), saved.numel() * saved.element_size(),
                                _ptr(scratch), scratch.numel() * scratch.element_size(), _stream(stream))
    _check(rc, "moe_lora_forward")


def moe_lora_backward(dims: Dims, plan_ws: torch.Tensor, saved: torch.Tensor, x: torch.Tensor,
                      topk_w: torch.Tensor, dy: torch.Tensor, weights: Dict[str, torch.Tensor],
                      dx: torch.Tensor, dw: torch.Tensor, grads: Dict[str, torch.Tensor],
                      scratch: torch.Tensor, stream=None) -> None:
    W = _weights(weights, dims)
    Gr = Grads(*[_ptr(grads[n], torch.float32, n) for n in ("dA1", "dA3", "dB1", "dB3", "dA2", "dB2")])
    rc = lib().moe_lora_backward(ctypes.byref(dims), _ptr(plan_ws), _ptr(saved), _ptr(x, torch.bfloat16, "x"),
                                 _ptr(topk_w, torch.float32, "topk_w"), _ptr(dy, torch.bfloat16, "dy"),
                                 ctypes.byref(W), _ptr(dx, torch.bfloat16, "dx"), _ptr(dw, torch.float32, "dw"),
                                 ctypes.byref(Gr), _ptr(scratch), scratch.numel() * scratch.element_size(),
                                 _stream(stream))
    _check(rc, "moe_lora_backward")


def moe_lora_get_error(dims: Dims, plan_ws: torch.Tensor, stream=None) -> int:
    rc = lib().moe_lora_get_error(ctypes.byref(dims), _ptr(plan_ws), _stream(stream))
    if rc < 0:
        raise MoeLoraError(rc, "moe_lora_get_error")
    return rc


def _offsets(adapter_offsets: Optional[Sequence[int]]):
    if adapter_offsets is None:
        return None
    vals = [int(v) for v in adapter_offsets]
    return (ctypes.c_int64 * len(vals))(*vals)


def moe_lora_router_forward(dims: Dims, x: torch.Tensor, Wr: torch.Tensor, topk_ids: torch.Tensor,
                            topk_w: torch.Tensor, logits: Optional[torch.Tensor], scratch: torch.Tensor,
                            stream=None, adapter_offsets: Optional[Sequence[int]] = None) -> None:
    """Softmax top-k router: topk_ids [T,k] int32, topk_w [T,k] fp32 (and logits [T,E] fp32 if given).
    W_r is [E,H] or [A,E,H]; adapter_offsets [A+1] (host) splits the tokens between adapters."""
    offs = _offsets(adapter_offsets)
    rc = lib().moe_lora_router_forward(ctypes.byref(dims), _ptr(x, torch.bfloat16, "x"),
                                       _ptr(Wr, torch.bfloat16, "Wr"),
                                       ctypes.cast(offs, ctypes.c_void_p) if offs is not None else None,
                                       _ptr(topk_ids, torch.int32, "topk_ids"),
                                       _ptr(topk_w, torch.float32, "topk_w"), _ptr(logits, torch.float32, "logits"),
                                       _ptr(scratch), scratch.numel() * scratch.element_size(), _stream(stream))
    _check(rc, "moe_lora_router_forward")


def moe_lora_router_backward(dims: Dims, x: torch.Tensor, Wr: torch.Tensor, topk_ids: torch.Tensor,
                             topk_w: torch.Tensor, dw: torch.Tensor, dlogits: Optional[torch.Tensor],
                             dWr: torch.Tensor, dx: torch.Tensor, scratch: torch.Tensor, stream=None,
                             adapter_offsets: Optional[Sequence[int]] = None) -> None:
    """Router backward: dWr [E,H] or [A,E,H] fp32 (and dlogits [T,E] fp32 if given); dx [T,H]
    bf16 is updated in place, dx <- bf16(dx + dlogits W_r)."""
    offs = _offsets(adapter_offsets)
    rc = lib().moe_lora_router_backward(ctypes.byref(dims), _ptr(x, torch.bfloat16, "x"),
                                        _ptr(Wr, torch.bfloat16, "Wr"),
                                        ctypes.cast(offs, ctypes.c_void_p) if offs is not None else None,
                                        _ptr(topk_ids, torch.int32, "topk_ids"),
                                        _ptr(topk_w, torch.float32, "topk_w"), _ptr(dw, torch.float32, "dw"),
                                        _ptr(dlogits, torch.float32, "dlogits"), _ptr(dWr, torch.float32, "dWr"),
                                        _ptr(dx, torch.bfloat16, "dx"), _ptr(scratch),
                                        scratch.numel() * scratch.element_size(), _stream(stream))
    _check(rc, "moe_lora_router_backward")


def moe_lora_router_get_error(scratch: torch.Tensor, stream=None) -> int:
    rc = lib().moe_lora_router_get_error(_ptr(scratch), _stream(stream))
    if rc < 0:
        raise MoeLoraError(rc, "moe_lora_router_get_error")
    return rc


def router_scratch(dims: Dims, device="cuda") -> torch.Tensor:
    n = moe_lora_workspace_bytes(dims, MOE_LORA_WS_ROUTER_SCRATCH)
    if n == 0:
        raise MoeLoraError(-5, "moe_lora_workspace_bytes(ROUTER_SCRATCH)")
    return torch.empty(n, dtype=torch.uint8, device=device)


def moe_lora_gemm_selftest(A: torch.Tensor, a_mn: bool, B: torch.Tensor, b_mn: bool, C: torch.Tensor,
                           stream=None) -> None:
    """C[M,N] = A(m,k) B(n,k) on the GEMM engine; A is [M,K] or, if a_mn, [K,M]; B is [N,K] or [K,N]."""
    M, N = C.shape
    K = A.shape[0] if a_mn else A.shape[1]
    rc = lib().moe_lora_gemm_selftest(M, N, K, _ptr(A, torch.bfloat16, "A"), int(a_mn),
                                      _ptr(B, torch.bfloat16, "B"), int(b_mn), _ptr(C, torch.float32, "C"),
                                      _stream(stream))
    _check(rc, "moe_lora_gemm_selftest")


def moe_lora_gemm_pair_selftest(A: torch.Tensor, a_mn: bool, B: torch.Tensor, b_mn: bool, C: torch.Tensor,
                                stream=None) -> None:
    """As moe_lora_gemm_selftest, on the two-SM (cta_group::2) engine."""
    M, N = C.shape
    K = A.shape[0] if a_mn else A.shape[1]
    rc = lib().moe_lora_gemm_pair_selftest(M, N, K, _ptr(A, torch.bfloat16, "A"), int(a_mn),
                                           _ptr(B, torch.bfloat16, "B"), int(b_mn), _ptr(C, torch.float32, "C"),
                                           _stream(stream))
    _check(rc, "moe_lora_gemm_pair_selftest")


def moe_lora_gemm_starved_selftest(A: torch.Tensor, a_mn: bool, B: torch.Tensor, b_mn: bool, C: torch.Tensor,
                                   pair: bool, stream=None) -> None:
    """The self-test GEMM with every operand copy withheld: its bounded waits must expire
    and set MOE_LORA_DEV_TIMEOUT (read with moe_lora_gemm_selftest_error)."""
    M, N = C.shape
    K = A.shape[0] if a_mn else A.shape[1]
    rc = lib().moe_lora_gemm_starved_selftest(M, N, K, _ptr(A, torch.bfloat16, "A"), int(a_mn),
                                              _ptr(B, torch.bfloat16, "B"), int(b_mn), _ptr(C, torch.float32, "C"),
                                              int(pair), _stream(stream))
    _check(rc, "moe_lora_gemm_starved_selftest")


def moe_lora_native_selftest(Aq: torch.Tensor, As: torch.Tensor, Bq: torch.Tensor, Bs: torch.Tensor,
                             C: torch.Tensor, layout: int = 0, stream=None) -> None:
    """Block-scaled FP4 self-test GEMM: C [M,N] fp32 from E4M3 codes Aq [M,K], packed
    E2M1 codes Bq [N,K/2] and UE8M0 scale bytes As, Bs in the tile-major layout
    [rows/128][K/128][128][4] (all uint8)."""
    M, K = Aq.shape
    N = Bq.shape[0]
    rc = lib().moe_lora_native_selftest(M, N, K, _ptr(Aq, torch.uint8, "Aq"), _ptr(As, torch.uint8, "As"),
                                        _ptr(Bq, torch.uint8, "Bq"), _ptr(Bs, torch.uint8, "Bs"),
                                        _ptr(C, torch.float32, "C"), int(layout), _stream(stream))
    _check(rc, "moe_lora_native_selftest")


def moe_lora_mxfp8_quantize(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    """MXFP8 (E4M3 codes, one UE8M0 scale byte per 32 along a row) of a bf16 matrix
    x [rows, n] into codes [rows, n] and scales [rows, n/32] (uint8, device)."""
    rows, n = x.shape
    rc = lib().moe_lora_mxfp8_quantize(_ptr(x, torch.bfloat16, "x"), rows, n, _ptr(codes, torch.uint8, "codes"),
                                       _ptr(scales, torch.uint8, "scales"), _stream(stream))
    _check(rc, "moe_lora_mxfp8_quantize")


def moe_lora_gemm_selftest_error(stream=None) -> int:
    return lib().moe_lora_gemm_selftest_error(_stream(stream))


def moe_lora_mxfp4_decode(packed: torch.Tensor, scales: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """MXFP4 (packed E2M1 pairs + one UE8M0 per 32) -> bf16 `out`, exactly, on the device."""
    elems = out.numel()
    if packed.numel() * 2 != elems or scales.numel() * 32 != elems:
        raise ValueError("packed must hold elems/2 bytes and scales elems/32 bytes")
    _check(lib().moe_lora_mxfp4_decode(_ptr(packed, torch.uint8, "packed"), _ptr(scales, torch.uint8, "scales"),
                                       _ptr(out, torch.bfloat16, "out"), elems, _stream(stream)),
           "moe_lora_mxfp4_decode")


def moe_lora_profile_enable(on: bool) -> None:
    lib().moe_lora_profile_enable(1 if on else 0)


def moe_lora_profile_select(kernel: Optional[str]) -> None:
    """Time only `kernel`'s launches (None: every kernel)."""
    rc = lib().moe_lora_profile_select(kernel.encode() if kernel is not None else None)
    _check(rc, "moe_lora_profile_select")


def moe_lora_profile_read() -> Dict[str, tuple]:
    """{kernel name: (total ms, launches)} since the last read (then reset)."""
    cap = 64
    names = (ctypes.c_char_p * cap)()
    ms = (ctypes.c_double * cap)()
    cnt = (ctypes.c_int64 * cap)()
    n = lib().moe_lora_profile_read(ctypes.cast(names, ctypes.c_void_p), ctypes.cast(ms, ctypes.c_void_p),
                                    ctypes.cast(cnt, ctypes.c_void_p), cap)
    if n < 0:
        raise MoeLoraError(n, "moe_lora_profile_read")
    return {names[i].decode(): (ms[i], int(cnt[i])) for i in range(n)}


def moe_lora_launch_count(reset: bool = False) -> int:
    return int(lib().moe_lora_launch_count(1 if reset else 0))


# ------------------------------------------------------------------ convenience
@dataclass
class Workspaces:
    """Device buffers for one problem size (allocated by torch, owned by the caller)."""
    plan: torch.Tensor
    saved: torch.Tensor
    fwd: torch.Tensor
    bwd: torch.Tensor

    @staticmethod
    def allocate(dims: Dims, device="cuda") -> "Workspaces":
        def buf(which):
            n = moe_lora_workspace_bytes(dims, which)
            if n == 0:
                raise MoeLoraError(-2, "moe_lora_workspace_bytes")
            return torch.empty(n, dtype=torch.uint8, device=device)
        return Workspaces(buf(MOE_LORA_WS_PLAN), buf(MOE_LORA_WS_SAVED), buf(MOE_LORA_WS_FWD_SCRATCH),
                          buf(MOE_LORA_WS_BWD_SCRATCH))


def alloc_grads(dims: Dims, device="cuda") -> Dict[str, torch.Tensor]:
    A, E, H, I, r = dims.A, dims.E, dims.H, dims.I, dims.r
    f = dict(dtype=torch.float32, device=device)
    return {"dA1": torch.empty(A, r, H, **f), "dA3": torch.empty(A, r, H, **f),
            "dB1": torch.empty(A, E, I, r, **f), "dB3": torch.empty(A, E, I, r, **f),
            "dA2": torch.empty(A, E, r, I, **f), "dB2": torch.empty(A, H, r, **f)}
