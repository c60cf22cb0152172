"""C-ABI checks that need no GPU: the library builds and loads, exports every
entry point include/moe_lora.h declares, sizes workspaces, and rejects bad calls
on the host before any launch (the pages' fail-fast rule: unsupported side-LoRA
placements and too-small scratch are refused before a kernel starts,
"feat(mega): add fused shared side-LoRA kernels", Summary)."""
import ctypes
import os
import re

import pytest
import torch

import moe_expert_ffn_top_gb300 as m
from moe_expert_ffn_top_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return m.lib()


def _declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"MOE_LORA_API\s+[\w\s\*]+?\b(moe_lora_\w+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n


def _dims(**kw):
    base = dict(T=256, H=512, I=256, E=16, k=2, r=16)
    base.update(kw)
    return m.make_dims(**base)


def test_workspace_sizes(L):
    d = _dims()
    sizes = [m.moe_lora_workspace_bytes(d, w) for w in range(4)]
    assert all(s > 0 for s in sizes)
    assert m.moe_lora_workspace_bytes(d, 9) == 0
    # production shape: bounded by T*k + E*(BM-1) rows
    p = m.make_dims(65536, 4096, 2048, 256, 6, 128)
    P = 65536 * 6 + 256 * 127
    assert m.moe_lora_workspace_bytes(p, m.MOE_LORA_WS_SAVED) >= 2 * P * (3 * 2048 + 256)
    for bad in (dict(H=500), dict(I=96), dict(H=32), dict(I=0), dict(r=12), dict(r=136), dict(k=0), dict(k=33), dict(E=0), dict(A=0)):
        assert m.moe_lora_workspace_bytes(_dims(**bad), 0) == 0, bad


FAKE = 1 << 20  # aligned, never dereferenced: every call below is rejected before any CUDA work


def _call_forward(L, d, **over):
    args = dict(plan=FAKE, x=FAKE, w=FAKE, y=FAKE, saved=FAKE, saved_bytes=1 << 40, scratch=FAKE,
                scratch_bytes=1 << 40)
    args.update(over)
    W = m.Weights(*([over.get("weight", FAKE)] * 9 + [over.get("scales")] * 3))
    if "w2" in over:
        W.W2 = over["w2"]
    return L.moe_lora_forward(ctypes.byref(d), args["plan"], args["x"], args["w"], ctypes.byref(W), args["y"],
                              args["saved"], args["saved_bytes"], args["scratch"], args["scratch_bytes"], None)


def test_forward_rejections(L):
    d = _dims()
    assert _call_forward(L, _dims(H=500)) == -2
    assert _call_forward(L, m.Dims(256, 512, 256, 16, 2, 16, 1, 128, 1.0, 2, 0)) == -5   # unknown activation
    assert _call_forward(L, m.Dims(256, 512, 256, 16, 2, 16, 1, 128, 1.0, 0, 0, -1.0)) == -2  # negative clamp
    assert _call_forward(L, m.Dims(256, 512, 256, 16, 2, 16, 1, 128, 1.0, 0, 5)) == -5   # unknown base format
    assert _call_forward(L, m.Dims(256, 576, 256, 16, 2, 16, 1, 128, 1.0, 0, 4)) == -2   # native + once: H % 128
    assert _call_forward(L, m.Dims(256, 576, 256, 16, 2, 16, 1, 128, 1.0, 0, 3)) == -2   # native: H % 128
    assert _call_forward(L, m.Dims(256, 512, 320, 16, 2, 16, 1, 128, 1.0, 0, 3)) == -2   # native: I % 128
    assert _call_forward(L, m.Dims(256, 512, 256, 16, 2, 16, 1, 128, 1.0, 0, 3), weight=FAKE + 16,
                         scales=FAKE) == -3                                            # native: W1/W3 32 B
    assert _call_forward(L, m.Dims(256, 512, 256, 16, 2, 16, 1, 128, 1.0, 0, 4), scales=FAKE,
                         w2=FAKE + 16) == -3                                           # native: W2 32 B
    assert _call_forward(L, m.Dims(256, 512, 256, 16, 2, 16, 1, 128, 1.0, 0, 1)) == -1   # MXFP4 without scales
    assert _call_forward(L, m.Dims(256, 512, 256, 16, 2, 16, 1, 64, 1.0, 0, 0)) == -2    # block_m != 128
    assert _call_forward(L, d, plan=None) == -1
    assert _call_forward(L, d, weight=FAKE + 8) == -3
    assert _call_forward(L, d, saved_bytes=16) == -4
    assert _call_forward(L, d, scratch_bytes=16) == -4
    assert _call_forward(L, d, x=FAKE + 2) == -3
    assert _call_forward(L, d, y=None) == -1


def test_plan_rejections(L):
    d = _dims()
    nbytes = m.moe_lora_workspace_bytes(d, 0)
    assert L.moe_lora_plan(ctypes.byref(d), FAKE, None, FAKE, nbytes - 1, None) == -4
    assert L.moe_lora_plan(ctypes.byref(d), None, None, FAKE, nbytes, None) == -1
    assert L.moe_lora_plan(ctypes.byref(d), FAKE, None, FAKE + 4, nbytes, None) == -3
    d2 = _dims(A=2)
    n2 = m.moe_lora_workspace_bytes(d2, 0)
    assert L.moe_lora_plan(ctypes.byref(d2), FAKE, None, FAKE, n2, None) == -1
    offs = (ctypes.c_int64 * 3)(0, 100, 256)        # adapter start not a multiple of 128
    assert L.moe_lora_plan(ctypes.byref(d2), FAKE, offs, FAKE, n2, None) == -2
    offs = (ctypes.c_int64 * 3)(0, 128, 200)        # does not end at T
    assert L.moe_lora_plan(ctypes.byref(d2), FAKE, offs, FAKE, n2, None) == -2


def test_backward_rejections(L):
    d = _dims()
    W = m.Weights(*([FAKE] * 9))
    G = m.Grads(*([FAKE] * 6))
    Gbad = m.Grads(*([FAKE] * 5 + [FAKE + 4]))
    bb = 1 << 40
    assert L.moe_lora_backward(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(W), FAKE, FAKE,
                               None, FAKE, bb, None) == -1
    assert L.moe_lora_backward(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(W), FAKE, FAKE,
                               ctypes.byref(Gbad), FAKE, bb, None) == -3
    assert L.moe_lora_backward(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(W), FAKE, FAKE,
                               ctypes.byref(G), FAKE, 100, None) == -4


def test_router_rejections(L):
    d = _dims()
    rb = m.moe_lora_workspace_bytes(d, m.MOE_LORA_WS_ROUTER_SCRATCH)
    assert rb >= 2 * 256 * 16
    # the router needs 16 <= E <= 256, E % 16 == 0
    for bad in (dict(E=8), dict(E=24), dict(E=272)):
        db = _dims(**bad)
        assert m.moe_lora_workspace_bytes(db, m.MOE_LORA_WS_ROUTER_SCRATCH) == 0, bad
        assert L.moe_lora_router_forward(ctypes.byref(db), FAKE, FAKE, None, FAKE, FAKE, None, FAKE, 1 << 40,
                                         None) == -5
    assert m.moe_lora_workspace_bytes(_dims(E=16, k=17), m.MOE_LORA_WS_ROUTER_SCRATCH) == 0
    dk = _dims(E=16, k=17)
    assert L.moe_lora_router_forward(ctypes.byref(dk), FAKE, FAKE, None, FAKE, FAKE, None, FAKE, 1 << 40, None) == -2
    f = L.moe_lora_router_forward
    assert f(ctypes.byref(d), FAKE, FAKE, None, FAKE, FAKE, None, FAKE, rb - 1, None) == -4
    assert f(ctypes.byref(d), None, FAKE, None, FAKE, FAKE, None, FAKE, rb, None) == -1
    assert f(ctypes.byref(d), FAKE, FAKE, None, FAKE + 4, FAKE, None, FAKE, rb, None) == -3
    assert f(ctypes.byref(d), FAKE, FAKE, None, FAKE, FAKE, FAKE + 8, FAKE, rb, None) == -3
    b = L.moe_lora_router_backward
    assert b(ctypes.byref(d), FAKE, FAKE, None, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, rb - 1, None) == -4
    assert b(ctypes.byref(d), FAKE, FAKE, None, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, rb, None) == -1
    assert b(ctypes.byref(d), FAKE, FAKE, None, FAKE, FAKE, FAKE, None, FAKE, FAKE + 2, FAKE, rb, None) == -3
    assert b(ctypes.byref(d), FAKE, FAKE, None, FAKE, FAKE, None, None, FAKE, FAKE, FAKE, rb, None) == -1
    assert L.moe_lora_router_get_error(None, None) == -1
    # several adapters (one router each): offsets required, with the plan's rules
    da = _dims(A=2, T=300)
    rba = m.moe_lora_workspace_bytes(da, m.MOE_LORA_WS_ROUTER_SCRATCH)
    assert rba > rb
    assert f(ctypes.byref(da), FAKE, FAKE, None, FAKE, FAKE, None, FAKE, rba, None) == -1
    for offs in ([0, 100, 300], [0, 256, 200], [0, 128, 299], [1, 128, 300]):
        o = (ctypes.c_int64 * 3)(*offs)
        assert f(ctypes.byref(da), FAKE, FAKE, o, FAKE, FAKE, None, FAKE, rba, None) == -2, offs
        assert b(ctypes.byref(da), FAKE, FAKE, o, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, rba, None) == -2, offs


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU answer")
def test_mxfp4_decode_rejections(L):
    """The decode entry point rejects bad sizes and pointers on the host; a zero-size
    call is a no-op that succeeds without a device."""
    assert L.moe_lora_mxfp4_decode(FAKE, FAKE, FAKE, 48, None) == -2        # not a multiple of 32
    assert L.moe_lora_mxfp4_decode(FAKE, FAKE, FAKE, -32, None) == -2
    assert L.moe_lora_mxfp4_decode(None, FAKE, FAKE, 64, None) == -1
    assert L.moe_lora_mxfp4_decode(FAKE, None, FAKE, 64, None) == -1
    assert L.moe_lora_mxfp4_decode(FAKE, FAKE, None, 64, None) == -1
    assert L.moe_lora_mxfp4_decode(FAKE + 4, FAKE, FAKE, 64, None) == -3    # packed not 16-byte aligned
    assert L.moe_lora_mxfp4_decode(FAKE, FAKE, FAKE + 2, 64, None) == -3    # out not 16-byte aligned
    assert L.moe_lora_mxfp4_decode(None, None, None, 0, None) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU answer")
def test_native_entry_rejections(L):
    """The MXFP8 quantiser and the block-scaled self-test GEMM reject bad sizes,
    pointers and layouts on the host."""
    assert L.moe_lora_mxfp8_quantize(FAKE, 4, 48, FAKE, FAKE, None) == -2      # n not a multiple of 32
    assert L.moe_lora_mxfp8_quantize(FAKE, -1, 64, FAKE, FAKE, None) == -2
    assert L.moe_lora_mxfp8_quantize(None, 4, 64, FAKE, FAKE, None) == -1
    assert L.moe_lora_mxfp8_quantize(FAKE, 4, 64, FAKE, None, None) == -1
    assert L.moe_lora_mxfp8_quantize(FAKE, 4, 64, FAKE + 8, FAKE, None) == -3
    assert L.moe_lora_mxfp8_quantize(None, 0, 64, None, None, None) == 0       # no rows: no-op
    assert L.moe_lora_mxfp8_quantize(FAKE, 4, 64, FAKE, FAKE, None) == -7      # no device
    ok = (256, 512, 256, FAKE, FAKE, FAKE, FAKE, FAKE)
    assert L.moe_lora_native_selftest(100, 512, 256, *ok[3:], 0, None) == -2   # M % 128
    assert L.moe_lora_native_selftest(256, 384, 256, *ok[3:], 0, None) == -2   # N % 256
    assert L.moe_lora_native_selftest(256, 512, 192, *ok[3:], 0, None) == -2   # K % 128
    assert L.moe_lora_native_selftest(*ok, 3, None) == -5                     # unknown layout
    assert L.moe_lora_native_selftest(256, 512, 256, FAKE, FAKE, FAKE + 16, FAKE, FAKE, 0, None) == -3  # Bq 32 B
    assert L.moe_lora_native_selftest(*ok, 0, None) == -7


def test_no_device_is_reported(L):
    d = _dims()
    nbytes = m.moe_lora_workspace_bytes(d, 0)
    assert L.moe_lora_plan(ctypes.byref(d), FAKE, None, FAKE, nbytes, None) == -7
    assert L.moe_lora_mxfp4_decode(FAKE, FAKE, FAKE, 64, None) == -7


def test_strerror(L):
    for c in range(-7, 1):
        assert m.moe_lora_strerror(c) and m.moe_lora_strerror(c) != "unknown error"
