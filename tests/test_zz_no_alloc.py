"""moe_lora_plan_noalloc: the routing plan for callers that cannot allocate.

Some callers may not call cudaMalloc (or any allocator) while they route tokens:
memory-planned serving runtimes that reserve all device memory up front and hand
out only pre-reserved buffers, and C hosts without an allocator binding of their
own.  This entry point serves them: its temporary histograms live in a fixed
array inside the library instead of in caller-provided workspace.  These checks
run it through the C ABI and compare it with moe_lora_plan() on the same inputs,
on consecutive calls whose stale scratch contents differ, drive a forward and
backward from its plan twice in a row, and check the size-limit rejection.  The
file is collected last, so a run that stops at the first failure has already run
every other test.
"""
import pytest
import torch

import moe_expert_ffn_top_gb300 as m
from synth import Shape, make_inputs

from gpu_common import ADAPTER_GRADS, run_gpu

pytestmark = pytest.mark.gpu

PLAN_FIELDS = ("counts", "offsets", "row_of_route", "route_of_row")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_ffn_top_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield


def _plan_only_bytes(d):
    """Bytes of the plan itself: the full plan workspace minus its histogram area."""
    full = m.moe_lora_workspace_bytes(d, m.MOE_LORA_WS_PLAN)
    nchunks = (d.T * d.k + 1023) // 1024
    hist = 4 * d.A * d.E * max(nchunks, 1)
    return full - (hist + 255) // 256 * 256


def _ids(T, k, E, mask, seed):
    g = torch.Generator().manual_seed(seed)
    ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    ids[torch.rand(T, k, generator=g) < mask] = -1
    return ids.cuda()


def _reference_plan(d, ids, offs):
    ws = torch.empty(m.moe_lora_workspace_bytes(d, m.MOE_LORA_WS_PLAN), dtype=torch.uint8, device="cuda")
    m.moe_lora_plan(d, ids, offs, ws)
    return m.moe_lora_plan_readback(d, ws)


@pytest.mark.parametrize("cases", [
    [(5000, 6, 256, 1, 0.2), (300, 2, 16, 1, 0.0)],       # large then small: stale histograms stay behind
    [(64, 8, 32, 1, 0.5), (4096, 6, 256, 1, 0.2)],
    [(16 * 128, 4, 32, 16, 0.1), (1, 1, 4, 1, 0.0)],      # several adapters, then a single token
])
def test_noalloc_plan_matches_plan_on_consecutive_calls(cases):
    for i, (T, k, E, A, mask) in enumerate(cases):
        d = m.make_dims(T, 256, 256, E, k, 8, A)
        ids = _ids(T, k, E, mask, seed=100 + i)
        offs = list(range(0, T + 1, T // A)) if A > 1 else None
        want = _reference_plan(d, ids, offs)
        n = _plan_only_bytes(d)
        ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
        m.moe_lora_plan_noalloc(d, ids, offs, ws)
        torch.cuda.synchronize()
        got = m.moe_lora_plan_readback(d, ws)
        assert m.moe_lora_get_error(d, ws) == 0
        for f in PLAN_FIELDS:
            assert torch.equal(got[f], want[f]), (i, f)


def test_noalloc_plan_drives_forward_backward_identically():
    shp = Shape(T=200, H=512, I=256, E=16, k=2, r=16, mask_frac=0.2)
    inp = make_inputs(shp, seed=21)
    ref = run_gpu(inp, shp)
    d = ref["dims"]
    ws = m.Workspaces.allocate(d)
    dev = {n: v.cuda() for n, v in inp.items() if n != "adapter_offsets"}
    for _ in range(2):  # two calls in a row
        m.moe_lora_plan_noalloc(d, dev["topk_ids"], None, ws.plan, _plan_only_bytes(d))
        y = torch.empty(shp.T, shp.H, dtype=torch.bfloat16, device="cuda")
        m.moe_lora_forward(d, ws.plan, dev["x"], dev["topk_w"], dev, y, ws.saved, ws.fwd)
        dx = torch.empty_like(y)
        dw = torch.empty(shp.T, shp.k, dtype=torch.float32, device="cuda")
        g = m.alloc_grads(d)
        m.moe_lora_backward(d, ws.plan, ws.saved, dev["x"], dev["topk_w"], dev["dy"], dev, dx, dw, g, ws.bwd)
        torch.cuda.synchronize()
        assert torch.equal(y, ref["y"]) and torch.equal(dx, ref["dx"]) and torch.equal(dw, ref["dw"])
        for n in ADAPTER_GRADS:
            assert torch.equal(g[n], ref[n]), n


def test_noalloc_plan_rejects_sizes_beyond_its_scratch():
    ids = torch.zeros(8, dtype=torch.int32, device="cuda")
    d = m.make_dims(76800, 256, 256, 2048, 8, 8)       # 2048 groups x 600 chunks > 1,048,576
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.MoeLoraError) as e:
        m.moe_lora_plan_noalloc(d, ids, None, ws, 1 << 40)
    assert e.value.code == -8
    d = m.make_dims(256, 256, 256, 16, 2, 8)
    with pytest.raises(m.MoeLoraError) as e:
        m.moe_lora_plan_noalloc(d, ids, None, ws, _plan_only_bytes(d) - 1)
    assert e.value.code == -4
