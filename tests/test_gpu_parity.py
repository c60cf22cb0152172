"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars: routing plan bit-exact; BF16 outputs and every gradient within relative L2
5e-3 and cosine 0.9999 (FP64 metrics over whole tensors), the accuracy gate the
side-LoRA pages use ("feat(mega): add fused shared side-LoRA kernels", Accuracy
and regression tests / Correctness coverage).  Inputs are seeded and synthetic
(synth.make_inputs); expected values come only from the oracle.
"""
import os

import pytest
import torch

import moe_expert_ffn_top_gb300 as m
import oracle
from synth import EDGE_TOKEN_COUNTS, Shape, make_inputs, shape

from gpu_common import (ADAPTER_GRADS, _full_check, _sampled_check, _sparse_dy, assert_close, dims_of, rel_l2,
                        run_gpu, sub_problem)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_ffn_top_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield


# ----------------------------------------------------------------------------- engine
@pytest.mark.parametrize("a_mn", [False, True])
@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 320), (128, 16, 128), (384, 144, 192)])
def test_engine_gemm(a_mn, b_mn, M, N, K):
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N + K)
    A = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    B = torch.randn(N, K, generator=g, device="cuda").to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), device="cuda")
    m.moe_lora_gemm_selftest(A.t().contiguous() if a_mn else A, a_mn, B.t().contiguous() if b_mn else B, b_mn, C)
    torch.cuda.synchronize()
    assert m.moe_lora_gemm_selftest_error() == 0
    ref = A.double() @ B.double().t()
    assert rel_l2(C, ref) < 1e-5


@pytest.mark.parametrize("a_mn", [False, True])
@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (384, 512, 320), (128, 16, 128), (640, 144, 192),
                                   (2432, 768, 1024)])
def test_engine_gemm_pair(a_mn, b_mn, M, N, K):
    """The two-SM engine: 256-row tiles shared by a CTA pair, including an odd last
    128-row tile (M = 128, 384, 640) and more tiles than clusters (M = 2432)."""
    g = torch.Generator(device="cuda").manual_seed(M * 5 + N + K)
    A = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    B = torch.randn(N, K, generator=g, device="cuda").to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), device="cuda")
    m.moe_lora_gemm_pair_selftest(A.t().contiguous() if a_mn else A, a_mn, B.t().contiguous() if b_mn else B, b_mn,
                                  C)
    torch.cuda.synchronize()
    assert m.moe_lora_gemm_selftest_error() == 0
    ref = A.double() @ B.double().t()
    assert rel_l2(C, ref) < 1e-5


@pytest.mark.parametrize("pair", [False, True])
def test_engine_wait_timeout_reports_and_recovers(pair):
    """Failure detection without a GPU fault: with every operand copy withheld (as if
    a copy were lost) the engine's bounded waits expire, the kernel ends with
    MOE_LORA_DEV_TIMEOUT in the error word the host reads, and the context stays
    usable for the next launch."""
    M, N, K = (256, 256, 128) if pair else (128, 256, 128)
    g = torch.Generator(device="cuda").manual_seed(7)
    A = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    B = torch.randn(N, K, generator=g, device="cuda").to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), device="cuda")
    assert m.moe_lora_gemm_selftest_error() == 0
    m.moe_lora_gemm_starved_selftest(A, False, B, False, C, pair)
    torch.cuda.synchronize()
    assert m.moe_lora_gemm_selftest_error() & m.MOE_LORA_DEV_TIMEOUT
    assert torch.isnan(C).all()  # the epilogue never ran
    run = m.moe_lora_gemm_pair_selftest if pair else m.moe_lora_gemm_selftest
    run(A, False, B, False, C)
    torch.cuda.synchronize()
    assert m.moe_lora_gemm_selftest_error() == 0
    assert rel_l2(C, A.double() @ B.double().t()) < 1e-5


# ----------------------------------------------------------------------------- plan
def _plan_check(ids_cpu, E, shp, offs=None, BM=128):
    d = m.make_dims(shp.T, shp.H, shp.I, E, shp.k, shp.r, shp.A)
    ws = m.Workspaces.allocate(d)
    m.moe_lora_plan(d, ids_cpu.cuda(), offs, ws.plan)
    got = m.moe_lora_plan_readback(d, ws.plan)
    want = oracle.plan(ids_cpu, E, torch.tensor(offs if offs else [0, shp.T]), BM)
    for n in ("counts", "offsets", "row_of_route", "route_of_row"):
        assert torch.equal(got[n], want[n]), n
    return d, ws, want


@pytest.mark.parametrize("T,k,E,mask,seed", [(1, 1, 4, 0.0, 0), (256, 2, 16, 0.0, 1), (1000, 6, 256, 0.2, 2),
                                             (5000, 8, 128, 0.3, 3), (2048, 6, 256, 0.2, 4)])
def test_plan_bit_exact(T, k, E, mask, seed):
    g = torch.Generator().manual_seed(seed)
    ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    ids[torch.rand(T, k, generator=g) < mask] = -1
    ids[:, 0][ids[:, 0] == 3] = -1
    shp = Shape(T=T, H=256, I=256, E=E, k=k, r=8)
    _plan_check(ids, E, shp)


def test_plan_multi_adapter_bit_exact():
    T, k, E, A = 16 * 128, 4, 32, 16
    g = torch.Generator().manual_seed(11)
    ids = torch.randint(-1, E, (T, k), generator=g, dtype=torch.int32)
    shp = Shape(T=T, H=256, I=256, E=E, k=k, r=8, A=A)
    _plan_check(ids, E, shp, offs=list(range(0, T + 1, 128)))


def test_plan_bad_ids_flagged_and_dropped():
    ids = torch.tensor([[0, 7], [-3, 1], [2, -1]], dtype=torch.int32)
    shp = Shape(T=3, H=256, I=256, E=4, k=2, r=8)
    d = m.make_dims(3, 256, 256, 4, 2, 8)
    ws = m.Workspaces.allocate(d)
    m.moe_lora_plan(d, ids.cuda(), None, ws.plan)
    got = m.moe_lora_plan_readback(d, ws.plan)
    assert m.moe_lora_get_error(d, ws.plan) & m.MOE_LORA_DEV_BAD_ID
    want = oracle.plan(ids, 4, torch.tensor([0, 3]), 128)
    assert torch.equal(got["row_of_route"], want["row_of_route"])


# ----------------------------------------------------------------------------- full path
@pytest.mark.parametrize("T,mask", [(256, 0.0), (200, 0.15), (17, 0.0)])
def test_tiny_forward_backward(T, mask):
    shp = Shape(T=T, H=512, I=256, E=16, k=2, r=16, mask_frac=mask)
    inp = make_inputs(shp, seed=0)
    out = run_gpu(inp, shp)
    assert out["err"] == 0
    _full_check(inp, shp, out)


@pytest.mark.parametrize("r", [24, 40, 64, 72, 120])
def test_ranks_off_the_tile_boundaries(r):
    """Ranks that are not multiples of 16, 32 or 64 (and 64 itself): partial MMA N
    widths, zero-filled TMA boxes and partial store chunks on every side path."""
    shp = Shape(T=150, H=512, I=256, E=8, k=2, r=r, mask_frac=0.1, scale=0.5)
    inp = make_inputs(shp, seed=40 + r)
    out = run_gpu(inp, shp, poison=True)
    assert out["err"] == 0
    _full_check(inp, shp, out)


@pytest.mark.parametrize("H,I", [(576, 320), (192, 64), (320, 448)])
def test_widths_off_the_tile_boundaries(H, I):
    """H and I multiples of 64 but not of the 128- and 256-wide tiles: a last W13
    column tile with 64 of its 128 columns (I % 128 = 64), last W2 / W13-dgrad /
    expand column tiles with 64 or 192 of 256 (H % 256), last dB2 row tiles with 64
    of 128 rows (H % 128 = 64), last dB1/dB3 row tiles (I % 128 = 64), last W2-dgrad
    and dA2 column tiles with 64 or 192 of 256 (I % 256); NaN-poisoned workspaces
    and outputs, so nothing past an edge can leak."""
    shp = Shape(T=300, H=H, I=I, E=8, k=2, r=24, mask_frac=0.1)
    inp = make_inputs(shp, seed=60 + H + I)
    out = run_gpu(inp, shp, poison=True)
    assert out["err"] == 0
    _full_check(inp, shp, out)


def test_saturated_gates():
    """x scaled by 64: gate pre-activations reach the hundreds, so silu sits at its
    limits (exp(-z) overflows to inf for z < -88, giving 0; z for large z) in the
    forward, the saved activation and the backward's sigmoid; all finite and within
    tolerance of the oracle."""
    shp = Shape(T=256, H=512, I=256, E=16, k=2, r=16)
    inp = make_inputs(shp, seed=21)
    inp["x"] = (inp["x"].float() * 64).to(torch.bfloat16)
    out = run_gpu(inp, shp)
    assert out["err"] == 0
    g = inp["x"].float() @ inp["W1"][0].float().t()
    assert (g < -88).float().mean() > 0.05  # the overflow branch is exercised
    _full_check(inp, shp, out)


def test_small_rank8_top8():
    shp = Shape(T=300, H=256, I=512, E=8, k=8, r=8, scale=0.5)
    inp = make_inputs(shp, seed=5)
    out = run_gpu(inp, shp)
    assert out["err"] == 0
    _full_check(inp, shp, out)


def test_rank128_wide():
    shp = Shape(T=130, H=1024, I=512, E=8, k=3, r=128, mask_frac=0.2, empty_experts=(0, 7))
    inp = make_inputs(shp, seed=6)
    out = run_gpu(inp, shp)
    assert out["err"] == 0
    _full_check(inp, shp, out)
    for n in ("dB1", "dB3", "dA2"):
        assert out[n][0, 0].abs().max().item() == 0 and out[n][0, 7].abs().max().item() == 0


def test_large_groups_row_chunks():
    """Groups far larger than one row chunk of the column-tile-major tile order (2,048
    rows): 7,000 tokens, top-2 over 3 experts (~4,700 rows each: two full chunks and a
    ragged one, 16 row tiles of 128 per chunk, 8 of 256 for the W13 dgrad), NaN-poisoned
    workspaces, checked against the oracle on sampled tokens of every expert."""
    shp = Shape(T=7000, H=1024, I=512, E=3, k=2, r=16)
    inp = make_inputs(shp, seed=21, device="cuda")
    sample = [0, 1, 2047, 2048, 2049, 3001, 4095, 4096, 5998, 6999]
    inp = _sparse_dy(inp, shp, sample)
    out = run_gpu(inp, shp, poison=True)
    assert out["err"] == 0
    counts = m.moe_lora_plan_readback(out["dims"], out["ws"].plan)["counts"]
    assert int(counts.max()) > 2 * 2048
    for n in ("y", "dx", "dw"):
        assert torch.isfinite(out[n]).all(), n
    _sampled_check(inp, shp, out, sample)


def test_zero_scale_is_plain_moe_bitwise():
    """Zero adapter scale reproduces the layer without side adapters bit for bit
    (the pages' zero-scale preservation check)."""
    shp = Shape(T=256, H=512, I=256, E=16, k=2, r=16)
    inp = make_inputs(shp, seed=7)
    out0 = run_gpu(inp, shp, scale=0.0)
    bare = dict(inp)
    for n in ("A1", "A3", "B1", "B3", "A2", "B2"):
        bare[n] = torch.zeros_like(inp[n])
    outp = run_gpu(bare, shp, scale=1.0)
    for n in ("y", "dx", "dw"):
        assert torch.equal(out0[n], outp[n]), n
    y_ref = oracle.forward(inp, shp, scale=0.0)
    assert_close("y(s=0)", out0["y"].cpu(), y_ref)


def test_deterministic_and_poison_free():
    """Two runs are bitwise identical, also with every workspace and output
    pre-filled with NaN (padding rows and stale scratch never leak)."""
    shp = Shape(T=200, H=512, I=256, E=16, k=2, r=16, mask_frac=0.2)
    inp = make_inputs(shp, seed=8)
    a = run_gpu(inp, shp)
    b = run_gpu(inp, shp, poison=True)
    for n in ("y", "dx", "dw") + ADAPTER_GRADS:
        assert torch.equal(a[n], b[n]), n


def test_empty_batch():
    shp = Shape(T=0, H=512, I=256, E=16, k=2, r=16)
    d = dims_of(shp)
    ws = m.Workspaces.allocate(d)
    ids = torch.empty(0, 2, dtype=torch.int32, device="cuda")
    m.moe_lora_plan(d, ids, None, ws.plan)
    g = m.alloc_grads(d)
    for t in g.values():
        t.fill_(float("nan"))
    e = torch.empty(0, device="cuda")
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    inp = make_inputs(Shape(T=1, H=512, I=256, E=16, k=2, r=16), seed=0)
    wts = {n: inp[n].cuda() for n in ("W1", "W3", "W2", "A1", "A3", "B1", "B3", "A2", "B2")}
    m.moe_lora_backward(d, ws.plan, ws.saved, x, e, x, wts, x, e, g, ws.bwd)
    torch.cuda.synchronize()
    for n, t in g.items():
        assert t.abs().max().item() == 0, n


def test_all_routes_masked():
    """Every route masked (ids all -1): no routed rows (P = 0, the grouped GEMMs have no
    tiles) while the per-token kernels still run; y, dx, dw and all six adapter
    gradients are exactly zero, and the oracle agrees."""
    shp = Shape(T=200, H=512, I=256, E=16, k=2, r=16)
    inp = make_inputs(shp, seed=31)
    inp["topk_ids"] = torch.full_like(inp["topk_ids"], -1)
    out = run_gpu(inp, shp, poison=True)
    assert out["err"] == 0
    got = m.moe_lora_plan_readback(out["dims"], out["ws"].plan)
    assert int(got["offsets"][-1]) == 0 and int(got["counts"].sum()) == 0
    for n in ("y", "dx", "dw") + ADAPTER_GRADS:
        assert out[n].abs().max().item() == 0, n
    y_ref = oracle.forward(inp, shp)
    assert y_ref.abs().max().item() == 0


# ----------------------------------------------------------------------------- production width
@pytest.mark.parametrize("T", EDGE_TOKEN_COUNTS)
def test_edge_sweep_production_width(T):
    """H=4096, I=2048, E=256, top-6, rank 128, a fifth of the routes masked, experts 0/127/255
    empty, at the 15 token counts of the pages' boundary sweep."""
    shp = shape("edge", T)
    inp = make_inputs(shp, seed=1000 + T, device="cuda")
    g = torch.Generator().manual_seed(T)
    # 6 sampled tokens (<= 36 experts' weights copied to the host per case): the sweep
    # churns far less host memory, which otherwise leaves the host compacting memory
    # (and stalling pinned copies) for minutes after the suite
    n = min(T, 6)
    sample = sorted(torch.randperm(T, generator=g)[:n].tolist())
    inp = _sparse_dy(inp, shp, sample)
    out = run_gpu(inp, shp)
    assert out["err"] == 0
    want = oracle.plan(inp["topk_ids"].cpu(), shp.E, torch.tensor([0, T]), 128)
    got = m.moe_lora_plan_readback(out["dims"], out["ws"].plan)
    for k in ("counts", "offsets", "row_of_route", "route_of_row"):
        assert torch.equal(got[k], want[k]), k
    _sampled_check(inp, shp, out, sample)


def _tile_sample(plan, k, per_kind=8, seed=0):
    """Tokens chosen from the plan so that the sample's routed rows land in (a) the
    second 128-row half of a 256-row tile (the wide GEMMs' second MMA and epilogue
    half), (b) the last, partly padded 128-row tile of a group of two or more tiles,
    (c) a group's first tile; `per_kind` tokens of each kind, each through an expert
    no earlier pick used where possible.  Returns (sorted tokens, experts covered)."""
    offs = plan["offsets"].long()
    counts = plan["counts"].long()
    ror = plan["row_of_route"].long()
    live = (ror >= 0).nonzero().flatten()
    rows = ror[live]
    grp = torch.searchsorted(offs, rows, right=True) - 1
    tile = (rows - offs[grp]) // 128
    ntile = (counts[grp] + 127) // 128
    kinds = [tile % 2 == 1, (tile == ntile - 1) & (counts[grp] % 128 != 0) & (ntile >= 2), tile == 0]
    g = torch.Generator().manual_seed(seed)
    chosen, experts = [], set()
    for sel in kinds:
        pos = sel.nonzero().flatten()
        pos = pos[torch.randperm(pos.numel(), generator=g)]
        picked = 0
        for fresh_only in (True, False):
            for i in pos.tolist():
                if picked == per_kind:
                    break
                t, e = int(live[i]) // k, int(grp[i])
                if t in chosen or (fresh_only and e in experts):
                    continue
                chosen.append(t)
                experts.add(e)
                picked += 1
        assert picked == per_kind, "too few candidate rows of one kind"
    return sorted(chosen), experts


def _chunked_sampled_check(inp, shp, out, sample, chunk=4):
    """_sampled_check for larger samples: the oracle runs on sub-problems of `chunk`
    tokens (a few experts' weights on the host at a time).  dy is zero outside the
    sample, and every gradient is linear in dy, so the adapter gradients of the
    whole sample are the sums of the chunks' gradients; y, dx and dw are per token."""
    E = shp.E
    tot = {n: None for n in ("dA1", "dA3", "dB2")}
    per_e = {n: {} for n in ("dB1", "dB3", "dA2")}
    ys, dxs, dws = [], [], []
    for c0 in range(0, len(sample), chunk):
        sub, sshp, used, tok = sub_problem(inp, shp, sample[c0:c0 + chunk])
        y_ref = oracle.forward(sub, sshp)
        g_ref = oracle.backward(sub, sshp)
        ys.append((tok, y_ref))
        dxs.append((tok, g_ref["dx"]))
        dws.append((tok, g_ref["dw"]))
        for n in tot:
            tot[n] = g_ref[n] if tot[n] is None else tot[n] + g_ref[n]
        for n in per_e:
            for i, e in enumerate(used):
                v = g_ref[n][:, i]
                per_e[n][e] = v if e not in per_e[n] else per_e[n][e] + v
    for name, parts, got in (("y", ys, out["y"]), ("dx", dxs, out["dx"]), ("dw", dws, out["dw"])):
        tk = torch.cat([t for t, _ in parts])
        assert_close(name, got[tk.cuda()].cpu(), torch.cat([v for _, v in parts]))
    mask = torch.ones(shp.T, dtype=torch.bool, device="cuda")
    mask[torch.as_tensor(sample, device="cuda")] = False
    assert out["dx"][mask].abs().max().item() == 0 and out["dw"][mask].abs().max().item() == 0
    for n in tot:
        assert_close(n, out[n].cpu(), tot[n])
    ex = sorted(per_e["dB1"])
    exd = torch.as_tensor(ex, device="cuda")
    for n in per_e:
        assert_close(n, out[n][:, exd].cpu(), torch.stack([per_e[n][e] for e in ex], dim=1))
        other = torch.ones(E, dtype=torch.bool, device="cuda")
        other[exd] = False
        if other.any():
            assert out[n][:, other].abs().max().item() == 0, n


@pytest.mark.slow
def test_production_shape_sampled():
    """65,536 tokens, H=4096, I=2048, E=256, top-6, rank 128: the benchmark's
    workload and launch configuration.  The plan is read back first; 24 tokens are
    chosen so that their routed rows land in second 128-row halves of 256-row
    tiles, in groups' last (padded) tiles and in groups' first tiles, across many
    experts, and the result is checked on them (sparse dy)."""
    shp = shape("prod")
    inp = make_inputs(shp, seed=2, device="cuda")
    d = dims_of(shp)
    ws = m.Workspaces.allocate(d)
    m.moe_lora_plan(d, inp["topk_ids"], None, ws.plan)
    got = m.moe_lora_plan_readback(d, ws.plan)
    want = oracle.plan(inp["topk_ids"].cpu(), shp.E, torch.tensor([0, shp.T]), 128)
    for k in ("counts", "offsets", "row_of_route", "route_of_row"):
        assert torch.equal(got[k], want[k]), k
    sample, experts = _tile_sample(got, shp.k, per_kind=8, seed=2)
    assert len(sample) >= 24 and len(experts) >= 8
    inp = _sparse_dy(inp, shp, sample)
    out = run_gpu(inp, shp, ws=ws)
    assert out["err"] == 0
    _chunked_sampled_check(inp, shp, out, sample)


@pytest.mark.parametrize("k,T", [(1, 65536), (2, 32768)])
def test_topk_small_production_width(k, T):
    """Top-k 1 and 2 (the pages' top-k 1/2/6 coverage) at production widths: H=4096,
    I=2048, E=256, rank 128, a fifth of the routes masked, experts 0/127/255 empty;
    ~200 rows per expert, so groups of two 128-row tiles (one full 256-row tile with a
    padded second half).  Plan bit-exact; 24 plan-chosen tokens checked against the
    oracle (sparse dy)."""
    shp = Shape(T=T, H=4096, I=2048, E=256, k=k, r=128, mask_frac=0.2, empty_experts=(0, 127, 255))
    inp = make_inputs(shp, seed=50 + k, device="cuda")
    d = dims_of(shp)
    ws = m.Workspaces.allocate(d)
    m.moe_lora_plan(d, inp["topk_ids"], None, ws.plan)
    got = m.moe_lora_plan_readback(d, ws.plan)
    want = oracle.plan(inp["topk_ids"].cpu(), shp.E, torch.tensor([0, shp.T]), 128)
    for n in ("counts", "offsets", "row_of_route", "route_of_row"):
        assert torch.equal(got[n], want[n]), n
    assert int(got["counts"][0]) == int(got["counts"][127]) == int(got["counts"][255]) == 0
    sample, experts = _tile_sample(got, k, per_kind=8, seed=k)
    assert len(sample) >= 24 and len(experts) >= 8
    inp = _sparse_dy(inp, shp, sample)
    out = run_gpu(inp, shp, ws=ws)
    assert out["err"] == 0
    _chunked_sampled_check(inp, shp, out, sample)


# ----------------------------------------------------------------------------- several adapters
def _adapter_slice(inp, shp, a):
    """Adapter a's standalone problem: its tokens and its factors, one adapter."""
    per = shp.T // shp.A
    sl = slice(a * per, (a + 1) * per)
    sub = {n: inp[n][sl] for n in ("x", "dy", "topk_ids", "topk_w")}
    for n in ("W1", "W3", "W2"):
        sub[n] = inp[n]
    for n in ("A1", "A3", "B1", "B3", "A2", "B2"):
        sub[n] = inp[n][a:a + 1].contiguous()
    sub["adapter_offsets"] = torch.tensor([0, per], dtype=torch.int64)
    return sub, Shape(T=per, H=shp.H, I=shp.I, E=shp.E, k=shp.k, r=shp.r, A=1, scale=shp.scale), sl


def test_multi_adapter_fused_equals_standalone_bitwise():
    """16 adapters (rank 8) share one layer, each with its own routing; every
    adapter's outputs and gradients from the fused pass equal its standalone
    single-adapter run bit for bit (OpenPipe/ART PR #1139, Validation)."""
    shp = shape("multi")
    inp = make_inputs(shp, seed=4, device="cuda")
    fused = run_gpu(inp, shp)
    assert fused["err"] == 0
    for a in (0, 7, 15):
        sub, sshp, sl = _adapter_slice(inp, shp, a)
        alone = run_gpu(sub, sshp)
        for n in ("y", "dx", "dw"):
            assert torch.equal(fused[n][sl], alone[n]), (a, n)
        for n in ADAPTER_GRADS:
            assert torch.equal(fused[n][a:a + 1], alone[n]), (a, n)


def test_multi_adapter_sampled_oracle():
    """Fused multi-adapter pass against the oracle: dy is non-zero only on tokens
    of adapter 3, so adapter 3's gradients come from that sample alone and every
    other adapter's gradients are exactly zero."""
    shp = shape("multi")
    inp = make_inputs(shp, seed=5, device="cuda")
    a, per = 3, shp.T // shp.A
    sample = [a * per + t for t in (0, 1, 100, 511, 777, 1023)]
    inp = _sparse_dy(inp, shp, sample)
    out = run_gpu(inp, shp)
    assert out["err"] == 0
    one, oshp, sl = _adapter_slice(inp, shp, a)
    local = [t - a * per for t in sample]
    sub, sshp, used, tok = sub_problem(one, oshp, local)
    y_ref = oracle.forward(sub, sshp)
    g_ref = oracle.backward(sub, sshp)
    gt = (tok + a * per).cuda()
    assert_close("y", out["y"][gt].cpu(), y_ref)
    assert_close("dx", out["dx"][gt].cpu(), g_ref["dx"])
    assert_close("dw", out["dw"][gt].cpu(), g_ref["dw"])
    ex = torch.as_tensor(used, device="cuda")
    for n in ("dA1", "dA3", "dB2"):
        assert_close(n, out[n][a:a + 1].cpu(), g_ref[n])
    for n in ("dB1", "dB3", "dA2"):
        assert_close(n, out[n][a:a + 1, ex].cpu(), g_ref[n])
    others = [b for b in range(shp.A) if b != a]
    for n in ADAPTER_GRADS:
        assert out[n][others].abs().max().item() == 0, n


# ----------------------------------------------------------------------------- MXFP4 base
def _decode_mxfp4_golden(packed, scales):
    """bf16 values of an MXFP4 tensor from the OCP table in tests/golden (host)."""
    rows = [l.split() for l in open(os.path.join(os.path.dirname(__file__), "golden", "e2m1_ue8m0.txt"))
            if l.strip() and l[0] != "#"]
    table = torch.tensor([float(v) for kd, c, v in rows if kd == "e2m1"], dtype=torch.float64)
    p = packed.cpu()
    codes = torch.stack([(p & 15).long(), (p >> 4).long()], dim=-1).reshape(*p.shape[:-1], p.shape[-1] * 2)
    sc = torch.exp2(scales.cpu().double() - 127).repeat_interleave(32, dim=-1)
    return (table[codes] * sc).to(torch.bfloat16)


def test_mxfp4_decode_every_code_and_scale():
    """The decode kernel on all 256 packed bytes (every pair of E2M1 codes, -0 included)
    under scale bytes from the subnormal 2^-127 to overflow, against the OCP table,
    bit for bit; scale byte 255 decodes to NaN."""
    scale_bytes = [0, 1, 2, 60, 120, 126, 127, 128, 129, 200, 253, 254]
    packed = torch.arange(256, dtype=torch.uint8).repeat(len(scale_bytes))  # 16 groups per scale
    scales = torch.tensor(scale_bytes, dtype=torch.uint8).repeat_interleave(16)
    want = _decode_mxfp4_golden(packed.view(1, -1), scales.view(1, -1)).view(-1)
    got = torch.empty(packed.numel() * 2, dtype=torch.bfloat16, device="cuda")
    m.moe_lora_mxfp4_decode(packed.cuda(), scales.cuda(), got)
    torch.cuda.synchronize()
    assert torch.equal(got.cpu().view(torch.int16), want.view(torch.int16))
    nan = torch.empty(64, dtype=torch.bfloat16, device="cuda")
    m.moe_lora_mxfp4_decode(torch.arange(32, dtype=torch.uint8).cuda(), torch.full((2,), 255, dtype=torch.uint8).cuda(),
                            nan)
    torch.cuda.synchronize()
    assert torch.isnan(nan.float()).all()


def test_mxfp4_tiny_forward_backward():
    shp = Shape(T=200, H=512, I=256, E=16, k=2, r=16, mask_frac=0.1, base_fmt="mxfp4")
    inp = make_inputs(shp, seed=31)
    out = run_gpu(inp, shp)
    assert out["err"] == 0
    _full_check(inp, shp, out)


@pytest.mark.parametrize("mx_once", [False, True])
def test_mxfp4_equals_decoded_bf16_base_bitwise(mx_once):
    """An MXFP4 base gives bit for bit what the same layer gives with the decoded
    values as a bf16 base (the decode is exact), decoded inside the GEMMs or once per
    pass."""
    shp = Shape(T=256, H=512, I=256, E=16, k=2, r=16, base_fmt="mxfp4")
    inp = make_inputs(shp, seed=32)
    q = run_gpu(inp, shp, mx_once=mx_once)
    deq = {n: v for n, v in inp.items() if n not in ("S1", "S3", "S2")}
    for n in ("W1", "W3", "W2"):
        deq[n] = _decode_mxfp4_golden(inp[n], inp["S" + n[1]])
    b = run_gpu(deq, Shape(T=256, H=512, I=256, E=16, k=2, r=16))
    for n in ("y", "dx", "dw") + ADAPTER_GRADS:
        assert torch.equal(q[n], b[n]), n


@pytest.mark.parametrize("A,act,clamp,T", [(2, "swiglu", 0.0, 256), (1, "geglu", 0.25, 200), (4, "geglu", 0.0, 512),
                                          (1, "swiglu", 0.0, 77)])
def test_mxfp4_in_gemm_decode_variants_bitwise(A, act, clamp, T):
    """The in-GEMM decode under several adapters (group index = adapter * E + expert),
    GeGLU with and without a binding clamp, and a ragged token count: bit for bit the
    layer with the decoded values as a bf16 base."""
    shp = Shape(T=T, H=512, I=256, E=8, k=2, r=16, A=A, mask_frac=0.1, base_fmt="mxfp4", act=act, clamp=clamp)
    inp = make_inputs(shp, seed=36 + A + T)
    q = run_gpu(inp, shp)
    deq = {n: v for n, v in inp.items() if n not in ("S1", "S3", "S2")}
    for n in ("W1", "W3", "W2"):
        deq[n] = _decode_mxfp4_golden(inp[n], inp["S" + n[1]])
    b = run_gpu(deq, Shape(T=T, H=512, I=256, E=8, k=2, r=16, A=A, mask_frac=0.1, act=act, clamp=clamp))
    assert q["err"] == 0 and b["err"] == 0
    for n in ("y", "dx", "dw") + ADAPTER_GRADS:
        assert torch.equal(q[n], b[n]), n


@pytest.mark.parametrize("H,I", [(576, 320), (192, 64)])
def test_mxfp4_in_gemm_decode_off_tile_boundaries_bitwise(H, I):
    """The in-GEMM decode on partial column tiles and K rows: H, I multiples of 64 but
    not of the tile widths; equal bit for bit to the decoded bf16 base."""
    shp = Shape(T=200, H=H, I=I, E=8, k=2, r=24, mask_frac=0.1, base_fmt="mxfp4")
    inp = make_inputs(shp, seed=35 + H)
    q = run_gpu(inp, shp, poison=True)
    deq = {n: v for n, v in inp.items() if n not in ("S1", "S3", "S2")}
    for n in ("W1", "W3", "W2"):
        deq[n] = _decode_mxfp4_golden(inp[n], inp["S" + n[1]])
    b = run_gpu(deq, Shape(T=200, H=H, I=I, E=8, k=2, r=24, mask_frac=0.1), poison=True)
    for n in ("y", "dx", "dw") + ADAPTER_GRADS:
        assert torch.equal(q[n], b[n]), n


def test_mxfp4_in_gemm_decode_extreme_scales_bitwise():
    """The in-GEMM decode takes a permute-and-multiply route for scale bytes 2..252 and
    the exact fp32 route for the rest (subnormal and overflowing products): with scale
    bytes 0, 1, 253 and 254 mixed into every weight tensor, the layer still gives, bit
    for bit, what it gives with the decoded values (OCP table) as a bf16 base."""
    shp = Shape(T=256, H=512, I=256, E=16, k=2, r=16, base_fmt="mxfp4")
    inp = make_inputs(shp, seed=34)
    g = torch.Generator().manual_seed(34)
    for n in ("S1", "S3", "S2"):
        sc = inp[n].clone()
        pick = torch.rand(sc.shape, generator=g) < 0.05
        sc[pick] = torch.tensor([0, 1, 253, 254], dtype=torch.uint8)[torch.randint(0, 4, (int(pick.sum()),),
                                                                                   generator=g)]
        inp[n] = sc
    q = run_gpu(inp, shp)
    deq = {n: v for n, v in inp.items() if n not in ("S1", "S3", "S2")}
    for n in ("W1", "W3", "W2"):
        deq[n] = _decode_mxfp4_golden(inp[n], inp["S" + n[1]])
    b = run_gpu(deq, Shape(T=256, H=512, I=256, E=16, k=2, r=16))
    for n in ("y", "dx"):
        assert torch.equal(q[n].view(torch.int16), b[n].view(torch.int16)), n
    for n in ("dw",) + ADAPTER_GRADS:
        assert torch.equal(q[n].view(torch.int32), b[n].view(torch.int32)), n


@pytest.mark.parametrize("mx_once", [False, True])
def test_mxfp4_production_width_sampled(mx_once):
    """MXFP4 base at production widths (H=4096, I=2048, E=256, top-6, rank 128),
    2,048 tokens, sampled sparse-dy parity against the oracle; decoded inside the
    GEMMs or once per pass."""
    shp = shape("prod_mxfp4", 2048)
    inp = make_inputs(shp, seed=33, device="cuda")
    sample = [0, 5, 333, 1024, 2047]
    inp = _sparse_dy(inp, shp, sample)
    out = run_gpu(inp, shp, mx_once=mx_once)
    assert out["err"] == 0
    _sampled_check(inp, shp, out, sample)


# ----------------------------------------------------------------------------- activation variants
@pytest.mark.parametrize("act,clamp", [("geglu", 0.0), ("swiglu", 0.25), ("geglu", 0.25)])
def test_activation_variants(act, clamp):
    """GeGLU (exact erf GELU) and the activation clamp on gate/up (the pages'
    SwiGLU/GeGLU and clamp variants); clamp 0.25 binds on these inputs."""
    shp = Shape(T=200, H=512, I=256, E=16, k=2, r=16, mask_frac=0.1, act=act, clamp=clamp)
    inp = make_inputs(shp, seed=41)
    out = run_gpu(inp, shp)
    assert out["err"] == 0
    _full_check(inp, shp, out)


def test_activation_clamp_production_width_sampled():
    """GeGLU with the production runs' clamp value 10 (PR #9, Direct old/new
    numerical comparison), production widths, 1,029 tokens, sampled sparse dy."""
    shp = Shape(T=1029, H=4096, I=2048, E=256, k=6, r=128, mask_frac=0.2, empty_experts=(0, 127, 255),
                act="geglu", clamp=10.0)
    inp = make_inputs(shp, seed=42, device="cuda")
    sample = [0, 3, 500, 1028]
    inp = _sparse_dy(inp, shp, sample)
    out = run_gpu(inp, shp)
    assert out["err"] == 0
    _sampled_check(inp, shp, out, sample)
