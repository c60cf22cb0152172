"""GPU parity of the native FP4 forward (base_fmt 3): the gate/up base products on
block-scaled FP4 tensor cores (tcgen05 kind::mxf8f6f4), MXFP8 routed rows times the
MXFP4 base as stored ("FP8/FP4/FP8 forwards", "feat(mega): add fused shared
side-LoRA kernels", Fresh validation; the native MXFP4 base timed beside the
dequantised one in its Performance notes).

Bars:
  * the MXFP8 quantiser: the oracle's codes and scale bytes, bit for bit;
  * the block-scaled GEMM engine: float64 within fp32 accumulation (relL2 1e-6);
  * the layer against the oracle's native mode (the same MXFP8 activations, a
    straight-through backward): relL2 5e-3 and cosine 0.9999 as everywhere;
  * the stated, looser gate against the BF16-activation layer: relL2 1e-1 on y.
    Both forward base products take E4M3 inputs (3 mantissa bits: a relative rounding
    error up to 2^-4 per element, ~0.03 RMS); two independent roundings give ~0.04,
    which the gate's derivative can amplify by up to ~1.5.
"""
import pytest
import torch

import moe_expert_ffn_top_gb300 as m
import oracle
from synth import Shape, make_inputs, shape

from gpu_common import _full_check, _sampled_check, _sparse_dy, rel_l2, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_ffn_top_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield


def _tables():
    e4 = torch.tensor([oracle.e4m3_value(c) for c in range(256)], dtype=torch.float64)
    e2 = torch.tensor([oracle.e2m1_value(c) for c in range(16)], dtype=torch.float64)
    return e4, e2


def _tiles(sc):
    """Scale bytes [rows, K/32] -> the tile-major layout [rows/128][K/128][32][4][4]:
    per 128-row block and 128-wide K step, row 32b + a's 4 bytes at word 4a + b."""
    rows, nb = sc.shape
    return sc.view(rows // 128, 4, 32, nb // 4, 4).permute(0, 3, 2, 1, 4).contiguous()


def _native_operands(M, N, K, seed, lo=118, hi=136):
    g = torch.Generator().manual_seed(seed)
    aq = (torch.randint(0, 127, (M, K), generator=g) | (torch.randint(0, 2, (M, K), generator=g) << 7)).to(torch.uint8)
    bc = torch.randint(0, 16, (N, K), generator=g)
    asc = torch.randint(lo, hi, (M, K // 32), generator=g).to(torch.uint8)
    bsc = torch.randint(lo, hi, (N, K // 32), generator=g).to(torch.uint8)
    bq = (bc[:, 0::2] | (bc[:, 1::2] << 4)).to(torch.uint8)
    e4, e2 = _tables()
    A = e4[aq.long()] * torch.exp2(asc.double() - 127).repeat_interleave(32, 1)
    B = e2[bc.long()] * torch.exp2(bsc.double() - 127).repeat_interleave(32, 1)
    return aq, asc, bq, bsc, A @ B.T


@pytest.mark.parametrize("layout", [0, 2])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 512), (640, 768, 1024)])
def test_native_engine_gemm(M, N, K, layout):
    """The block-scaled MMA path of the engine (E4M3 x E2M1, UE8M0 per 32 on both
    sides, scale words in tensor memory, written by the epilogue warps (0) or copied
    by the MMA thread (2)) against float64."""
    aq, asc, bq, bsc, ref = _native_operands(M, N, K, seed=M + N + K)
    C = torch.full((M, N), float("nan"), device="cuda")
    m.moe_lora_native_selftest(aq.cuda(), _tiles(asc).cuda(), bq.cuda(), _tiles(bsc).cuda(), C, layout=layout)
    torch.cuda.synchronize()
    assert m.moe_lora_gemm_selftest_error() == 0
    assert rel_l2(C, ref) < 1e-6


def test_native_engine_scale_placement_matters():
    """The scale words really are read where the engine puts them: the one-row-per-lane
    placement gives a different, wrong product on the same operands."""
    aq, asc, bq, bsc, ref = _native_operands(256, 512, 256, seed=5)
    C = torch.full((256, 512), float("nan"), device="cuda")
    m.moe_lora_native_selftest(aq.cuda(), _tiles(asc).cuda(), bq.cuda(), _tiles(bsc).cuda(), C, layout=1)
    torch.cuda.synchronize()
    assert m.moe_lora_gemm_selftest_error() == 0
    assert rel_l2(C, ref) > 1e-2


def _quant_inputs(rows, n, seed):
    """bf16 rows with per-block magnitudes from 2^-40 to 2^40, all-zero blocks,
    bf16 subnormals, E4M3 ties and values that saturate."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, n, generator=g, dtype=torch.float64)
    mag = torch.exp2(torch.randint(-40, 40, (rows, n // 32), generator=g).double()).repeat_interleave(32, 1)
    x = x * mag
    x[0, :32] = 0.0
    x[1, :32] = torch.randn(32, generator=g, dtype=torch.float64) * 2.0 ** -133   # bf16 subnormals
    x[2, :32] = torch.tensor([256.0, 264.0, 272.0, 280.0, 448.0, 456.0, 464.0, 470.0, 480.0, 500.0, 511.0,
                              -264.0, -456.0, -470.0, 1.0, -1.0, 0.5, 0.0, -0.0] + [3.0] * 13, dtype=torch.float64)
    return x.to(torch.bfloat16)


def test_mxfp8_quantizer_bitwise():
    """The library's MXFP8 quantiser against the oracle's: scale bytes bit for bit,
    element codes bit for bit wherever the value is non-zero (a zero may carry
    either sign bit)."""
    rows, n = 96, 4096
    x = _quant_inputs(rows, n, seed=3)
    codes = torch.empty(rows, n, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, n // 32, dtype=torch.uint8, device="cuda")
    m.moe_lora_mxfp8_quantize(x.cuda(), codes, scales)
    torch.cuda.synchronize()
    codes, scales = codes.cpu(), scales.cpu()
    for i in range(rows):
        wc, ws, _ = oracle.mxfp8_quantize(x[i].double())
        assert torch.equal(scales[i], ws), i
        nz = (wc & 0x7F) != 0
        assert torch.equal(codes[i][nz], wc[nz]), i
        assert ((codes[i][~nz] & 0x7F) == 0).all(), i


@pytest.mark.parametrize("once", [False, True])
def test_native_tiny_forward_backward(once):
    """base_fmt 3 (the rest decoded in the GEMMs) and 4 (decoded once per pass)."""
    shp = Shape(T=200, H=512, I=256, E=16, k=2, r=16, mask_frac=0.1, base_fmt="mxfp4_native")
    inp = make_inputs(shp, seed=61)
    out = run_gpu(inp, shp, poison=True, mx_once=once)
    assert out["err"] == 0
    _full_check(inp, shp, out)


def test_native_modes_agree_bitwise():
    """base_fmt 3 and 4 differ only in where the MXFP4 weights are decoded (exactly)
    outside the native products: every output and gradient equal bit for bit."""
    shp = Shape(T=256, H=512, I=256, E=16, k=2, r=16, base_fmt="mxfp4_native")
    inp = make_inputs(shp, seed=65)
    a = run_gpu(inp, shp)
    b = run_gpu(inp, shp, mx_once=True)
    for n in ("y", "dx", "dw", "dA1", "dA3", "dB1", "dB3", "dA2", "dB2"):
        assert torch.equal(a[n], b[n]), n


@pytest.mark.parametrize("A,act,clamp,T,H,I", [(2, "swiglu", 0.0, 256, 512, 256), (1, "geglu", 0.25, 77, 640, 384),
                                               (4, "geglu", 0.0, 512, 256, 128)])
def test_native_variants(A, act, clamp, T, H, I):
    """Several adapters, GeGLU with and without a binding clamp, a ragged token count,
    and widths that are multiples of 128 but not of 256."""
    shp = Shape(T=T, H=H, I=I, E=8, k=2, r=16, A=A, mask_frac=0.1, base_fmt="mxfp4_native", act=act, clamp=clamp)
    inp = make_inputs(shp, seed=62 + A + T)
    out = run_gpu(inp, shp, poison=True)
    assert out["err"] == 0
    _full_check(inp, shp, out)


def test_native_looser_gate_against_bf16_activations():
    """The stated gate of the native forward against the same layer with BF16
    activations (the MXFP4 base decoded inside the GEMMs): relL2 <= 1e-1 on y (two
    E4M3 roundings, see the module docstring), and the two differ (the activations
    really are quantised)."""
    shp = Shape(T=256, H=512, I=256, E=16, k=2, r=16, base_fmt="mxfp4_native")
    inp = make_inputs(shp, seed=63)
    nat = run_gpu(inp, shp, backward=False)
    ref = run_gpu(inp, Shape(**{**shp.__dict__, "base_fmt": "mxfp4"}), backward=False)
    d = rel_l2(nat["y"], ref["y"])
    assert 1e-4 < d <= 1e-1, d


@pytest.mark.parametrize("once", [False, True])
def test_native_production_width_sampled(once):
    """Production widths (H=4096, I=2048, E=256, top-6, rank 128), 2,048 tokens,
    sampled sparse-dy parity against the oracle's native mode (base_fmt 3 and 4)."""
    shp = shape("prod_native", 2048)
    inp = make_inputs(shp, seed=64, device="cuda")
    sample = [0, 7, 700, 1500, 2047]
    inp = _sparse_dy(inp, shp, sample)
    out = run_gpu(inp, shp, mx_once=once)
    assert out["err"] == 0
    _sampled_check(inp, shp, out, sample)


@pytest.mark.parametrize("once", [False, True])
def test_native_edge_production_width_sampled(once):
    """The native forward on the pages' boundary sweep shape: production widths, a
    fifth of the routes masked, experts 0/127/255 empty, an odd token count (1,029),
    GeGLU with the production clamp 10; sampled sparse-dy parity against the oracle's
    native mode, and the routed rows' padding never reaching an output."""
    shp = Shape(T=1029, H=4096, I=2048, E=256, k=6, r=128, mask_frac=0.2, empty_experts=(0, 127, 255),
                base_fmt="mxfp4_native", act="geglu", clamp=10.0)
    inp = make_inputs(shp, seed=66, device="cuda")
    sample = [0, 1, 514, 1028]
    inp = _sparse_dy(inp, shp, sample)
    out = run_gpu(inp, shp, poison=True, mx_once=once)
    assert out["err"] == 0
    _sampled_check(inp, shp, out, sample)
