"""Host-side logic of bench.py (no GPU): the FLOP model behind `value` and the
roofline, the per-kernel source hash that keys the committed DRAM-traffic counters, and the
multi-rank helpers on one rank."""
import importlib.util
import json
import os
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


@pytest.mark.parametrize("T,R,H,I,r,k,E", [(65536, 393216, 4096, 2048, 128, 6, 256),
                                           (16384, 131072, 2048, 768, 8, 8, 128), (256, 400, 512, 256, 16, 2, 16)])
def test_kernel_flops_sum_to_the_step(bench, T, R, H, I, r, k, E):
    """The per-kernel algorithmic FLOPs (roofline, per-kernel rates) add up exactly to
    the step's FLOPs (`value`): 12RHI + 18THr + 18RIr.  The native FP4 forward's two
    GEMMs replace w13_lora_swiglu / w2_a2 with the same work, so they are counted once
    (as those) and must equal them."""
    fl, _ = bench.kernel_work(T, R, H, I, r, k, E)
    assert fl["w13_native"] == fl["w13_lora_swiglu"] and fl["w2_native"] == fl["w2_a2"]
    step = sum(v for n, v in fl.items() if not n.endswith("_native"))
    assert step == pytest.approx(bench.step_flops(T, R, H, I, r), rel=1e-12)


def test_dominant_kernel_is_one_the_configuration_launches(bench):
    """The roofline's kernel is W13 (tied with the W13 dgrad, the forward first): the
    BF16/MXFP4 W13 GEMM, or the native one when the forward's base products run on FP4
    tensor cores (that configuration never launches w13_lora_swiglu)."""
    fl, _ = bench.kernel_work(65536, 393216, 4096, 2048, 128, 6, 256)
    assert bench.dominant_kernel(fl, native=False) == "w13_lora_swiglu"
    assert bench.dominant_kernel(fl, native=True) == "w13_native"


def test_production_step_flops(bench):
    """42.06 TFLOP at 65,536 tokens, H4096 I2048, top-6, rank 128 (every route live)."""
    assert bench.step_flops(65536, 393216, 4096, 2048, 128) / 1e12 == pytest.approx(42.056, abs=1e-3)


def _copy_tree(bench, tmp_path):
    src = os.path.join(ROOT, "moe_expert_ffn_top_gb300")
    shutil.copytree(src, tmp_path / "moe_expert_ffn_top_gb300",
                    ignore=shutil.ignore_patterns("*.so", "*.o", "__pycache__", "_build*"))
    return tmp_path / "moe_expert_ffn_top_gb300" / "csrc"


def test_source_hash_ignores_comments_only(bench, tmp_path):
    dst = _copy_tree(bench, tmp_path)
    root = bench.ROOT
    try:
        bench.ROOT = str(tmp_path)
        h0 = bench.src_hash("w13_lora_swiglu")
        p = dst / "gemm_engine.cuh"
        text = p.read_text()
        p.write_text("// a comment\n/* a block\n   comment */\n\n" + text.replace("\n", "  // note\n", 3))
        assert bench.src_hash("w13_lora_swiglu") == h0
        p.write_text(text + "\nstatic const int kUnused = 1;\n")
        assert bench.src_hash("w13_lora_swiglu") != h0
    finally:
        bench.ROOT = root


def test_source_hash_is_per_problem(bench, tmp_path):
    """A code change inside one problem type (or its host launch block) re-keys that
    kernel's record only."""
    dst = _copy_tree(bench, tmp_path)
    root = bench.ROOT
    try:
        bench.ROOT = str(tmp_path)
        names = list(bench.PROBLEM_OF)
        h0 = {n: bench.src_hash(n) for n in names}
        assert len(set(h0.values())) == len(names)
        p = dst / "gemm_problems.cuh"
        text = p.read_text()
        marker = "struct ProbA13Expand {"
        assert marker in text
        p.write_text(text.replace(marker, marker + "\n  static constexpr int kProbe = 1;"))
        h1 = {n: bench.src_hash(n) for n in names}
        assert [n for n in names if h1[n] != h0[n]] == ["a13_expand"]
        p.write_text(text)
        f = dst / "forward.cu"
        ftext = f.read_text()
        f.write_text(ftext.replace("p.clamp = d->act_clamp;", "p.clamp = d->act_clamp + 0.0f;", 1))
        h2 = {n: bench.src_hash(n) for n in names}
        assert [n for n in names if h2[n] != h0[n]] == ["w13_lora_swiglu"]
    finally:
        bench.ROOT = root


def test_traffic_follows_the_source_hash(bench, tmp_path):
    _copy_tree(bench, tmp_path)
    root = bench.ROOT
    try:
        bench.ROOT = str(tmp_path)
        rec = {"w13_lora_swiglu": {"bytes_per_launch": 123, "src_hash": bench.src_hash("w13_lora_swiglu")}}
        (tmp_path / "profiles").mkdir()
        (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
        assert bench.traffic_for("w13_lora_swiglu") == 123
        assert bench.traffic_for("w2_a2") is None
        rec["w13_lora_swiglu"]["src_hash"] = "0" * 16
        (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
        assert bench.traffic_for("w13_lora_swiglu") is None
    finally:
        bench.ROOT = root


def test_single_rank_helpers(bench):
    assert bench.max_over_ranks(None, 3.5, "cpu") == 3.5
    assert bench.job_tflops(1, 42.056e12, 30.0) == pytest.approx(1401.87, rel=1e-4)
    assert bench.job_tflops(4, 1e12, 1.0) == pytest.approx(4000.0)
