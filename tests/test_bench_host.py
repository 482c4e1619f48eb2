"""Host-side arithmetic of bench.py (no GPU): flop and byte accounting and
the rule that a recorded ncu traffic figure is only used for the kernel
sources it was taken on."""
import os

import pytest

import bench


def test_flops_of_each_workload():
    from coda_inputs import WORKLOADS
    fl = bench.gemm_flops_by_kernel(WORKLOADS["llama1b_attn_out_swiglu"])
    assert fl["gemm_residual_partial_rms"] == 2 * 8192 * 2048 * 2048
    assert fl["gemm_swiglu"] == 2 * 8192 * 16384 * 2048
    assert sum(fl.values()) / 1e9 == pytest.approx(618.5, abs=0.1)
    # the per-kernel split agrees with the workload's own flop count
    for name in ("llama1b_mlp_down_qkv", "llama8b_chain", "llama8b_chain_fp8"):
        w = WORKLOADS[name]
        assert sum(bench.gemm_flops_by_kernel(w).values()) == pytest.approx(w.gemm_flops())
    assert sum(bench.gemm_flops_by_kernel(WORKLOADS["llama8b_chain"]).values()) / 1e9 == pytest.approx(7146.8, abs=1)


def test_fused_moves_fewer_bytes_than_unfused():
    fused, unfused = bench.algorithmic_bytes(8192, 2048, 2048, 8192, 16)
    assert sum(fused.values()) / 1e6 == pytest.approx(345.0, abs=2.0)
    assert unfused / 1e6 == pytest.approx(1015.0, abs=10.0)
    assert unfused / sum(fused.values()) > 2.5


def test_recorded_traffic_requires_matching_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", {"gemm": ["k.cu", "k.cuh"], "aux": ["a.cu"]})
    csrc = tmp_path / "gemm_epilogue_fusion_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1")
    (csrc / "k.cuh").write_text("header v1")
    (csrc / "a.cu").write_text("aux v1")
    (tmp_path / "profiles").mkdir()
    sha = bench.kernel_source_sha()
    (tmp_path / "profiles" / "ncu_x.md").write_text(f"source_sha: {sha}\ndram_bytes_per_launch: 1.5e8\n")
    assert bench.recorded_traffic("x") == 1.5e8
    (csrc / "a.cu").write_text("aux v2")  # another kernel family: the GEMM figure stays valid
    assert bench.recorded_traffic("x") == 1.5e8
    (csrc / "k.cu").write_text("kernel   v1 // a comment\n/* and a\n block */")  # comments and spacing only
    assert bench.recorded_traffic("x") == 1.5e8
    (csrc / "k.cuh").write_text("header v2")
    assert bench.recorded_traffic("x") is None
    assert bench.recorded_traffic("missing") is None


def test_timed_kernel_bytes_of_the_block_launches():
    from coda_inputs import WORKLOADS
    # LLaMA-3-1B attention-out block in one launch: X, Wo, R, h, P, then h, Wg, Wu, act, P, r
    assert bench.timed_kernel_bytes(WORKLOADS["llama1b_attn_out_swiglu"], "block", 16) / 1e6 == \
        pytest.approx(345.0, abs=1.0)
    # LLaMA-3-8B chain, first block (Wo + gate/up): 438.3 MB of phase A, 841.0 MB of phase B
    w = WORKLOADS["llama8b_chain"]
    M, H, I, T = w.M, w.N, w.inter, 32
    phase_a = 2 * (M * H + H * H + 2 * M * H) + 4 * M * T
    phase_b = 2 * (M * H + 2 * I * H + M * I) + 4 * M * T + 4 * M
    assert bench.timed_kernel_bytes(w, "block", T) == phase_a + phase_b
    assert bench.timed_kernel_bytes(w, "fused", T) == phase_b
    assert (phase_a + phase_b) / 1e6 == pytest.approx(1279.3, abs=0.5)


def test_config_names_the_workload_only():
    """Both arms print config_of(w): it holds the workload's keys, none that
    depend on how an arm runs it, so the two arms' configs are identical."""
    from coda_inputs import WORKLOADS
    for w in WORKLOADS.values():
        c = bench.config_of(w)
        assert c["workload"] == w.name and c["M"] == w.M and c["dtype"] == w.dtype
        assert "chain" not in c and not any("launch" in str(v) for v in c.values())


def test_default_workload_is_the_8b_chain(monkeypatch):
    seen = {}
    monkeypatch.setattr(bench, "run_coda", lambda args, w: seen.update(w=w, args=args))
    monkeypatch.setattr("sys.argv", ["bench.py"])
    bench.main()
    assert seen["w"].name == "llama8b_chain" and seen["args"].reduce in ("auto", "block")
    assert seen["args"].sustained_s >= 2.0


def test_chain_bytes_of_the_8b_chain():
    """The 8B chain's compulsory bytes: 2525.1 MB through the two one-launch
    blocks against 5469.4 MB for the unfused sequence (2.17x)."""
    from coda_inputs import WORKLOADS
    fused, unfused = bench.chain_bytes_full(WORKLOADS["llama8b_chain"], 32)
    assert fused / 1e6 == pytest.approx(2525.1, abs=0.1)
    assert unfused / 1e6 == pytest.approx(5469.4, abs=0.1)
    # the first block's share equals the timed kernel's bytes
    w = WORKLOADS["llama8b_chain"]
    assert bench.timed_kernel_bytes(w, "block", 32) < fused
