"""CPU checks of the arithmetic behind bench.py's JSON line: the step's FLOP
count, the per-kernel algorithmic work behind `roofline`, the peak lookup and
the source hash that keys the committed DRAM-traffic record."""
import bench


def test_step_flops_is_the_causal_fwd_plus_bwd_count():
    w = bench.WORKLOAD
    full = 4.0 * w["B"] * w["H"] * w["M"] * w["N"] * w["D"]
    assert bench.step_flops() == full * 0.5 * 3.5  # causal half; backward 2.5x the forward
    assert bench.flops_fwd(1, 1, 128, 128, 64, False) == 4.0 * 128 * 128 * 64


def test_kernel_algorithmic_work_adds_up_to_the_step():
    """The tensor kernels' algorithmic FLOPs sum to the step's 7
    matmul-equivalents either way the backward runs: forward 2 + dK/dV 4 +
    dQ 1 (the step's attn_bwd), or forward 2 + fused backward 5
    (attn_bwd_fused).  The delta kernel's bytes are O and dO read plus delta
    written; the fused path's convert pass reads the fp32 accumulator and
    writes dQ."""
    for names in (("attn_fwd", "attn_bwd_fused"), ("attn_fwd", "attn_bwd_dkdv", "attn_bwd_dq")):
        f = [bench.kernel_algorithmic(k) for k in names]
        assert all(b == "tensor" for b, _ in f)
        assert abs(sum(x for _, x in f) - bench.step_flops()) < 1.0
    w = bench.WORKLOAD
    rows = w["B"] * w["H"] * w["M"]
    assert bench.kernel_algorithmic("bwd_delta") == ("hbm", rows * w["D"] * 2 * 2 + rows * 4)
    assert bench.kernel_algorithmic("bwd_dq_convert") == ("hbm", rows * w["D"] * 6)
    assert bench.kernel_algorithmic("no_such_kernel") is None


def test_job_tflops_counts_every_rank():
    f = bench.step_flops()
    assert abs(bench.job_tflops(f, 1, 1.0) - f / 1e-3 / 1e12) < 1e-6
    assert abs(bench.job_tflops(f, 4, 1.0) - 4 * bench.job_tflops(f, 1, 1.0)) < 1e-6


def test_source_hash_ignores_comments_only():
    a = "int x = 1; // note\n/* block\n comment */\nint y = 2;\n\n"
    b = "int x = 1;\nint y = 2;"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only("int x = 1;") != bench._code_only("int x = 2;")
    h = bench.kernel_source_hash()
    assert len(h) == 16 and h == bench.kernel_source_hash()
    # each measured kernel is keyed by its own sources: the forward's key does
    # not move with the backward's file, and both kernels of bwd.cu share one
    assert bench.kernel_source_hash("attn_fwd") != bench.kernel_source_hash("attn_bwd_dkdv")
    assert bench.kernel_source_hash("attn_bwd_dq") == bench.kernel_source_hash("attn_bwd_dkdv")
    assert bench.ncu_traffic("no_such_kernel") is None


def test_peak_lookup_accepts_plain_and_nested_values():
    assert bench.peak_value({"hbm_gbs": 7000.0}, "hbm_gbs") == 7000.0
    assert bench.peak_value({"bf16_tflops": {"value": 1900.0}}, "bf16_tflops") == 1900.0
    # a sustained figure falls back to the burst one, then to the stated fallback
    assert bench.peak_value({"bf16_tflops": 1800.0}, "bf16_tflops_sustained") == 1800.0
    assert bench.peak_value({}, "hbm_gbs") == bench.FALLBACK_PEAKS["hbm_gbs"]
