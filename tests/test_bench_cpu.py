"""Host-side logic of the benchmark: the weight bytes a step streams and the L2 rule.

A workload whose weights per step would fit in twice the 129 MB L2 gets an L2
flush before every timed step; the others stream more than the L2 holds. The
weight bytes are every active expert's prepared weights and scales (0.5625 B
per weight), once per GEMM of the step.
"""

import bench as B
import synth as S


def test_weight_bytes_count_active_experts_once_per_gemm():
    per_weight = 0.5625
    wl, _ = B.resolve("decode_gate_up")
    assert B.weight_bytes_of(wl) == 48 * per_weight * 7168 * 4096          # 48 active experts (skewed routing)
    wl, _ = B.resolve("tp8_decode_gate_up")
    assert B.weight_bytes_of(wl) == 48 * per_weight * 7168 * 512
    wl, _ = B.resolve("tiny_indexed")
    assert B.weight_bytes_of(wl) == 8 * per_weight * 512 * 256
    wl = S.get_workload("prefill_ffn")
    assert B.weight_bytes_of(wl) == 384 * per_weight * (7168 * 4096 + 2048 * 7168)


def test_l2_flush_only_where_weights_fit_in_twice_the_l2():
    flushed = {n: B.needs_l2_flush(B.weight_bytes_of(B.resolve(n)[0]))
               for n in ("tiny_indexed", "tp8_decode_gate_up", "decode_gate_up", "decode_down_combine", "prefill_ffn",
                         "tp8_prefill_ffn")}
    assert flushed == {"tiny_indexed": True, "tp8_decode_gate_up": True, "decode_gate_up": False,
                       "decode_down_combine": False, "prefill_ffn": False, "tp8_prefill_ffn": False}
    wl, layout = B.resolve("tp8_decode_gate_up")
    assert B.config_of(wl, layout, B.weight_bytes_of(wl))["l2"].startswith("L2 flushed before every timed step")
    wl, layout = B.resolve("decode_gate_up")
    assert B.config_of(wl, layout, B.weight_bytes_of(wl))["l2"].startswith("inputs larger than L2")


class _FakeArm:
    dominant_name = "gate_up GEMM"

    def __init__(self, flops, nbytes):
        self.dom_flops, self.dom_bytes = flops, nbytes


def test_roofline_picks_the_binding_bound_and_quotes_the_burst_peak():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    # 4e12 flop at 2000 TFLOP/s = 2000 us > 6e9 B at 6000 GB/s = 1000 us: tensor-bound
    r = B.roofline_of(_FakeArm(4e12, 6e9), 2500.0, peaks, "measured")
    assert r["bound"] == "tensor" and r["peak"] == 2000.0
    assert abs(r["achieved"] - 1600.0) < 1e-9 and abs(r["frac"] - 0.8) < 1e-12
    assert abs(r["sustained"]["frac"] - 1.0) < 1e-12
    # 1e11 flop = 50 us < 6e9 B = 1000 us: HBM-bound
    r = B.roofline_of(_FakeArm(1e11, 6e9), 1250.0, peaks, "measured")
    assert r["bound"] == "hbm" and abs(r["achieved"] - 4800.0) < 1e-9 and abs(r["frac"] - 0.8) < 1e-12


def test_clock_summary_keeps_samples_inside_timed_windows():
    c = B.ClockSampler(0)
    row = "0, {mhz}, 2070, 500.0, 0x0, Not Active, Not Active, Not Active, {cap}"
    c.lines = [(1.0, row.format(mhz=800, cap="Not Active")),      # idle, before the window
               (2.0, row.format(mhz=2060, cap="Not Active")),
               (2.5, row.format(mhz=2040, cap="Active")),
               (5.0, row.format(mhz=900, cap="Not Active"))]       # after the window
    c.mark(1.95, 2.6)
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 2050 and s["reasons"] == ["sw_power_cap"]
    assert c.summary([])["samples"] == 4


def test_regimes_cover_decode_and_every_sweep_point():
    names = set(B.REGIMES)
    assert {"decode_gate_up", "decode_gate_up_masked", "decode_down_combine"} <= names
    for t in S.SWEEP_TOKENS:
        for skew in ("uniform", "zipf"):
            assert f"sweep_gate_up_t{t}_{skew}" in names
    for n in names:
        B.resolve(n)


def test_masked_workloads_budget_covers_their_hottest_expert():
    """Every masked workload the bench times holds its hottest expert's rows within its row budget (else the call
    would record a capacity error instead of a result), and the masked sweep point is a split call (expected_m, the
    mean rows of its active experts, between 24 and 127)."""
    import numpy as np
    for name, alias in B.WORKLOAD_ALIASES.items():
        wl, layout = B.resolve(name)
        if layout != "masked":
            continue
        ids, _ = S.routing(wl)
        counts = np.bincount(ids.reshape(-1), minlength=wl.num_experts)
        assert wl.max_m >= counts.max(), name
        if name.startswith("sweep_"):
            expected_m = int(counts[counts > 0].mean())
            assert 24 <= expected_m < 128, (name, expected_m)
