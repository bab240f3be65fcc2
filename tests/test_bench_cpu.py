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
