"""Host logic of the benchmark: the re-planning variants and the roofline arithmetic."""
import numpy as np

import bench
from paged_kv_attention_25_gb300 import workloads as wl


def test_replan_variants_are_valid_and_distinct():
    b = wl.llama13b_mixed()
    vs = bench.replan_variants(b, bench.REPLAN_VARIANTS)
    q_lens = np.diff(b.cu_q_lens)
    seen = set()
    for ctx, pos in vs:
        assert ctx.shape == b.ctx_lens.shape and pos.shape == b.q_positions.shape
        for r in range(b.num_reqs):
            p = pos[b.cu_q_lens[r]:b.cu_q_lens[r + 1]]
            assert (p >= 0).all() and (p < ctx[r]).all() and ctx[r] <= b.ctx_lens[r]
            if q_lens[r] > 1:   # multi-token requests are unchanged
                assert ctx[r] == b.ctx_lens[r] and np.array_equal(p, b.q_positions[b.cu_q_lens[r]:b.cu_q_lens[r + 1]])
        seen.add((ctx.tobytes(), pos.tobytes()))
    assert len(seen) == len(vs)
    assert np.array_equal(vs[0][0], b.ctx_lens) and np.array_equal(vs[0][1], b.q_positions)


def test_kernel_roofline_arithmetic():
    st = {"decode_kv_bytes": 6_000_000_000, "decode_io_bytes": 0, "decode_flops": 10**9,
          "tc_kv_bytes": 10**9, "tc_io_bytes": 0, "tc_flops": 2 * 10**15}
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}
    r = bench.kernel_roofline(st, "split_kv", 2e-3, peaks, "test", "none")
    assert r["bound"] == "hbm" and abs(r["achieved"] - 3000.0) < 1e-6 and abs(r["frac"] - 0.5) < 1e-12
    r = bench.kernel_roofline(st, "tensor_core", 2.0, peaks, "test", "none")
    assert r["bound"] == "tensor" and abs(r["achieved"] - 1000.0) < 1e-6 and abs(r["frac"] - 0.5) < 1e-12
    assert r["traffic"] is None


def test_both_arms_describe_the_same_config():
    b = wl.tiny_mixed()
    args = bench.parse_args(["--workload", "tiny_mixed"])
    assert bench.config_of(b, args) == bench.config_of(b, bench.parse_args(["--workload", "tiny_mixed",
                                                                             "--impl", "reference"]))
