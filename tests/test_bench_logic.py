"""Host logic of bench.py that needs no GPU: the attention flop count of multi-row steps
(4 Hq d per visible query-key pair, checked against brute-force pair counting) and the
choice of roofline (tensor above the bf16 / HBM ridge, HBM below)."""
import pytest

import bench

PEAK_HBM_GBS, PEAK_BF16_TFLOPS = 6769.8, 1910.4


def brute_pairs(lengths, qlen, c):
    # query i of a sequence with n cached tokens, at step c, sits at position n + qlen*c + i
    # and sees that position and every earlier one
    return sum(n + qlen * c + i + 1 for n in lengths for i in range(qlen))


@pytest.mark.parametrize("name", ["prefix_chunk", "verify4"])
@pytest.mark.parametrize("c", [0, 1, 5])
def test_attention_flops_count_every_visible_pair(name, c):
    wl = bench.WORKLOADS[name]()
    s = wl.spec
    assert wl.attn_flops(c) == 4 * s.q_heads * s.head_dim * brute_pairs(wl.lengths, wl.qlen, c)


def test_sample_flops_match_the_first_step_of_the_sampled_sequences():
    wl = bench.WORKLOADS["prefix_chunk"]()
    s = wl.spec
    assert wl.sample_flops(1) == 4 * s.q_heads * s.head_dim * brute_pairs(wl.lengths[:1], wl.qlen, 0)


def test_roofline_choice():
    # the 512-row chunk over a 4096-token prefix is far above the ridge (~282 flop/byte);
    # one query or four per sequence stay HBM-bound
    assert bench.WORKLOADS["prefix_chunk"]().tensor_bound(PEAK_HBM_GBS, PEAK_BF16_TFLOPS)
    assert not bench.WORKLOADS["verify4"]().tensor_bound(PEAK_HBM_GBS, PEAK_BF16_TFLOPS)
    assert not bench.WORKLOADS["gqa70b"]().tensor_bound(PEAK_HBM_GBS, PEAK_BF16_TFLOPS)
    assert not bench.WORKLOADS["long_mqa"]().tensor_bound(PEAK_HBM_GBS, PEAK_BF16_TFLOPS)


def test_config_set_covers_the_five_configurations():
    """The default run measures every configuration of the workload set (1 tiny, 2 7B MHA,
    3 70B GQA, 4 the prefix-sharing mix, 5 long GQA, long MQA and the varlen prefill)."""
    keys = [k for k, _, _ in bench.CONFIG_SET]
    assert sorted({k.split("_")[0] for k in keys}) == ["1", "2", "3", "4", "5"]
    assert {name for _, name, _ in bench.CONFIG_SET} == {"tiny", "mha7b", "gqa70b", "mix", "long_gqa",
                                                         "long_mqa", "prefill"}
    assert all(name in bench.WORKLOADS for _, name, _ in bench.CONFIG_SET)
    tiny = bench.WORKLOADS["tiny"]()
    used = sum(bench.gen.blocks_needed(n + 1) for n in tiny.lengths)
    assert (used, used + tiny.spare_blocks) == (5, 8)


def test_config_summary_keeps_the_reported_keys():
    line = {"value": 1.0, "unit": "GB/s", "ms_per_step": 0.2, "pct_hbm_peak": 10.0, "tokens_per_s_per_layer": 5.0,
            "gpu_launches": 20, "steps": 20, "warmup": 5, "other": 1,
            "config": {"workload": "w"}, "cpu_baseline": {"value": 2.0, "cores": 16},
            "roofline": {"bound": "hbm", "achieved": 1.1, "peak": 2.0, "unit": "GB/s", "frac": 0.55,
                         "avg_launch_ms": 0.19, "traffic": None},
            "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3}}
    s = bench.config_summary(line)
    assert s["workload"] == "w" and s["roofline"]["frac"] == 0.55 and s["cpu_baseline"]["cores"] == 16
    assert "other" not in s and "traffic" not in s["roofline"] and s["clocks"]["reasons"] == []
