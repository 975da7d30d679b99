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
