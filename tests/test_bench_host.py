"""Host-side pieces of bench.py that need no GPU: the workload's algorithmic
bytes and FLOPs, and the choice of the attention kernel's binding roof."""
import pytest

import bench
from mla_decode_attention_uk_gb300.inputs import make_inputs, workload_inputs


def test_workload_stats_count_each_cached_token_once_per_sequence():
    lens = [70, 5, 300]
    inp = make_inputs(len(lens), lens, 2, 32, seed=5)
    st = bench.workload_stats(inp)
    assert st["cache_bytes"] == 1152 * sum(lens)
    # Query t of a 2-token block sees L - 2 + t + 1 keys.
    row_keys = sum(32 * ((L - 1) + L) for L in lens)
    assert st["attn_flops"] == 2 * (576 + 512) * row_keys
    assert st["flops"] == st["attn_flops"] + 2 * 2 * 128 * 512 * len(lens) * 2 * 32
    assert st["weight_bytes"] == 32 * 2 * 128 * 512 * 2
    assert bench.workload_stats(inp, fp8_weights=True)["weight_bytes"] == 32 * 2 * (128 * 512 + 16)
    assert st["tokens"] == len(lens) * 2


@pytest.mark.parametrize("name,bound", [("tp_shard", "hbm"), ("long", "hbm"),
                                        ("full_head", "hbm"), ("mixed_spec", "tensor"),
                                        ("draft_q8", "tensor")])
def test_attention_roofline_binds_the_slower_roof(name, bound):
    st = bench.workload_stats(workload_inputs(name))
    hbm, bf16 = 6784.0, 1937.0
    t = 1e-4
    roof = bench.attention_roofline(st, t, hbm, bf16, "measured", 12345)
    assert roof["bound"] == bound
    gbs, tf = st["cache_bytes"] / t / 1e9, st["attn_flops"] / t / 1e12
    assert roof["hbm_frac"] == pytest.approx(gbs / hbm)
    assert roof["tensor_frac"] == pytest.approx(tf / bf16)
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    assert roof["achieved"] == pytest.approx(gbs if bound == "hbm" else tf)
    assert roof["traffic"] == 12345 and roof["kernel_us"] == pytest.approx(100.0)
