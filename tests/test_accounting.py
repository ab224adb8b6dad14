"""The byte and flop counts the benchmark divides by, pinned to the pages."""
import json
import os

from grouped_query_attention_09_b300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_kv_cache_size_worked_example():
    """GQA paper notes (51969.com), "QA 相关": Llama2-7B, b=1, s=4000,
    h=4096, l=32 in fp16 -> 4bshl = 2,097,152,000 bytes (about 1.95 GB)."""
    g = json.load(open(os.path.join(GOLDEN, "kv_cache_size_llama2_7b.json")))
    got = W.kv_cache_bytes(g["b"], g["s"], g["h"], g["l"], g["elem_bytes"])
    assert got == g["bytes"]
    assert abs(got / 2**30 - g["approx_gb"]) < 0.005


def test_decode_bytes_of_the_llama3_8b_workload():
    """B=16, Hkv=8, D=128, 4096 keys each: 16*4096 tokens x 8 heads x 128 x 2 tensors x 2 bytes."""
    w = W.WORKLOADS["llama3_8b"]
    _, _, _, sl = W.make_decode_inputs(W.DecodeWorkload("s", w.B, w.Hq, w.Hkv, w.D, 64, 64, 64, 0))
    assert W.decode_kv_bytes(sl * 64, w.Hkv, w.D) == 268435456


def test_bandwidth_model_scales_with_kv_heads():
    """Per-step cache traffic is O(Hkv * seq * d) ("手把手教你用PyTorch实现GQA",
    section 2.1): MHA (Hkv = H) reads H times what MQA (Hkv = 1) reads."""
    sl = [1024]
    assert W.decode_kv_bytes(sl, 32, 128) == 32 * W.decode_kv_bytes(sl, 1, 128)
    assert W.decode_kv_bytes(sl, 4, 128) == 4 * W.decode_kv_bytes(sl, 1, 128)


def test_prefill_flops():
    assert W.prefill_flops(4, 32, 2048, 128, True) == 137506062336
    assert W.prefill_flops(4, 32, 2048, 128, False) == 2 * 137438953472
    assert W.prefill_flops(1, 1, 1, 1, True) == 4


def test_seeded_inputs_are_reproducible():
    w = W.DecodeWorkload("r", 3, 4, 2, 8, 16, 3, 16, 123)
    a = W.make_decode_inputs(w)
    b = W.make_decode_inputs(w)
    for x, y in zip(a, b):
        assert x.equal(y)
    assert int(a[3].min()) >= 3 and int(a[3].max()) <= 16


def test_cpu_baseline_sampler_cycles_whole_steps():
    """bench.py's CPU baseline: with cycling, a step shorter than the budget is
    timed repeatedly (the sample names whole steps, the rate is the step's K/V
    bytes over the mean step time); without it, one step at most."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    gbs, step_s, sample, threads = bench.oracle_decode_rate(W, "tiny", budget_s=0.3, cycle=True)
    w = W.WORKLOADS["tiny"]
    nbytes = W.decode_kv_bytes(W.make_decode_inputs(w)[3], w.Hkv, w.D)
    assert "steps of" in sample and threads >= 1 and step_s > 0
    assert abs(gbs - nbytes / step_s / 1e9) <= 1e-9 * gbs
    _, _, one, _ = bench.oracle_decode_rate(W, "tiny", budget_s=0.3, cycle=False)
    assert "of one step" in one
