"""Prefill parity: the tcgen05 CUDA path (through the C ABI) against the fp64
oracle, at the bar of tests/parity.py.

Small shapes are compared element by element; they span several 128-row
query tiles and 128-key blocks, ragged tails, both causal settings, even G
(two query heads share each K/V block) and odd G (one head per unit), the MHA
and MQA endpoints, and grids where every CTA walks several units.  The
full-size causal workload (B=4, L=2048, Hq=32, Hkv=8, D=128) is checked on
every element, in the launch configuration the benchmark times.
"""
import pytest
import torch

from grouped_query_attention_09_b300 import workloads as W
from parity import assert_parity

pytestmark = pytest.mark.gpu


def run_prefill(g, q, k, v, causal, dev):
    out = g.gqa_prefill(q.to(dev), k.to(dev), v.to(dev), causal=causal)
    flags = g.gqa_get_device_status()
    return out.cpu(), flags


def oracle_prefill(oracle_mod, q, k, v, causal, rows=None):
    return oracle_mod.prefill(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), causal=causal, rows=rows)


@pytest.mark.parametrize("B,Hq,Hkv,L,causal", [
    (1, 2, 1, 128, True),      # one unit: two heads, one tile, one diagonal block
    (1, 4, 2, 300, True),      # ragged last tile, three query tiles
    (2, 8, 2, 129, False),     # full attention, ragged last key block
    (1, 3, 1, 200, True),      # odd G: one head per unit
    (1, 4, 4, 256, True),      # MHA endpoint
    (1, 8, 1, 1, True),        # a single token
    (1, 2, 1, 100, False),     # shorter than one tile
    (1, 32, 1, 640, True),     # MQA endpoint, G = 32
    (2, 6, 3, 384, False),     # G = 2, full attention
    (4, 16, 4, 1152, True),    # 288 units: every CTA walks two of them
])
def test_shapes_parity(gqa_lib, oracle_mod, cuda_device, B, Hq, Hkv, L, causal):
    w = W.PrefillWorkload("case", B, L, Hq, Hkv, 128, causal, 500 + B * Hq + L)
    q, k, v = W.make_prefill_inputs(w)
    out, flags = run_prefill(gqa_lib, q, k, v, causal, cuda_device)
    assert flags == 0
    ref = oracle_prefill(oracle_mod, q, k, v, causal)
    assert_parity(out.double().numpy(), ref, f"{B},{Hq},{Hkv},{L},{causal}")


# ---- D = 64 (the head size d_model / num_heads of the Huawei Cloud post,
# section 5, is not fixed at 128): 16 KiB tiles and blocks, one 64-column
# box per row, an 8-slot ring, PV with N = 64.
@pytest.mark.parametrize("B,Hq,Hkv,L,causal", [
    (1, 2, 1, 128, True),      # one unit, one diagonal block
    (1, 4, 2, 300, True),      # ragged last tile, three query tiles
    (2, 8, 2, 129, False),     # full attention, ragged last key block
    (1, 3, 1, 200, True),      # odd G: one head per unit
    (1, 8, 1, 1, True),        # a single token
    (1, 32, 4, 640, True),     # G = 8
    (4, 16, 4, 1152, True),    # 288 units: every CTA walks two of them
])
def test_d64_shapes_parity(gqa_lib, oracle_mod, cuda_device, B, Hq, Hkv, L, causal):
    w = W.PrefillWorkload("case64", B, L, Hq, Hkv, 64, causal, 700 + B * Hq + L)
    q, k, v = W.make_prefill_inputs(w)
    out, flags = run_prefill(gqa_lib, q, k, v, causal, cuda_device)
    assert flags == 0
    ref = oracle_prefill(oracle_mod, q, k, v, causal)
    assert_parity(out.double().numpy(), ref, f"D=64 {B},{Hq},{Hkv},{L},{causal}")


def test_d64_peaky_and_full_size(gqa_lib, oracle_mod, cuda_device):
    """D = 64 with q x 8 (re-based running max), then every element of a
    causal B=4, L=2048, Hq=32, Hkv=8 prompt (the benchmark's prefill shape at
    half the head size)."""
    w = W.PrefillWorkload("peaky64", 2, 768, 8, 2, 64, True, 72)
    q, k, v = W.make_prefill_inputs(w, q_mult=8.0)
    for causal in (True, False):
        out, flags = run_prefill(gqa_lib, q, k, v, causal, cuda_device)
        assert flags == 0
        assert_parity(out.double().numpy(), oracle_prefill(oracle_mod, q, k, v, causal), f"D=64 peaky {causal}")
    w = W.PrefillWorkload("full64", 4, 2048, 32, 8, 64, True, 73)
    q, k, v = W.make_prefill_inputs(w)
    out, flags = run_prefill(gqa_lib, q, k, v, True, cuda_device)
    assert flags == 0
    assert_parity(out.double().numpy(), oracle_prefill(oracle_mod, q, k, v, True), "D=64 full size")


def test_peaky_softmax_rebases_running_max(gqa_lib, oracle_mod, cuda_device):
    """q x 8: logits with a spread of tens, so the running max of a row grows
    by more than the re-base margin from block to block and the rescale of the
    partial output is exercised."""
    w = W.PrefillWorkload("peaky", 2, 768, 8, 2, 128, True, 71)
    q, k, v = W.make_prefill_inputs(w, q_mult=8.0)
    for causal in (True, False):
        out, flags = run_prefill(gqa_lib, q, k, v, causal, cuda_device)
        assert flags == 0
        assert_parity(out.double().numpy(), oracle_prefill(oracle_mod, q, k, v, causal), f"peaky causal={causal}")


def test_full_size_causal_workload_every_element(gqa_lib, oracle_mod, cuda_device):
    """The benchmark's prefill workload at full size (B=4, L=2048, Hq=32,
    Hkv=8, D=128, causal), in the launch configuration the benchmark times:
    every element of the output against the oracle (about 137 GFLOP of fp64
    on the host cores, a few seconds with OpenMP)."""
    w = W.WORKLOADS["prefill"]
    q, k, v = W.make_prefill_inputs(w)
    out, flags = run_prefill(gqa_lib, q, k, v, w.causal, cuda_device)
    assert flags == 0
    ref = oracle_prefill(oracle_mod, q, k, v, w.causal)
    assert_parity(out.double().numpy(), ref, "prefill full size")


def test_repeatable_side_stream_and_host_entry(gqa_lib, cuda_device):
    """Identical calls give identical bits, on another stream too, and
    gqa_prefill_host on host buffers matches gqa_prefill on device buffers."""
    w = W.PrefillWorkload("rep", 2, 640, 8, 2, 128, True, 81)
    q, k, v = W.make_prefill_inputs(w)
    qd, kd, vd = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device)
    a = gqa_lib.gqa_prefill(qd, kd, vd).clone()
    s = torch.cuda.Stream(cuda_device)
    s.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(s):
        b = gqa_lib.gqa_prefill(qd, kd, vd, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    host = gqa_lib.gqa_prefill_host(q.pin_memory(), k.pin_memory(), v.pin_memory())
    assert torch.equal(a.cpu(), host)
    assert gqa_lib.gqa_get_device_status() == 0
