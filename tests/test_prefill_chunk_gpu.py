"""Chunked prefill (gqa_prefill_chunk through the C ABI) against the fp64
oracle's prefill_chunk, at the bar of tests/parity.py."""
import pytest
import torch

from grouped_query_attention_09_b300 import workloads as W
from parity import assert_parity

pytestmark = pytest.mark.gpu


def _inputs(B, Hq, Hkv, Lq, Lk, seed, D=128):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, Lq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, Lk, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, Lk, D, generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,causal", [
    (1, 4, 2, 128, 300, True),     # prefix 172: the mask crosses key blocks
    (2, 8, 2, 300, 1000, True),    # ragged chunk after a 700-token prefix
    (1, 8, 1, 1, 129, True),       # one token: a decode step
    (1, 4, 2, 256, 512, True),     # prefix a multiple of the tile
    (2, 6, 2, 200, 333, False),    # full attention over prefix + chunk
    (1, 3, 1, 150, 400, True),     # odd G: one head per unit
])
def test_chunk_parity(gqa_lib, oracle_mod, cuda_device, B, Hq, Hkv, Lq, Lk, causal):
    q, k, v = _inputs(B, Hq, Hkv, Lq, Lk, 6000 + Lq + Lk)
    d = cuda_device
    out = gqa_lib.gqa_prefill_chunk(q.to(d), k.to(d), v.to(d), causal=causal)
    assert gqa_lib.gqa_get_device_status() == 0
    ref = oracle_mod.prefill_chunk(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), causal=causal)
    assert_parity(out.double().cpu().numpy(), ref, f"chunk {B},{Hq},{Hkv},{Lq},{Lk},{causal}")


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lk,causal", [
    (2, 8, 2, 300, 1000, True),    # ragged chunk after a 700-token prefix
    (1, 8, 1, 1, 129, True),       # one token
    (2, 6, 2, 200, 333, False),    # full attention over prefix + chunk
])
def test_chunk_d64_parity(gqa_lib, oracle_mod, cuda_device, B, Hq, Hkv, Lq, Lk, causal):
    q, k, v = _inputs(B, Hq, Hkv, Lq, Lk, 6300 + Lq + Lk, D=64)
    d = cuda_device
    out = gqa_lib.gqa_prefill_chunk(q.to(d), k.to(d), v.to(d), causal=causal)
    assert gqa_lib.gqa_get_device_status() == 0
    ref = oracle_mod.prefill_chunk(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), causal=causal)
    assert_parity(out.double().cpu().numpy(), ref, f"chunk D=64 {B},{Hq},{Hkv},{Lq},{Lk},{causal}")


def test_chunk_full_size_every_element(gqa_lib, oracle_mod, cuda_device):
    """A 512-token chunk after a 1536-token prefix at the prefill workload's
    head shape (B=4, Hq=32, Hkv=8, D=128), the chunk the benchmark times:
    every element against the oracle."""
    B, Hq, Hkv, Lq, Lk = 4, 32, 8, 512, 2048
    q, k, v = _inputs(B, Hq, Hkv, Lq, Lk, 6100)
    d = cuda_device
    out = gqa_lib.gqa_prefill_chunk(q.to(d), k.to(d), v.to(d), causal=True)
    assert gqa_lib.gqa_get_device_status() == 0
    ref = oracle_mod.prefill_chunk(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), causal=True)
    assert_parity(out.double().cpu().numpy(), ref, "chunk full size")


def test_plain_prefill_is_the_chunk_without_prefix(gqa_lib, cuda_device):
    q, k, v = _inputs(2, 8, 2, 640, 640, 6200)
    d = cuda_device
    a = gqa_lib.gqa_prefill(q.to(d), k.to(d), v.to(d))
    b = gqa_lib.gqa_prefill_chunk(q.to(d), k.to(d), v.to(d))
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    with pytest.raises(gqa_lib.GQAError) as e:
        gqa_lib.gqa_prefill_chunk(q.to(d), k[:, :, :100].contiguous().to(d), v[:, :, :100].contiguous().to(d))
    assert e.value.status == gqa_lib.GQA_ERR_INVALID_ARG
