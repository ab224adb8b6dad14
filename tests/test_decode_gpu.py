"""Decode parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bar (tests/parity.py, applied element-wise): |gpu - oracle| <= 1e-2 + 1e-2 |oracle|
on the same seeded bf16 inputs.
"""
import numpy as np
import pytest
import torch

from grouped_query_attention_09_b300 import workloads as W
from parity import assert_parity

pytestmark = pytest.mark.gpu


def run_decode(g, q, k, v, sl, scale, dev, stream=None):
    qd, kd, vd, sld = q.to(dev), k.to(dev), v.to(dev), sl.to(dev)
    out = g.gqa_decode(qd, kd, vd, sld, scale=scale, stream=stream)
    flags = g.gqa_get_device_status(stream=stream)
    return out.double().cpu().numpy(), flags


def oracle_decode(oracle_mod, q, k, v, sl, scale, check=True):
    return oracle_mod.decode(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), sl.numpy(), scale, check=check)


@pytest.mark.parametrize("name", ["tiny", "llama3_8b", "llama2_70b", "mqa"])
def test_workload_parity_full(gqa_lib, oracle_mod, cuda_device, name):
    """Every output element of the four decode workloads at full size, in the
    launch configuration the benchmark times."""
    w = W.WORKLOADS[name]
    q, k, v, sl = W.make_decode_inputs(w)
    out, flags = run_decode(gqa_lib, q, k, v, sl, w.scale, cuda_device)
    assert flags == 0
    assert_parity(out, oracle_decode(oracle_mod, q, k, v, sl, w.scale), name)


@pytest.mark.parametrize("B,Hq,Hkv,D,Lmax,lens", [
    (3, 8, 2, 128, 700, [700, 333, 65]),      # ragged tails, many tiles, every pair split
    (2, 8, 2, 64, 128, [1, 128]),             # single key; exactly two tiles
    (4, 4, 4, 128, 257, [63, 64, 65, 257]),   # MHA endpoint; tile boundaries
    (5, 16, 1, 128, 300, [300, 1, 150, 64, 129]),  # MQA endpoint G = 16
    (2, 32, 1, 64, 1000, [999, 1000]),        # G = 32 (two head slices) at D = 64
    (2, 6, 2, 64, 96, [96, 17]),              # G = 3 (padded heads)
    (1, 1, 1, 128, 5000, [4999]),             # one head, long
    (2, 16, 2, 128, 640, [640, 600]),         # G = 8
])
def test_shapes_parity(gqa_lib, oracle_mod, cuda_device, B, Hq, Hkv, D, Lmax, lens):
    w = W.DecodeWorkload("case", B, Hq, Hkv, D, Lmax, 1, Lmax, 1000 + B * Hq + D + Lmax)
    q, k, v, _ = W.make_decode_inputs(w)
    sl = torch.tensor(lens, dtype=torch.int32)
    out, flags = run_decode(gqa_lib, q, k, v, sl, w.scale, cuda_device)
    assert flags == 0
    assert_parity(out, oracle_decode(oracle_mod, q, k, v, sl, w.scale), f"{B},{Hq},{Hkv},{D},{lens}")


def test_many_short_sequences_complete_in_one_cta(gqa_lib, oracle_mod, cuda_device):
    """Short sequences in a big batch: most (b, kv head) pairs fall inside one
    CTA's share and take the direct-output path rather than the merge."""
    w = W.DecodeWorkload("short", 512, 8, 2, 64, 200, 1, 200, 77)
    q, k, v, sl = W.make_decode_inputs(w)
    out, flags = run_decode(gqa_lib, q, k, v, sl, w.scale, cuda_device)
    assert flags == 0
    assert_parity(out, oracle_decode(oracle_mod, q, k, v, sl, w.scale), "short")


def test_one_cta_per_pair_with_unequal_lengths(gqa_lib, oracle_mod, cuda_device):
    """128 (b, kv head) pairs nearly fill the GPU, so the plan takes one CTA per
    pair and each CTA prefetches its pair's first tiles into L2 before it reads
    seqlens; with unequal lengths the shares are not the pairs (the prefetch is
    wasted) and the result must not care.  FP8 cache too."""
    B, Hq, Hkv, D, Lmax = 16, 32, 8, 128, 1024
    tk, ctas = gqa_lib.gqa_decode_plan(B, Hq, Hkv, D, Lmax)
    assert ctas == B * Hkv
    w = W.DecodeWorkload("pairs", B, Hq, Hkv, D, Lmax, 1, Lmax, 4242)
    q, k, v, _ = W.make_decode_inputs(w)
    sl = torch.tensor([1024, 1, 700, 65, 64, 1000, 3, 512, 1024, 129, 900, 2, 640, 33, 1023, 256],
                      dtype=torch.int32)
    out, flags = run_decode(gqa_lib, q, k, v, sl, w.scale, cuda_device)
    assert flags == 0
    assert_parity(out, oracle_decode(oracle_mod, q, k, v, sl, w.scale), "one CTA per pair, unequal")
    k8, v8, ks, vs = W.quantize_kv_fp8(k, v)
    dev = cuda_device
    out8 = gqa_lib.gqa_decode_fp8(q.to(dev), k8.to(dev), v8.to(dev), ks.to(dev), vs.to(dev), sl.to(dev),
                                  scale=w.scale)
    assert gqa_lib.gqa_get_device_status() == 0
    ref8 = oracle_mod.decode_fp8(W.bf16_bits(q), k8.numpy(), v8.numpy(), ks.numpy(), vs.numpy(), sl.numpy(),
                                 scale=w.scale)
    assert_parity(out8.double().cpu().numpy(), ref8, "fp8, one CTA per pair, unequal")


def test_nan_tail_is_never_read(gqa_lib, oracle_mod, cuda_device):
    """Cache rows past seqlens[b] filled with NaN (the poison test): the kernel
    must neither read them into a score nor let 0 * NaN into P V."""
    w = W.DecodeWorkload("poison", 4, 16, 4, 128, 1024, 1, 1024, 31)
    q, k, v, _ = W.make_decode_inputs(w)
    sl = torch.tensor([1024, 1, 700, 65], dtype=torch.int32)
    W.poison_tail(k, v, sl)
    out, flags = run_decode(gqa_lib, q, k, v, sl, w.scale, cuda_device)
    assert flags == 0
    assert_parity(out, oracle_decode(oracle_mod, q, k, v, sl, w.scale), "nan tail")


def test_peaky_softmax(gqa_lib, oracle_mod, cuda_device):
    """q scaled x8 makes the softmax sharp, so weight errors are not hidden by
    near-uniform attention."""
    w = W.DecodeWorkload("peaky", 4, 32, 8, 128, 2048, 100, 2048, 41)
    q, k, v, sl = W.make_decode_inputs(w, q_mult=8.0)
    out, flags = run_decode(gqa_lib, q, k, v, sl, w.scale, cuda_device)
    assert flags == 0
    assert_parity(out, oracle_decode(oracle_mod, q, k, v, sl, w.scale), "peaky")


def test_scale_argument(gqa_lib, oracle_mod, cuda_device):
    w = W.DecodeWorkload("scale", 2, 8, 2, 128, 300, 1, 300, 51)
    q, k, v, sl = W.make_decode_inputs(w)
    for scale in (0.02, 0.3):
        out, flags = run_decode(gqa_lib, q, k, v, sl, scale, cuda_device)
        assert_parity(out, oracle_decode(oracle_mod, q, k, v, sl, scale), f"scale {scale}")


def test_empty_and_clamped_lengths_are_flagged(gqa_lib, oracle_mod, cuda_device):
    """seqlens[b] <= 0 -> zero row + GQA_DEV_EMPTY_CONTEXT; seqlens[b] > Lmax ->
    Lmax keys + GQA_DEV_SEQLEN_CLAMPED; the other rows are unaffected."""
    w = W.DecodeWorkload("edge", 4, 8, 2, 128, 256, 1, 256, 61)
    q, k, v, _ = W.make_decode_inputs(w)
    sl = torch.tensor([0, 256, 9999, -5], dtype=torch.int32)
    out, flags = run_decode(gqa_lib, q, k, v, sl, w.scale, cuda_device)
    assert flags == (gqa_lib.GQA_DEV_EMPTY_CONTEXT | gqa_lib.GQA_DEV_SEQLEN_CLAMPED)
    assert np.all(out[0] == 0) and np.all(out[3] == 0)
    ref = oracle_decode(oracle_mod, q, k, v, torch.tensor([1, 256, 256, 1], dtype=torch.int32), w.scale)
    assert_parity(out[1:3], ref[1:3], "clamped")
    assert gqa_lib.gqa_get_device_status() == 0  # read-and-clear


def test_repeatable_and_counters_reset(gqa_lib, cuda_device):
    """Two identical calls give identical bits: the arrival counters of the
    in-kernel merge are back at zero after every call."""
    w = W.WORKLOADS["mqa"]
    q, k, v, sl = [t.to(cuda_device) for t in W.make_decode_inputs(w)]
    a = gqa_lib.gqa_decode(q, k, v, sl).clone()
    for _ in range(3):
        b = gqa_lib.gqa_decode(q, k, v, sl)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert gqa_lib.gqa_get_device_status() == 0


def test_side_stream_and_host_entry_point(gqa_lib, cuda_device):
    """A non-default stream gives the same bits; gqa_decode_host on host
    buffers gives the same bits as gqa_decode on device buffers."""
    w = W.WORKLOADS["tiny"]
    q, k, v, sl = W.make_decode_inputs(w)
    ref = gqa_lib.gqa_decode(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device), sl.to(cuda_device))
    s = torch.cuda.Stream(cuda_device)
    with torch.cuda.stream(s):
        qd, kd, vd, sld = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device), sl.to(cuda_device)
        other = gqa_lib.gqa_decode(qd, kd, vd, sld, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(ref, other)
    host = gqa_lib.gqa_decode_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), sl.pin_memory())
    assert torch.equal(ref.cpu(), host)


# ---- wide groups (G > 8 at D = 128): the tcgen05 decode kernel, the
# group's heads as the MMA rows

@pytest.mark.parametrize("B,Hq,Hkv,Lmax,lens", [
    (3, 16, 1, 700, [700, 129, 1]),          # G = 16; one key; one past a block edge
    (2, 24, 1, 400, [400, 255]),             # G = 24 (not a power of two)
    (3, 36, 3, 260, [260, 1, 200]),          # G = 12
    (2, 64, 1, 1000, [1000, 513]),           # G = 64: two warps of heads
    (1, 128, 1, 384, [384]),                 # G = 128: every TMEM lane a head
    (4, 64, 2, 900, [900, 128, 127, 640]),   # G = 32, two KV heads; block-exact lengths
    (2, 9, 1, 500, [500, 77]),               # G = 9: smallest group on the tcgen05 kernel
    (2, 34, 2, 300, [300, 129]),             # G = 17
    (1, 33, 1, 256, [256]),                  # G = 33: rows of a second lane quarter
    (5, 80, 4, 1500, [1500, 1, 384, 1023, 700]),  # G = 20, four KV heads (whole-pair shares)
    (2, 32, 1, 8192, [8192, 300]),          # one long pair cut into many pieces (split shares, > 4 pieces)
    (4, 64, 2, 4096, [4096, 100, 2000, 4096]),  # G = 32, split shares over every SM, cut pairs
])
def test_wide_group_shapes(gqa_lib, oracle_mod, cuda_device, B, Hq, Hkv, Lmax, lens):
    w = W.DecodeWorkload("wide", B, Hq, Hkv, 128, Lmax, 1, Lmax, 2000 + B * Hq + Lmax)
    q, k, v, _ = W.make_decode_inputs(w)
    sl = torch.tensor(lens, dtype=torch.int32)
    out, flags = run_decode(gqa_lib, q, k, v, sl, w.scale, cuda_device)
    assert flags == 0
    assert_parity(out, oracle_decode(oracle_mod, q, k, v, sl, w.scale), f"wide {B},{Hq},{Hkv},{lens}")


def test_wide_group_nan_tail_peaky_and_edges(gqa_lib, oracle_mod, cuda_device):
    """G = 32: NaN-poisoned cache tail, peaky q (x8), an empty context and a
    clamped length in one batch."""
    w = W.DecodeWorkload("wide_edges", 6, 32, 1, 128, 1024, 1, 1024, 91)
    q, k, v, _ = W.make_decode_inputs(w, q_mult=8.0)
    sl = torch.tensor([1024, 1, 700, 0, 5000, 333], dtype=torch.int32)
    W.poison_tail(k, v, sl.clamp(max=1024))
    out, flags = run_decode(gqa_lib, q, k, v, sl, w.scale, cuda_device)
    assert flags == (gqa_lib.GQA_DEV_EMPTY_CONTEXT | gqa_lib.GQA_DEV_SEQLEN_CLAMPED)
    assert np.all(out[3] == 0)
    ref = oracle_decode(oracle_mod, q, k, v, sl.clamp(min=1, max=1024), w.scale)
    keep = [0, 1, 2, 4, 5]
    assert_parity(out[keep], ref[keep], "wide edges")


def test_wide_group_many_short_sequences_and_repeat(gqa_lib, oracle_mod, cuda_device):
    """Many short MQA sequences (most pieces complete inside one CTA), twice in
    a row: identical bits, counters back at zero."""
    w = W.DecodeWorkload("wide_short", 300, 32, 1, 128, 300, 1, 300, 93)
    q, k, v, sl = W.make_decode_inputs(w)
    qd, kd, vd, sld = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device), sl.to(cuda_device)
    a = gqa_lib.gqa_decode(qd, kd, vd, sld).clone()
    b = gqa_lib.gqa_decode(qd, kd, vd, sld)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert gqa_lib.gqa_get_device_status() == 0
    assert_parity(a.double().cpu().numpy(), oracle_decode(oracle_mod, q, k, v, sl, w.scale), "wide short")


# ---- wide groups over many (b, kv head) pairs: equal shares of the flattened
# block space cut pairs into two to many pieces (merged by the CTA that
# completes each pair's count), including pairs longer than several shares.

def _many_pairs_case(B, Hq, Hkv, Lmax, lens, seed, q_mult=1.0):
    w = W.DecodeWorkload("many_pairs", B, Hq, Hkv, 128, Lmax, 1, Lmax, seed)
    q, k, v, _ = W.make_decode_inputs(w, q_mult=q_mult)
    return w, q, k, v, torch.tensor(lens, dtype=torch.int32)


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,lens", [
    (16, 32, 1, 5120, [5120, 1024] * 8),   # 40-block pairs among 8-block pairs
    # G = 16, four KV heads: 64 pairs of ragged length
    (16, 64, 4, 1024, [1024, 1, 700, 129, 512, 900, 33, 256, 640, 1000, 77, 128, 384, 1023, 255, 800]),
    (32, 18, 2, 600, [600 - 17 * i for i in range(32)]),  # G = 9, two KV heads
    (16, 16, 1, 9472, [9472] + [100] * 15),  # one 74-block pair among 15 one-block pairs
    (16, 32, 1, 8192, [8192] * 16),          # equal 64-block pairs
])
def test_wide_group_many_pairs(gqa_lib, oracle_mod, cuda_device, B, Hq, Hkv, Lmax, lens):
    w, q, k, v, sl = _many_pairs_case(B, Hq, Hkv, Lmax, lens, 4000 + B * Hq + Lmax)
    out, flags = run_decode(gqa_lib, q, k, v, sl, w.scale, cuda_device)
    assert flags == 0
    assert_parity(out, oracle_decode(oracle_mod, q, k, v, sl, w.scale), f"many pairs {B},{Hq},{Hkv},{Lmax}")


def test_wide_group_many_pairs_edges_and_repeat(gqa_lib, oracle_mod, cuda_device):
    """Many pairs with NaN past every sequence end, q x 8, an empty context
    and a clamped length; two calls give identical bits."""
    lens = [1500, 1, 700, 0, 5000, 333, 1024, 1499, 128, 129, 1, 64, 900, 1200, 10, 1500, 777, 256, 1400, 3]
    w, q, k, v, sl = _many_pairs_case(20, 32, 1, 1500, lens, 4321, q_mult=8.0)
    W.poison_tail(k, v, sl.clamp(max=1500))
    d = cuda_device
    qd, kd, vd, sld = q.to(d), k.to(d), v.to(d), sl.to(d)
    a = gqa_lib.gqa_decode(qd, kd, vd, sld, scale=w.scale).clone()
    assert gqa_lib.gqa_get_device_status() == (gqa_lib.GQA_DEV_EMPTY_CONTEXT | gqa_lib.GQA_DEV_SEQLEN_CLAMPED)
    b = gqa_lib.gqa_decode(qd, kd, vd, sld, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert gqa_lib.gqa_get_device_status() == (gqa_lib.GQA_DEV_EMPTY_CONTEXT | gqa_lib.GQA_DEV_SEQLEN_CLAMPED)
    out = a.double().cpu().numpy()
    assert np.all(out[3] == 0)
    ref = oracle_decode(oracle_mod, q, k, v, sl.clamp(min=1, max=1500), w.scale)
    keep = [i for i in range(20) if i != 3]
    assert_parity(out[keep], ref[keep], "many pairs edges")


# ---- limits: the largest batch the kernels take (B = 1024: the per-CTA
# prefix scan of the lengths holds 1025 entries), and a long context.

@pytest.mark.parametrize("Hq,Hkv,Lmax", [(8, 2, 64), (32, 1, 256)])
def test_max_batch(gqa_lib, oracle_mod, cuda_device, Hq, Hkv, Lmax):
    """B = 1024 short ragged sequences, some empty: both kernels (G = 4 on the
    warp-level kernel, G = 32 on the tcgen05 kernel)."""
    g = torch.Generator().manual_seed(77 + Hq)
    sl = torch.randint(0, Lmax + 1, (1024,), generator=g, dtype=torch.int32)
    w = W.DecodeWorkload("maxb", 1024, Hq, Hkv, 128, Lmax, 1, Lmax, 500 + Hq)
    q, k, v, _ = W.make_decode_inputs(w)
    out, flags = run_decode(gqa_lib, q, k, v, sl, w.scale, cuda_device)
    empty = sl <= 0
    assert flags == (gqa_lib.GQA_DEV_EMPTY_CONTEXT if bool(empty.any()) else 0)
    assert np.all(out[empty.numpy()] == 0)
    keep = (~empty).numpy()
    ref = oracle_decode(oracle_mod, q, k, v, sl.clamp(min=1), w.scale)
    assert_parity(out[keep], ref[keep], f"max batch G={Hq // Hkv}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (16, 1)])
def test_long_context(gqa_lib, oracle_mod, cuda_device, Hq, Hkv):
    """131072 cached keys (1024 or 2048 tiles in one pair): the pair is cut
    into many pieces on both kernels."""
    w = W.DecodeWorkload("long", 2, Hq, Hkv, 128, 131072, 1, 131072, 600 + Hq)
    q, k, v, _ = W.make_decode_inputs(w)
    sl = torch.tensor([131072, 70001], dtype=torch.int32)
    out, flags = run_decode(gqa_lib, q, k, v, sl, w.scale, cuda_device)
    assert flags == 0
    assert_parity(out, oracle_decode(oracle_mod, q, k, v, sl, w.scale), f"long context G={Hq // Hkv}")
