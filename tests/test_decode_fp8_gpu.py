"""FP8 (E4M3) KV-cache decode: the CUDA path (gqa_decode_fp8 through the C ABI)
against the fp64 oracle's decode_fp8 on the same bytes and scales, at the bar
of tests/parity.py.  The oracle dequantises exactly (E4M3 value times the
per-(b, kv head) scale); the kernel converts E4M3 exactly to fp16, rounds q and
P to fp16 and accumulates in fp32."""
import numpy as np
import pytest
import torch

from grouped_query_attention_09_b300 import workloads as W
from parity import assert_parity

pytestmark = pytest.mark.gpu


def run_fp8(g, q, k8, v8, ks, vs, sl, scale, dev):
    out = g.gqa_decode_fp8(q.to(dev), k8.to(dev), v8.to(dev), ks.to(dev), vs.to(dev), sl.to(dev), scale=scale)
    flags = g.gqa_get_device_status()
    return out.double().cpu().numpy(), flags


def oracle_fp8(o, q, k8, v8, ks, vs, sl, scale):
    return o.decode_fp8(W.bf16_bits(q), k8.numpy(), v8.numpy(), ks.double().numpy(), vs.double().numpy(),
                        sl.numpy(), scale)


@pytest.mark.parametrize("name", ["llama3_8b", "llama2_70b", "mqa"])
def test_fp8_workload_parity_full(gqa_lib, oracle_mod, cuda_device, name):
    """Every output element of the Llama-shaped workloads and of the ragged
    MQA batch (G = 32: the tcgen05 kernel with its E4M3 -> fp16 converter
    warps) with the cache in FP8."""
    w = W.WORKLOADS[name]
    q, k8, v8, ks, vs, sl = W.make_decode_fp8_inputs(w)
    out, flags = run_fp8(gqa_lib, q, k8, v8, ks, vs, sl, w.scale, cuda_device)
    assert flags == 0
    assert_parity(out, oracle_fp8(oracle_mod, q, k8, v8, ks, vs, sl, w.scale), name + " fp8")


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,lens", [
    (3, 8, 2, 700, [700, 333, 65]),       # ragged tails, many tiles
    (2, 8, 2, 128, [1, 128]),             # a single key; exactly two tiles
    (4, 4, 4, 257, [63, 64, 65, 257]),    # MHA endpoint; tile boundaries
    (2, 6, 2, 300, [300, 17]),            # G = 3
    (1, 1, 1, 3000, [2999]),              # one head, long
    (3, 16, 1, 700, [700, 129, 1]),       # G = 16 (tcgen05 kernel): one key; one past a block edge
    (2, 24, 1, 400, [400, 255]),          # G = 24
    (3, 36, 3, 260, [260, 1, 200]),       # G = 12
    (2, 64, 1, 1000, [1000, 513]),        # G = 64
    (1, 128, 1, 384, [384]),              # G = 128: every TMEM lane a head
    (2, 32, 1, 8192, [8192, 300]),        # one long pair cut into many pieces (> 4-piece merge)
    (4, 64, 2, 4096, [4096, 100, 2000, 4096]),  # G = 32 over every SM, cut pairs
])
def test_fp8_shapes(gqa_lib, oracle_mod, cuda_device, B, Hq, Hkv, Lmax, lens):
    w = W.DecodeWorkload("fp8", B, Hq, Hkv, 128, Lmax, 1, Lmax, 3000 + B * Hq + Lmax)
    q, k8, v8, ks, vs, _ = W.make_decode_fp8_inputs(w)
    sl = torch.tensor(lens, dtype=torch.int32)
    out, flags = run_fp8(gqa_lib, q, k8, v8, ks, vs, sl, w.scale, cuda_device)
    assert flags == 0
    assert_parity(out, oracle_fp8(oracle_mod, q, k8, v8, ks, vs, sl, w.scale), f"fp8 {B},{Hq},{Hkv},{lens}")


def test_fp8_nan_tail_peaky_and_edges(gqa_lib, oracle_mod, cuda_device):
    """E4M3 NaN bytes in every cache row past seqlens[b], q x 8, an empty
    context and a clamped length in one batch."""
    w = W.DecodeWorkload("fp8_edges", 5, 16, 4, 128, 1024, 1, 1024, 97)
    sl = torch.tensor([1024, 1, 700, 0, 9999], dtype=torch.int32)
    q, k8, v8, ks, vs, _ = W.make_decode_fp8_inputs(w, q_mult=8.0)
    for b in range(5):
        n = int(sl[b].clamp(0, 1024))
        k8[b, :, n:, :] = W.E4M3_NAN
        v8[b, :, n:, :] = W.E4M3_NAN
    out, flags = run_fp8(gqa_lib, q, k8, v8, ks, vs, sl, w.scale, cuda_device)
    assert flags == (gqa_lib.GQA_DEV_EMPTY_CONTEXT | gqa_lib.GQA_DEV_SEQLEN_CLAMPED)
    assert np.all(out[3] == 0)
    ref = oracle_fp8(oracle_mod, q, k8, v8, ks, vs, sl.clamp(min=1, max=1024), w.scale)
    keep = [0, 1, 2, 4]
    assert_parity(out[keep], ref[keep], "fp8 edges")


@pytest.mark.parametrize("Hq,Hkv", [(16, 2), (32, 1)])
def test_fp8_scales_and_repeat(gqa_lib, cuda_device, Hq, Hkv):
    """Doubling every V scale doubles the output (to bf16 rounding); two calls
    give identical bits (the warp-level kernel at G = 8, the tcgen05 kernel
    at G = 32)."""
    w = W.DecodeWorkload("fp8_scale", 4, Hq, Hkv, 128, 600, 1, 600, 99)
    q, k8, v8, ks, vs, sl = [t.to(cuda_device) for t in W.make_decode_fp8_inputs(w)]
    a = gqa_lib.gqa_decode_fp8(q, k8, v8, ks, vs, sl).clone()
    b = gqa_lib.gqa_decode_fp8(q, k8, v8, ks, vs, sl).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    d = gqa_lib.gqa_decode_fp8(q, k8, v8, ks, 2 * vs, sl)
    torch.cuda.synchronize()
    assert torch.allclose(d.float(), 2 * a.float(), rtol=2 ** -7, atol=1e-6)
    assert gqa_lib.gqa_get_device_status() == 0


def test_fp8_wide_group_nan_tail_and_edges(gqa_lib, oracle_mod, cuda_device):
    """G = 32: E4M3 NaN bytes past every sequence end (the converter warps
    must write zeros for those V rows), q x 8, an empty context and a clamped
    length in one batch."""
    w = W.DecodeWorkload("fp8_wide_edges", 6, 32, 1, 128, 1024, 1, 1024, 101)
    sl = torch.tensor([1024, 1, 700, 0, 5000, 333], dtype=torch.int32)
    q, k8, v8, ks, vs, _ = W.make_decode_fp8_inputs(w, q_mult=8.0)
    for b in range(6):
        n = int(sl[b].clamp(0, 1024))
        k8[b, :, n:, :] = W.E4M3_NAN
        v8[b, :, n:, :] = W.E4M3_NAN
    out, flags = run_fp8(gqa_lib, q, k8, v8, ks, vs, sl, w.scale, cuda_device)
    assert flags == (gqa_lib.GQA_DEV_EMPTY_CONTEXT | gqa_lib.GQA_DEV_SEQLEN_CLAMPED)
    assert np.all(out[3] == 0)
    ref = oracle_fp8(oracle_mod, q, k8, v8, ks, vs, sl.clamp(min=1, max=1024), w.scale)
    keep = [0, 1, 2, 4, 5]
    assert_parity(out[keep], ref[keep], "fp8 wide edges")


# ---- D = 64: rows of 64 E4M3 bytes (64-byte swizzle), G <= 8
@pytest.mark.parametrize("B,Hq,Hkv,Lmax,lens", [
    (2, 8, 2, 128, [128, 77]),            # the tiny decode shape
    (3, 8, 2, 700, [700, 333, 65]),       # ragged tails, many tiles
    (4, 4, 4, 257, [63, 64, 65, 257]),    # MHA endpoint; tile boundaries
    (2, 6, 2, 300, [300, 17]),            # G = 3
    (16, 32, 8, 2048, [2048] * 16),       # one CTA per pair, L2 prefetch at launch
])
def test_fp8_d64_shapes(gqa_lib, oracle_mod, cuda_device, B, Hq, Hkv, Lmax, lens):
    w = W.DecodeWorkload("fp8_d64", B, Hq, Hkv, 64, Lmax, 1, Lmax, 3100 + B * Hq + Lmax)
    q, k8, v8, ks, vs, _ = W.make_decode_fp8_inputs(w)
    sl = torch.tensor(lens, dtype=torch.int32)
    out, flags = run_fp8(gqa_lib, q, k8, v8, ks, vs, sl, w.scale, cuda_device)
    assert flags == 0
    assert_parity(out, oracle_fp8(oracle_mod, q, k8, v8, ks, vs, sl, w.scale), f"fp8 D=64 {B},{Hq},{Hkv},{lens}")


def test_fp8_d64_nan_tail_and_edges(gqa_lib, oracle_mod, cuda_device):
    """D = 64: E4M3 NaN bytes past every sequence end, q x 8, an empty
    context and a clamped length in one batch."""
    w = W.DecodeWorkload("fp8_d64_edges", 5, 16, 4, 64, 1024, 1, 1024, 98)
    sl = torch.tensor([1024, 1, 700, 0, 9999], dtype=torch.int32)
    q, k8, v8, ks, vs, _ = W.make_decode_fp8_inputs(w, q_mult=8.0)
    for b in range(5):
        n = int(sl[b].clamp(0, 1024))
        k8[b, :, n:, :] = W.E4M3_NAN
        v8[b, :, n:, :] = W.E4M3_NAN
    out, flags = run_fp8(gqa_lib, q, k8, v8, ks, vs, sl, w.scale, cuda_device)
    assert flags == (gqa_lib.GQA_DEV_EMPTY_CONTEXT | gqa_lib.GQA_DEV_SEQLEN_CLAMPED)
    assert np.all(out[3] == 0)
    ref = oracle_fp8(oracle_mod, q, k8, v8, ks, vs, sl.clamp(min=1, max=1024), w.scale)
    keep = [0, 1, 2, 4]
    assert_parity(out[keep], ref[keep], "fp8 D=64 edges")


def test_fp8_rejects_d64_wide_groups(gqa_lib, cuda_device):
    """D = 64 with 16 heads per KV head has no FP8 kernel."""
    w = W.DecodeWorkload("fp8_d64_g16", 2, 16, 1, 64, 128, 1, 128, 102)
    q = torch.zeros(2, 16, 64, dtype=torch.bfloat16, device=cuda_device)
    k8 = torch.zeros(2, 1, 128, 64, dtype=torch.uint8, device=cuda_device)
    sc = torch.ones(2, 1, device=cuda_device)
    sl = torch.full((2,), 128, dtype=torch.int32, device=cuda_device)
    with pytest.raises(gqa_lib.GQAError) as e:
        gqa_lib.gqa_decode_fp8(q, k8, k8, sc, sc, sl, scale=w.scale)
    assert e.value.status == gqa_lib.GQA_ERR_UNSUPPORTED


def test_fp8_max_batch(gqa_lib, oracle_mod, cuda_device):
    """B = 1024 short ragged sequences with an E4M3 cache (G = 4 and G = 32)."""
    for Hq, Hkv, Lmax in ((8, 2, 64), (32, 1, 256)):
        g = torch.Generator().manual_seed(91 + Hq)
        sl = torch.randint(1, Lmax + 1, (1024,), generator=g, dtype=torch.int32)
        w = W.DecodeWorkload("fp8_maxb", 1024, Hq, Hkv, 128, Lmax, 1, Lmax, 700 + Hq)
        q, k8, v8, ks, vs, _ = W.make_decode_fp8_inputs(w)
        out, flags = run_fp8(gqa_lib, q, k8, v8, ks, vs, sl, w.scale, cuda_device)
        assert flags == 0
        assert_parity(out, oracle_fp8(oracle_mod, q, k8, v8, ks, vs, sl, w.scale), f"fp8 max batch G={Hq // Hkv}")


@pytest.mark.parametrize("name,D,page_size", [
    ("llama3_8b", 128, 256),   # one CTA per pair: the launch-time prefetch walks the block table
    ("mqa", 128, 128),         # G = 32: the tcgen05 kernel's producer maps 128-key blocks to pages
    ("ragged_d64", 64, 64),    # D = 64, G = 4, ragged lengths
])
def test_fp8_paged_parity_and_bits(gqa_lib, oracle_mod, cuda_device, name, D, page_size):
    """gqa_decode_fp8_paged over E4M3 pages cut from the workload's cache in a
    seeded random order: bit-identical to gqa_decode_fp8 on the contiguous
    cache, and at the oracle's bar."""
    if name == "ragged_d64":
        w = W.DecodeWorkload("fp8_paged_d64", 5, 16, 4, D, 900, 1, 900, 3333)
    else:
        w = W.WORKLOADS[name]
    q, k8, v8, ks, vs, sl = W.make_decode_fp8_inputs(w)
    kp, vp, bt = W.page_cache(k8, v8, page_size, seed=w.seed + 77)
    d = cuda_device
    qd, ksd, vsd, sld = q.to(d), ks.to(d), vs.to(d), sl.to(d)
    out_p = gqa_lib.gqa_decode_fp8_paged(qd, kp.to(d), vp.to(d), ksd, vsd, bt.to(d), sld, scale=w.scale)
    assert gqa_lib.gqa_get_device_status() == 0
    out_c = gqa_lib.gqa_decode_fp8(qd, k8.to(d), v8.to(d), ksd, vsd, sld, scale=w.scale)
    assert gqa_lib.gqa_get_device_status() == 0
    assert torch.equal(out_p, out_c)
    assert_parity(out_p.double().cpu().numpy(), oracle_fp8(oracle_mod, q, k8, v8, ks, vs, sl, w.scale),
                  f"{name} fp8 paged")


def test_fp8_paged_bad_entry_is_flagged(gqa_lib, oracle_mod, cuda_device):
    """A needed block-table entry outside the pool sets GQA_DEV_BAD_PAGE; the
    other sequences stay exact (both kernels)."""
    d = cuda_device
    for Hq, page_size in ((8, 64), (32, 128)):
        w = W.DecodeWorkload("fp8_paged_bad", 4, Hq, 2, 128, 1000, 1, 1000, 4444 + Hq)
        q, k8, v8, ks, vs, _ = W.make_decode_fp8_inputs(w)
        sl = torch.tensor([1000, 37, 512, 800], dtype=torch.int32)
        kp, vp, bt = W.page_cache(k8, v8, page_size, seed=5)
        bt[2, 1] = 10 ** 6  # sequence 2 needs its second page
        out = gqa_lib.gqa_decode_fp8_paged(q.to(d), kp.to(d), vp.to(d), ks.to(d), vs.to(d), bt.to(d), sl.to(d),
                                           scale=w.scale)
        assert gqa_lib.gqa_get_device_status() == gqa_lib.GQA_DEV_BAD_PAGE
        ref = oracle_fp8(oracle_mod, q, k8, v8, ks, vs, sl, w.scale)
        o = out.double().cpu().numpy()
        assert np.isfinite(o).all()
        keep = [0, 1, 3]
        assert_parity(o[keep], ref[keep], f"fp8 paged G={Hq // 2}, other sequences")


def test_fp8_paged_nan_tail(gqa_lib, oracle_mod, cuda_device):
    """E4M3 NaN bytes in every row past a sequence's end, inside its pages:
    never read into the result (both kernels), equal to the contiguous call."""
    d = cuda_device
    for Hq, page_size in ((8, 64), (32, 128)):
        w = W.DecodeWorkload("fp8_paged_nan", 3, Hq, 2, 128, 700, 1, 700, 5555 + Hq)
        q, k8, v8, ks, vs, _ = W.make_decode_fp8_inputs(w)
        sl = torch.tensor([700, 1, 333], dtype=torch.int32)
        for b in range(3):
            n = int(sl[b])
            k8[b, :, n:, :] = W.E4M3_NAN
            v8[b, :, n:, :] = W.E4M3_NAN
        kp, vp, bt = W.page_cache(k8, v8, page_size, seed=9)
        args = (q.to(d), kp.to(d), vp.to(d), ks.to(d), vs.to(d), bt.to(d), sl.to(d))
        out = gqa_lib.gqa_decode_fp8_paged(*args, scale=w.scale)
        assert gqa_lib.gqa_get_device_status() == 0
        o = out.double().cpu().numpy()
        assert np.isfinite(o).all()
        ref = oracle_fp8(oracle_mod, q, k8, v8, ks, vs, sl, w.scale)
        assert_parity(o, ref, f"fp8 paged NaN tail G={Hq // 2}")
        out_c = gqa_lib.gqa_decode_fp8(q.to(d), k8.to(d), v8.to(d), ks.to(d), vs.to(d), sl.to(d), scale=w.scale)
        assert torch.equal(out, out_c)
