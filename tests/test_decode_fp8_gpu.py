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


@pytest.mark.parametrize("name", ["llama3_8b", "llama2_70b"])
def test_fp8_workload_parity_full(gqa_lib, oracle_mod, cuda_device, name):
    """Every output element of the Llama-shaped workloads with the cache in FP8."""
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


def test_fp8_scales_and_repeat(gqa_lib, cuda_device):
    """Doubling every V scale doubles the output (to bf16 rounding); two calls
    give identical bits; wide groups are rejected."""
    w = W.DecodeWorkload("fp8_scale", 4, 16, 2, 128, 600, 1, 600, 99)
    q, k8, v8, ks, vs, sl = [t.to(cuda_device) for t in W.make_decode_fp8_inputs(w)]
    a = gqa_lib.gqa_decode_fp8(q, k8, v8, ks, vs, sl).clone()
    b = gqa_lib.gqa_decode_fp8(q, k8, v8, ks, vs, sl).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    d = gqa_lib.gqa_decode_fp8(q, k8, v8, ks, 2 * vs, sl)
    torch.cuda.synchronize()
    assert torch.allclose(d.float(), 2 * a.float(), rtol=2 ** -7, atol=1e-6)
    wide = W.DecodeWorkload("fp8_wide", 2, 32, 1, 128, 256, 1, 256, 100)
    qw, k8w, v8w, ksw, vsw, slw = [t.to(cuda_device) for t in W.make_decode_fp8_inputs(wide)]
    with pytest.raises(gqa_lib.GQAError) as e:
        gqa_lib.gqa_decode_fp8(qw, k8w, v8w, ksw, vsw, slw)
    assert e.value.status == gqa_lib.GQA_ERR_UNSUPPORTED
