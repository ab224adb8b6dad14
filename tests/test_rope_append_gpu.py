"""gqa_rope_append (rotary embedding of the new token + cache append) through
the C ABI against the fp64 oracle's rope_append, at the bar of
tests/parity.py; the value row and every cache row other than the appended
one must be bit-exact, and seqlens must advance by exactly one."""
import numpy as np
import pytest
import torch

from grouped_query_attention_09_b300 import workloads as W
from parity import assert_parity

pytestmark = pytest.mark.gpu


def _inputs(B, Hq, Hkv, D, Lmax, lens, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16)
    kn = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    vn = torch.randn(B, Hkv, D, generator=g).to(torch.bfloat16)
    kc = torch.randn(B, Hkv, Lmax, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(B, Hkv, Lmax, D, generator=g).to(torch.bfloat16)
    sl = torch.tensor(lens, dtype=torch.int32)
    return q, kn, vn, kc, vc, sl


@pytest.mark.parametrize("B,Hq,Hkv,D,Lmax,lens", [
    (16, 32, 8, 128, 4097, [4096] * 15 + [0]),              # Llama-3-8B shape, one empty sequence
    (4, 64, 8, 128, 16384, [16000, 4095, 1, 12345]),         # long positions
    (3, 8, 2, 64, 300, [17, 299, 150]),                      # D = 64
    (2, 4, 4, 128, 64, [63, 64]),                            # MHA; the second cache is full
])
def test_rope_append_parity(gqa_lib, oracle_mod, cuda_device, B, Hq, Hkv, D, Lmax, lens):
    q, kn, vn, kc, vc, sl = _inputs(B, Hq, Hkv, D, Lmax, lens, 4000 + B + Lmax)
    dev = cuda_device
    qd, knd, vnd, kcd, vcd, sld = (t.to(dev) for t in (q, kn, vn, kc, vc, sl))
    q_out = gqa_lib.gqa_rope_append(qd, knd, vnd, kcd, vcd, sld)
    flags = gqa_lib.gqa_get_device_status()
    full = [i for i, n in enumerate(lens) if n >= Lmax]
    assert flags == (gqa_lib.GQA_DEV_CACHE_FULL if full else 0)
    qo, ko, vo = oracle_mod.rope_append(W.bf16_bits(q), W.bf16_bits(kn), W.bf16_bits(vn),
                                        np.minimum(lens, Lmax), Lmax=10 ** 9)
    assert_parity(q_out.double().cpu().numpy(), qo, "q_out")
    kcn, vcn = kcd.cpu(), vcd.cpu()
    new_len = sld.cpu()
    for b, n in enumerate(lens):
        if n >= Lmax:
            assert int(new_len[b]) == n
            assert torch.equal(kcn[b], kc[b]) and torch.equal(vcn[b], vc[b])
            continue
        assert int(new_len[b]) == n + 1
        assert_parity(kcn[b, :, n].double().numpy(), ko[b], f"k row b={b}")
        assert torch.equal(vcn[b, :, n], vn[b])
        keep = [t for t in range(Lmax) if t != n]
        assert torch.equal(kcn[b, :, keep], kc[b, :, keep]) and torch.equal(vcn[b, :, keep], vc[b, :, keep])


def test_rope_append_in_place_then_decode(gqa_lib, oracle_mod, cuda_device):
    """Append the new token (q rotated in place), then decode over the grown
    cache: equals the oracle's rotation followed by its decode."""
    B, Hq, Hkv, D, Lmax = 4, 32, 8, 128, 2048
    lens = [2047, 1000, 1, 1500]
    q, kn, vn, kc, vc, sl = _inputs(B, Hq, Hkv, D, Lmax, lens, 4100)
    dev = cuda_device
    qd, knd, vnd, kcd, vcd, sld = (t.to(dev) for t in (q, kn, vn, kc, vc, sl))
    gqa_lib.gqa_rope_append(qd, knd, vnd, kcd, vcd, sld, q_out=qd)
    out = gqa_lib.gqa_decode(qd, kcd, vcd, sld)
    assert gqa_lib.gqa_get_device_status() == 0
    qo, ko, vo = oracle_mod.rope_append(W.bf16_bits(q), W.bf16_bits(kn), W.bf16_bits(vn), lens, Lmax=Lmax)
    kref = kc.double().numpy().copy()
    vref = vc.double().numpy().copy()
    for b, n in enumerate(lens):
        kref[b, :, n] = ko[b]
        vref[b, :, n] = vo[b]
    ref = oracle_mod.decode(qo, kref, vref, np.array(lens) + 1, D ** -0.5)
    assert_parity(out.double().cpu().numpy(), ref, "append + decode")
