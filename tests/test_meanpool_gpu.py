"""gqa_meanpool_kv_heads (MHA -> GQA checkpoint conversion of a K/V
projection, the GQA paper notes on 51969.com, "Uptraining", figures 1 and 4)
through the C ABI against the fp64 oracle's meanpool_heads.

Bar: the kernel sums the group in fp32, divides once (correctly rounded) and
rounds to bf16; the fp32 sum can itself round when the group's values span
more than 24 bits, so the bf16 result is within one bf16 ulp of the exact
mean (a correctly rounded one would be within half an ulp): |gpu - oracle| <=
ulp_bf16(oracle) = 2^(floor(log2 |oracle|) - 7), and exact for a zero mean.
"First" copies bits and must be bit-exact, as must G = 1 (a copy through the
mean path: a sum of one value divided by 1)."""
import numpy as np
import pytest
import torch

from grouped_query_attention_09_b300 import workloads as W

pytestmark = pytest.mark.gpu


def _weights(H, rows, cols, seed, scale=0.02):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(H, rows, cols, generator=g) * scale).to(torch.bfloat16)


def _check_mean(got, want):
    got = got.double().cpu().numpy()
    err = np.abs(got - want)
    _, e = np.frexp(np.abs(want))  # |want| = m 2^e, m in [0.5, 1)
    bound = np.where(want == 0, 0.0, np.ldexp(1.0, np.maximum(e - 8, -133)))
    assert np.all(err <= bound), f"max excess {np.max(err - bound):.3e}"


@pytest.mark.parametrize("H,Hkv,rows,cols", [
    (32, 8, 128, 4096),   # Llama-3-8B K (or V) projection: 32 heads -> 8 groups, d_model 4096
    (64, 8, 128, 8192),   # Llama-2-70B shape: 64 -> 8
    (32, 1, 128, 4096),   # MHA -> MQA (figure 1)
    (12, 4, 64, 40),      # 3 heads per group, 16-byte chunks
    (6, 2, 5, 7),         # blocks of 35 values: the one-value-per-thread path
    (8, 8, 16, 24),       # G = 1
])
def test_meanpool_parity(gqa_lib, oracle_mod, cuda_device, H, Hkv, rows, cols):
    w = _weights(H, rows, cols, 9000 + H + cols)
    out = gqa_lib.gqa_meanpool_kv_heads(w.to(cuda_device), Hkv)
    torch.cuda.synchronize()
    want = oracle_mod.meanpool_heads(W.bf16_bits(w), Hkv)
    if H == Hkv:
        assert torch.equal(out.cpu(), w)
    _check_mean(out, want)


@pytest.mark.parametrize("H,Hkv,rows,cols", [(32, 8, 128, 4096), (6, 3, 5, 7)])
def test_first_head_is_bit_exact(gqa_lib, oracle_mod, cuda_device, H, Hkv, rows, cols):
    w = _weights(H, rows, cols, 9100 + cols)
    out = gqa_lib.gqa_meanpool_kv_heads(w.to(cuda_device), Hkv, mode="first").cpu()
    want = oracle_mod.meanpool_heads(W.bf16_bits(w), Hkv, mode="first")
    np.testing.assert_array_equal(out.double().numpy(), want)
    assert torch.equal(out, w[:: H // Hkv])


def test_bias_and_wide_range(gqa_lib, oracle_mod, cuda_device):
    # a bias (cols = 1) with values spread over many binades, and a group whose
    # heads cancel exactly
    g = torch.Generator().manual_seed(9200)
    b = (torch.randn(16, 128, 1, generator=g) * torch.logspace(-20, 20, 128).reshape(1, 128, 1)).to(torch.bfloat16)
    b[4:8] = torch.stack([b[4], -b[4], b[6], -b[6]])
    out = gqa_lib.gqa_meanpool_kv_heads(b.to(cuda_device), 4)
    want = oracle_mod.meanpool_heads(W.bf16_bits(b), 4)
    _check_mean(out, want)
    assert torch.all(out[1].cpu() == 0)


def test_converted_keys_match_the_group_mean(gqa_lib, cuda_device):
    # what the conversion is for: projecting x with the converted weight gives
    # (to the bf16 rounding of the weight) the mean of the group's keys
    H, Hkv, D, dm = 32, 8, 128, 512
    w = _weights(H, D, dm, 9300)
    x = torch.randn(64, dm, generator=torch.Generator().manual_seed(9301), dtype=torch.float64)
    out = gqa_lib.gqa_meanpool_kv_heads(w.to(cuda_device), Hkv).cpu().double()
    keys = torch.einsum("nc,hdc->hnd", x, w.double())
    for j in range(Hkv):
        ref = keys[j * 4:(j + 1) * 4].mean(dim=0)
        got = x @ out[j].T
        assert torch.allclose(got, ref, rtol=0, atol=2.0 ** -8 * float(ref.abs().max()) * 4)
