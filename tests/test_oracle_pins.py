"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test names the passage it follows.  The pins are chosen so that a
plausible slip in the oracle fails at least one of them:

* a wrong head -> KV-head map (h mod Hkv instead of h div G): group-constant V,
  library SDPA with enable_gqa, materialised repeat_interleave;
* a dropped or wrong scale, a transposed operand: library SDPA, the two-key
  logistic closed form;
* a missing normalisation: constant V;
* a causal diagonal off by one / a mask that leaks the future: row 0 = v_0,
  the i/2 staircase, future-perturbation invariance;
* reading cache rows past seqlens[b]: the NaN-tail test;
* a lossy bf16 widening: exact bit patterns;
* a rotary embedding with the wrong pairing ((2i, 2i + 1) instead of
  (i, i + D/2)) or the wrong rate (base^(-i/D)): the basis-vector closed form
  and an independent numpy rotate-half statement (both slips are planted and
  shown to fail).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from grouped_query_attention_09_b300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore")


def bf16(a):
    """Rounds an fp64 array to bf16 (RNE) and returns (bits uint16, exact fp64 values)."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return W.bf16_bits(t), t.double().numpy()


def rnd(shape, seed, mult=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * mult


def sdpa(q, k, v, causal=False, scale=None):
    """torch fp64 scaled_dot_product_attention with grouped K/V (a library routine)."""
    return F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
                                          is_causal=causal, scale=scale, enable_gqa=True).numpy()


# ----------------------------------------------------------- library cross-checks
@pytest.mark.parametrize("B,Hq,Hkv,L,D", [(1, 4, 4, 5, 3), (2, 8, 2, 7, 4), (1, 6, 1, 9, 8), (3, 8, 4, 1, 5),
                                          (2, 12, 3, 16, 16)])
@pytest.mark.parametrize("causal", [False, True])
def test_prefill_matches_torch_sdpa_gqa(oracle_mod, B, Hq, Hkv, L, D, causal):
    """Scaled dot-product attention of the Huawei Cloud post (section 5 code)
    with one K/V head per group; torch's fp64 SDPA with enable_gqa is an
    independent implementation of the same definition."""
    _, q = bf16(rnd((B, Hq, L, D), 1))
    _, k = bf16(rnd((B, Hkv, L, D), 2))
    _, v = bf16(rnd((B, Hkv, L, D), 3))
    got = oracle_mod.prefill(q, k, v, causal=causal)
    ref = sdpa(q, k, v, causal=causal, scale=1 / math.sqrt(D))
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,D", [(2, 8, 2, 9, 4), (3, 4, 1, 6, 3), (1, 4, 4, 12, 8)])
def test_decode_matches_materialised_repeat_interleave(oracle_mod, B, Hq, Hkv, Lmax, D):
    """The GQA module of "手把手教你用PyTorch实现GQA" (section 1.3) and
    `repeat_kv` of the GQA paper notes expand K/V with repeat_interleave over
    the head axis; after that the computation is plain multi-head attention."""
    _, q = bf16(rnd((B, Hq, D), 4, 2.0))
    _, k = bf16(rnd((B, Hkv, Lmax, D), 5))
    _, v = bf16(rnd((B, Hkv, Lmax, D), 6))
    seqlens = np.array([Lmax - b for b in range(B)], dtype=np.int32)
    scale = 0.37
    got = oracle_mod.decode(q, k, v, seqlens, scale)
    kx = np.repeat(k, Hq // Hkv, axis=1)  # repeat_interleave on dim 1
    vx = np.repeat(v, Hq // Hkv, axis=1)
    for b in range(B):
        n = seqlens[b]
        ref = F.scaled_dot_product_attention(torch.from_numpy(q[b][:, None, :]), torch.from_numpy(kx[b, :, :n]),
                                             torch.from_numpy(vx[b, :, :n]), scale=scale).numpy()[:, 0, :]
        np.testing.assert_allclose(got[b], ref, rtol=0, atol=1e-13)


def test_huawei_demo_shapes(oracle_mod):
    """The two demos of the Huawei Cloud post: d_model 12 with 4 heads (head
    size 3) and d_model 32 with 8 heads in groups of 2 (head size 4); a 5-token
    pass with the cache on (no mask: `masked` defaults to False) then two
    single-token steps that see the whole cache."""
    for Hq, D, per_group, seed in ((4, 3, 1, 10), (8, 4, 2, 11)):
        Hkv = Hq // per_group
        _, q5 = bf16(rnd((1, Hq, 5, D), seed))
        _, k7 = bf16(rnd((1, Hkv, 7, D), seed + 1))
        _, v7 = bf16(rnd((1, Hkv, 7, D), seed + 2))
        _, qd = bf16(rnd((1, Hq, 2, D), seed + 3))
        out5 = oracle_mod.prefill(q5, k7[:, :, :5].copy(), v7[:, :, :5].copy(), causal=False)
        np.testing.assert_allclose(out5, sdpa(q5, k7[:, :, :5], v7[:, :, :5]), atol=1e-13, rtol=0)
        for step, n in ((0, 6), (1, 7)):
            o = oracle_mod.decode(qd[:, :, step, :].copy(), k7, v7, np.array([n], np.int32))
            ref = sdpa(qd[:, :, step:step + 1, :], k7[:, :, :n], v7[:, :, :n])[:, :, 0, :]
            np.testing.assert_allclose(o, ref, atol=1e-13, rtol=0)


# ----------------------------------------------------------- closed forms
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (6, 3), (4, 4), (8, 1)])
def test_group_constant_values_pin_head_to_group_map(oracle_mod, Hq, Hkv):
    """Group j's V rows all equal j+1: whatever the weights, head h returns
    exactly (h div G) + 1 -- the grouping `head_index // n_head_per_group` of
    the Huawei Cloud post (section 5) and repeat_interleave of section 1.3 of
    the bjdmk page; the tiling map h mod Hkv would give a different answer."""
    B, Lmax, D = 2, 11, 4
    _, q = bf16(rnd((B, Hq, D), 20, 3.0))
    _, k = bf16(rnd((B, Hkv, Lmax, D), 21))
    v = np.zeros((B, Hkv, Lmax, D))
    for j in range(Hkv):
        v[:, j] = j + 1
    out = oracle_mod.decode(q, k, v, np.array([Lmax, 5], np.int32))
    G = Hq // Hkv
    for h in range(Hq):
        np.testing.assert_allclose(out[:, h, :], h // G + 1, rtol=1e-14, atol=0)
    outp = oracle_mod.prefill(np.repeat(q[:, :, None, :], Lmax, axis=2), k, v, causal=True)
    for h in range(Hq):
        np.testing.assert_allclose(outp[:, h], h // G + 1, rtol=1e-14, atol=0)


def test_constant_values_pin_normalisation(oracle_mod):
    """Softmax rows sum to one (Huawei Cloud post, softmax over dim -1), so a
    constant V comes back unchanged."""
    _, q = bf16(rnd((2, 4, 3, 8), 30, 4.0))
    _, k = bf16(rnd((2, 2, 3, 8), 31))
    v = np.full((2, 2, 3, 8), -1.75)
    for causal in (False, True):
        np.testing.assert_allclose(oracle_mod.prefill(q, k, v, causal=causal), -1.75, rtol=1e-14, atol=0)


def test_single_key_returns_v_exactly(oracle_mod):
    """softmax of a single logit is exactly 1: a one-key context returns V."""
    _, q = bf16(rnd((3, 4, 8), 40, 5.0))
    _, k = bf16(rnd((3, 2, 6, 8), 41))
    _, v = bf16(rnd((3, 2, 6, 8), 42))
    out = oracle_mod.decode(q, k, v, np.array([1, 1, 1], np.int32))
    for h in range(4):
        np.testing.assert_array_equal(out[:, h], v[:, h // 2, 0])


def test_two_key_logistic_closed_form(oracle_mod):
    """Two keys: the weight of key 0 is the logistic function of the scaled
    logit gap, sigma(scale (a - b)), with a = <q,k0>, b = <q,k1>."""
    D = 4
    q = np.array([[[1.0, 0.5, -2.0, 0.25]]])
    k = np.array([[[[0.5, 1.0, 0.0, 2.0], [-1.0, 0.0, 0.5, 1.0]]]])
    v = np.array([[[[1.0, 2.0, 3.0, 4.0], [-4.0, 0.0, 8.0, 0.5]]]])
    a = float(q[0, 0] @ k[0, 0, 0])
    b = float(q[0, 0] @ k[0, 0, 1])
    for scale in (0.5, 1.0 / math.sqrt(D), 3.0):
        w0 = 1.0 / (1.0 + math.exp(-scale * (a - b)))
        ref = w0 * v[0, 0, 0] + (1 - w0) * v[0, 0, 1]
        got = oracle_mod.decode(q, k, v, np.array([2], np.int32), scale)
        np.testing.assert_allclose(got[0, 0], ref, rtol=1e-14, atol=1e-15)


def test_zero_query_gives_mean_of_visible_values(oracle_mod):
    """q = 0 makes every logit 0: the weights are uniform over visible keys."""
    _, k = bf16(rnd((1, 1, 9, 4), 50))
    _, v = bf16(rnd((1, 1, 9, 4), 51))
    q = np.zeros((1, 3, 4))
    out = oracle_mod.decode(q, k, v, np.array([6], np.int32))
    for h in range(3):
        np.testing.assert_allclose(out[0, h], v[0, 0, :6].mean(axis=0), rtol=1e-14, atol=1e-15)


def test_dominant_logit_selects_its_value(oracle_mod):
    """One logit 50 above all others: its weight is 1 - O(e^-50)."""
    D, n = 4, 7
    q = np.zeros((1, 1, D)); q[0, 0, 0] = 1.0
    k = np.zeros((1, 1, n, D)); k[0, 0, 3, 0] = 50.0
    _, v = bf16(rnd((1, 1, n, D), 60))
    out = oracle_mod.decode(q, k, v, np.array([n], np.int32), 1.0)
    np.testing.assert_allclose(out[0, 0], v[0, 0, 3], rtol=0, atol=1e-12)


def test_causal_staircase(oracle_mod):
    """Causal mask triu(ones, diagonal=1) -> -inf (Huawei Cloud post): with
    K = 0 every visible key weighs the same, so with V[t] = t row i returns
    the mean of 0..i = i/2 -- the diagonal key is visible, later ones are not.
    Row 0 returns v_0 exactly."""
    L, D = 9, 3
    _, q = bf16(rnd((1, 2, L, D), 70, 2.0))
    k = np.zeros((1, 1, L, D))
    v = np.repeat(np.arange(L, dtype=np.float64)[None, None, :, None], D, axis=3)
    out = oracle_mod.prefill(q, k, v, causal=True)
    for i in range(L):
        np.testing.assert_allclose(out[0, :, i], i / 2, rtol=1e-14, atol=1e-15)
    _, k2 = bf16(rnd((1, 1, L, D), 71))
    _, v2 = bf16(rnd((1, 1, L, D), 72))
    out2 = oracle_mod.prefill(q, k2, v2, causal=True)
    np.testing.assert_array_equal(out2[0, :, 0], np.repeat(v2[0, :, 0], 2, axis=0))


def test_causal_rows_ignore_future_keys(oracle_mod):
    """Changing K/V at positions t > i leaves row i unchanged (bit for bit)."""
    L, D = 10, 8
    _, q = bf16(rnd((2, 4, L, D), 80))
    _, k = bf16(rnd((2, 2, L, D), 81))
    _, v = bf16(rnd((2, 2, L, D), 82))
    base = oracle_mod.prefill(q, k, v, causal=True)
    for i in (0, 3, 8):
        k2, v2 = k.copy(), v.copy()
        k2[:, :, i + 1:] = 1e3
        v2[:, :, i + 1:] = -7.0
        pert = oracle_mod.prefill(q, k2, v2, causal=True)
        np.testing.assert_array_equal(pert[:, :, : i + 1], base[:, :, : i + 1])


# ----------------------------------------------------------- invariants
def test_mha_endpoint_is_per_head_attention(oracle_mod):
    """GQA-H (Hkv = Hq) is MHA (GQA paper notes): each head is an independent
    single-head attention over its own K/V."""
    B, H, L, D = 2, 4, 6, 8
    _, q = bf16(rnd((B, H, L, D), 90))
    _, k = bf16(rnd((B, H, L, D), 91))
    _, v = bf16(rnd((B, H, L, D), 92))
    full = oracle_mod.prefill(q, k, v, causal=True)
    for h in range(H):
        one = oracle_mod.prefill(q[:, h:h + 1].copy(), k[:, h:h + 1].copy(), v[:, h:h + 1].copy(), causal=True)
        np.testing.assert_array_equal(full[:, h:h + 1], one)


def test_mqa_endpoint_is_broadcast(oracle_mod):
    """GQA-1 is MQA (GQA paper notes; the MQA module of the bjdmk page
    broadcasts one K/V head with unsqueeze(1)): Hkv = 1 equals MHA on the
    K/V head copied to every query head."""
    B, H, Lmax, D = 2, 6, 8, 4
    _, q = bf16(rnd((B, H, D), 93))
    _, k = bf16(rnd((B, 1, Lmax, D), 94))
    _, v = bf16(rnd((B, 1, Lmax, D), 95))
    sl = np.array([8, 3], np.int32)
    mqa = oracle_mod.decode(q, k, v, sl)
    mha = oracle_mod.decode(q, np.repeat(k, H, axis=1), np.repeat(v, H, axis=1), sl)
    np.testing.assert_array_equal(mqa, mha)


def test_decode_is_last_row_of_causal_prefill(oracle_mod):
    """A decode step of the token at position n-1 over n cached keys is row
    n-1 of a causal pass over those n tokens."""
    B, Hq, Hkv, n, D = 2, 8, 2, 7, 8
    _, q = bf16(rnd((B, Hq, n, D), 96))
    _, k = bf16(rnd((B, Hkv, n, D), 97))
    _, v = bf16(rnd((B, Hkv, n, D), 98))
    pre = oracle_mod.prefill(q, k, v, causal=True)
    dec = oracle_mod.decode(q[:, :, n - 1, :].copy(), k, v, np.array([n, n], np.int32))
    np.testing.assert_allclose(dec, pre[:, :, n - 1], rtol=0, atol=1e-15)


def test_nan_tail_is_not_read(oracle_mod):
    """Rows at or past seqlens[b] are outside the context: NaN there changes nothing."""
    B, Hq, Hkv, Lmax, D = 2, 4, 2, 10, 8
    _, q = bf16(rnd((B, Hq, D), 99))
    _, k = bf16(rnd((B, Hkv, Lmax, D), 100))
    _, v = bf16(rnd((B, Hkv, Lmax, D), 101))
    sl = np.array([4, 10], np.int32)
    clean = oracle_mod.decode(q, k, v, sl)
    k[0, :, 4:] = np.nan
    v[0, :, 4:] = np.nan
    np.testing.assert_array_equal(oracle_mod.decode(q, k, v, sl), clean)


def test_empty_context_is_flagged_and_zero(oracle_mod):
    _, q = bf16(rnd((2, 2, 4), 102))
    _, k = bf16(rnd((2, 1, 3, 4), 103))
    out = oracle_mod.decode(q, k, k, np.array([0, 3], np.int32), check=False)
    assert np.all(out[0] == 0)
    with pytest.raises(ValueError):
        oracle_mod.decode(q, k, k, np.array([0, 3], np.int32))


def test_bf16_widening_is_exact(oracle_mod):
    """bf16 inputs given as bit patterns give the same result as their exact
    fp64 values (0x3F80 = 1.0, 0xC020 = -2.5, 0x3E00 = 0.125, 0x4120 = 10.0)."""
    bits = np.array([0x3F80, 0xC020, 0x3E00, 0x4120], dtype=np.uint16)
    vals = np.array([1.0, -2.5, 0.125, 10.0])
    q_b = bits.reshape(1, 1, 4); q_f = vals.reshape(1, 1, 4)
    k_b = np.tile(bits, 3).reshape(1, 1, 3, 4); k_f = np.tile(vals, 3).reshape(1, 1, 3, 4)
    v_b = np.roll(k_b, 1); v_f = np.roll(k_f, 1)
    a = oracle_mod.decode(q_b, k_b, v_b, np.array([3], np.int32), 0.01)
    b = oracle_mod.decode(q_f, k_f, v_f, np.array([3], np.int32), 0.01)
    np.testing.assert_array_equal(a, b)


def test_sampled_rows_equal_full_evaluation(oracle_mod):
    """Evaluating a subset of rows gives the same rows as the full pass."""
    w = W.DecodeWorkload("t", 3, 8, 2, 16, 20, 5, 20, 7)
    q, k, v, sl = W.make_decode_inputs(w)
    full = oracle_mod.decode(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), sl.numpy())
    rows = np.array([[2, 7], [0, 0], [1, 3]])
    part = oracle_mod.decode(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), sl.numpy(), rows=rows)
    for r, (b, h) in enumerate(rows):
        np.testing.assert_array_equal(part[r], full[b, h])
    qp, kp, vp = W.make_prefill_inputs(W.PrefillWorkload("p", 1, 9, 4, 2, 8, True, 8))
    fullp = oracle_mod.prefill(W.bf16_bits(qp), W.bf16_bits(kp), W.bf16_bits(vp))
    rows3 = np.array([[0, 3, 8], [0, 0, 0], [0, 2, 4]])
    partp = oracle_mod.prefill(W.bf16_bits(qp), W.bf16_bits(kp), W.bf16_bits(vp), rows=rows3)
    for r, (b, h, i) in enumerate(rows3):
        np.testing.assert_array_equal(partp[r], fullp[b, h, i])


# ---- FP8 E4M3 cache (decode_fp8) --------------------------------------------

def test_e4m3_decoding_matches_torch_on_all_bytes(oracle_mod):
    """The oracle's E4M3 decoding against torch's float8_e4m3fn (a library
    routine) on every byte value."""
    b = np.arange(256, dtype=np.uint8)
    mine = oracle_mod.e4m3_values(b)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_e4m3_closed_forms(oracle_mod):
    """Format definition: bias 7, 3 mantissa bits, subnormals m/8 * 2^-6,
    S.1111.111 NaN, largest 448."""
    vals = oracle_mod.e4m3_values(np.array([0x38, 0xB8, 0x7E, 0x08, 0x01, 0x07, 0x00, 0x80, 0x3C], dtype=np.uint8))
    assert list(vals) == [1.0, -1.0, 448.0, 2.0 ** -6, 2.0 ** -9, 7 * 2.0 ** -9, 0.0, -0.0, 1.5]
    assert np.isnan(oracle_mod.e4m3_values(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def _fp8_case(seed, B=3, Hq=8, Hkv=2, D=16, Lmax=40):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, D, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, Lmax, D, generator=g)
    v = torch.randn(B, Hkv, Lmax, D, generator=g)
    k8 = (k * 40).clamp(-448, 448).to(torch.float8_e4m3fn)
    v8 = (v * 40).clamp(-448, 448).to(torch.float8_e4m3fn)
    ks = torch.rand(B, Hkv, generator=g, dtype=torch.float64) * 0.05 + 0.01
    vs = torch.rand(B, Hkv, generator=g, dtype=torch.float64) * 0.05 + 0.01
    sl = torch.tensor([Lmax, 1, 17][:B], dtype=torch.int32)
    return q, k8, v8, ks, vs, sl


def test_decode_fp8_equals_decode_of_dequantized_cache(oracle_mod):
    """decode_fp8 = decode over the cache dequantised by torch (fp8 -> fp64,
    times the per-(b, kv head) scale): the scales are applied per head."""
    q, k8, v8, ks, vs, sl = _fp8_case(11)
    kd = k8.double() * ks[:, :, None, None]
    vd = v8.double() * vs[:, :, None, None]
    a = oracle_mod.decode_fp8(q.numpy(), k8.view(torch.uint8).numpy(), v8.view(torch.uint8).numpy(),
                              ks.numpy(), vs.numpy(), sl.numpy(), 0.3)
    b = oracle_mod.decode(q.numpy(), kd.numpy(), vd.numpy(), sl.numpy(), 0.3)
    assert np.array_equal(a, b)


def test_decode_fp8_scale_identities(oracle_mod):
    """Doubling a head's V scale doubles its output exactly; multiplying its K
    scale by c is the same as multiplying the logit scale by c."""
    q, k8, v8, ks, vs, sl = _fp8_case(12)
    k8u, v8u = k8.view(torch.uint8).numpy(), v8.view(torch.uint8).numpy()
    base = oracle_mod.decode_fp8(q.numpy(), k8u, v8u, ks.numpy(), vs.numpy(), sl.numpy(), 0.25)
    dbl = oracle_mod.decode_fp8(q.numpy(), k8u, v8u, ks.numpy(), 2 * vs.numpy(), sl.numpy(), 0.25)
    assert np.array_equal(dbl, 2 * base)
    kc = oracle_mod.decode_fp8(q.numpy(), k8u, v8u, 4 * ks.numpy(), vs.numpy(), sl.numpy(), 0.25)
    sc = oracle_mod.decode_fp8(q.numpy(), k8u, v8u, ks.numpy(), vs.numpy(), sl.numpy(), 1.0)
    np.testing.assert_allclose(kc, sc, rtol=1e-12, atol=1e-12)
    # group map: head h reads KV head h // G (group-constant V makes it visible)
    v8c = np.zeros_like(v8u)
    v8c[:, 0] = 0x38   # 1.0
    v8c[:, 1] = 0x40   # 2.0
    out = oracle_mod.decode_fp8(q.numpy(), k8u, v8c, ks.numpy(), np.ones((3, 2)), sl.numpy(), 0.25)
    for h in range(8):
        np.testing.assert_allclose(out[:, h, :], 1.0 + (h // 4), rtol=0, atol=1e-12)


# ---- rotary embedding of the new token + cache append (rope_append) ---------

def _rope(oracle_mod, x, pos, base=10000.0):
    """Rotate rows x [n, D] (fp64) at integer positions pos [n] with the oracle."""
    n, D = x.shape
    qo, _, _ = oracle_mod.rope_append(x.reshape(n, 1, D), np.zeros((n, 1, D)), np.zeros((n, 1, D)),
                                      np.asarray(pos, dtype=np.int32), Lmax=1 << 30, base=base)
    return qo.reshape(n, D)


def test_rope_position_zero_is_identity(oracle_mod):
    x = np.random.default_rng(1).standard_normal((5, 64))
    assert np.array_equal(_rope(oracle_mod, x, [0] * 5), x)


def test_rope_preserves_pair_norms(oracle_mod):
    """Each (x_i, x_{i+D/2}) pair is rotated, so its length is unchanged."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 128))
    y = _rope(oracle_mod, x, rng.integers(0, 20000, 7))
    h = 64
    np.testing.assert_allclose(np.hypot(y[:, :h], y[:, h:]), np.hypot(x[:, :h], x[:, h:]), rtol=1e-12)
    assert not np.allclose(y, x)


def test_rope_composition_adds_angles(oracle_mod):
    """Rotating at a then at b equals rotating at a + b."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 32))
    a = rng.integers(0, 500, 6)
    b = rng.integers(0, 500, 6)
    np.testing.assert_allclose(_rope(oracle_mod, _rope(oracle_mod, x, a), b), _rope(oracle_mod, x, a + b),
                               rtol=1e-9, atol=1e-9)


def test_rope_scores_depend_only_on_relative_position(oracle_mod):
    """<rope(q, m), rope(k, n)> depends on m - n only -- the property the
    rotary embedding is built for."""
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 128))
    k = rng.standard_normal((1, 128))
    vals = []
    for m, n in [(10, 3), (107, 100), (5007, 5000)]:
        vals.append(float((_rope(oracle_mod, q, [m]) @ _rope(oracle_mod, k, [n]).T)[0, 0]))
    np.testing.assert_allclose(vals, vals[0], rtol=1e-9)
    other = float((_rope(oracle_mod, q, [11]) @ _rope(oracle_mod, k, [3]).T)[0, 0])
    assert abs(other - vals[0]) > 1e-6


# The next pins fix the two conventions the pages leave open (the GQA paper
# notes, "QA 相关", call apply_rotary_pos_emb without defining it; the reading
# taken is the Llama "rotate half" form): WHICH coordinates form a rotated pair
# -- (i, i + D/2), not (2i, 2i + 1) -- and the angular rate of pair i,
# base^(-2i/D), not base^(-i/D).  The identity / norm / composition /
# relative-position pins above hold for any pairing and any rate, so they
# cannot tell these apart.  Each check below is written as a function of the
# rotation under test, and the last test plants both plausible slips (as
# numpy stand-ins for a mistaken oracle) to show that each one fails.

def _theta(D, base):
    return base ** (-2.0 * np.arange(D // 2) / D)


def _basis_closed_form_errors(rope, D, base, positions):
    """Largest deviation of rope(e_j, p) from the rotate-half closed form over
    every basis vector e_j and the given positions: for i < D/2,
      e_i        -> cos(p t_i) e_i + sin(p t_i) e_{i+D/2}
      e_{i+D/2}  -> -sin(p t_i) e_i + cos(p t_i) e_{i+D/2},   t_i = base^(-2i/D)."""
    h = D // 2
    eye = np.eye(D)
    worst = 0.0
    for p in positions:
        y = rope(eye, [p] * D, base)  # row j = image of e_j
        ang = p * _theta(D, base)
        want = np.zeros((D, D))
        idx = np.arange(h)
        want[idx, idx] = np.cos(ang)
        want[idx, idx + h] = np.sin(ang)
        want[idx + h, idx] = -np.sin(ang)
        want[idx + h, idx + h] = np.cos(ang)
        worst = max(worst, float(np.abs(y - want).max()))
    return worst


def _numpy_rotate_half(x, pos, base):
    """The Llama statement, written independently of the oracle: a table of
    angles pos x inv_freq by np.outer, duplicated over both halves, then
    x * cos + rotate_half(x) * sin with rotate_half(x) = [-x2, x1]."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    inv_freq = 1.0 / (base ** (np.arange(0, D, 2, dtype=np.float64) / D))
    ang = np.outer(np.asarray(pos, dtype=np.float64), inv_freq)
    emb = np.concatenate([ang, ang], axis=-1)
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    rot = np.concatenate([-x2, x1], axis=-1)
    return x * np.cos(emb) + rot * np.sin(emb)


def _oracle_rope(oracle_mod):
    return lambda x, pos, base: _rope(oracle_mod, np.asarray(x, dtype=np.float64), pos, base)


_CONV_CASES = [(8, 10000.0, [1, 3, 77]), (16, 500.0, [2, 1000]), (64, 10000.0, [1, 4095]),
               (128, 10000.0, [1, 5, 16000]), (128, 1e6, [7, 131071])]


@pytest.mark.parametrize("D,base,positions", _CONV_CASES)
def test_rope_basis_vectors_closed_form(oracle_mod, D, base, positions):
    """Pins the pairing (i, i + D/2) and the rate base^(-2i/D) exactly: the
    image of every basis vector is one cos/sin pair at a known place (the
    bound allows the rounding of angles up to ~1.3e5 rad)."""
    assert _basis_closed_form_errors(_oracle_rope(oracle_mod), D, base, positions) < 1e-10


@pytest.mark.parametrize("D,base", [(16, 10000.0), (128, 10000.0), (128, 500000.0), (256, 10000.0)])
def test_rope_matches_numpy_rotate_half(oracle_mod, D, base):
    rng = np.random.default_rng(D)
    x = rng.standard_normal((9, D))
    pos = rng.integers(0, 20000, 9)
    np.testing.assert_allclose(_rope(oracle_mod, x, pos, base), _numpy_rotate_half(x, pos, base),
                               rtol=0, atol=1e-10)


def _mistaken_adjacent_pairs(x, pos, base):
    """Slip 1: GPT-J style pairs (2i, 2i + 1) at rate base^(-2i/D)."""
    x = np.asarray(x, dtype=np.float64).copy()
    D = x.shape[-1]
    ang = np.outer(np.asarray(pos, dtype=np.float64), _theta(D, base))
    a, b = x[..., 0::2].copy(), x[..., 1::2].copy()
    x[..., 0::2] = a * np.cos(ang) - b * np.sin(ang)
    x[..., 1::2] = b * np.cos(ang) + a * np.sin(ang)
    return x


def _mistaken_rate(x, pos, base):
    """Slip 2: rotate-half pairs at rate base^(-i/D)."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    ang = np.outer(np.asarray(pos, dtype=np.float64), base ** (-np.arange(D // 2) / D))
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    return np.concatenate([x1 * np.cos(ang) - x2 * np.sin(ang), x2 * np.cos(ang) + x1 * np.sin(ang)], axis=-1)


@pytest.mark.parametrize("mistake", [_mistaken_adjacent_pairs, _mistaken_rate])
def test_rope_convention_pins_catch_planted_slips(oracle_mod, mistake):
    """Each plausible slip passes the convention-blind pins (identity at p = 0,
    pair norms up to its own pairing, composition) yet fails both pins above."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal((4, 32))
    assert np.array_equal(mistake(x, [0] * 4, 10000.0), x)  # it is a rotation too
    a, b = rng.integers(0, 500, 4), rng.integers(0, 500, 4)
    np.testing.assert_allclose(mistake(mistake(x, a, 10000.0), b, 10000.0), mistake(x, a + b, 10000.0),
                               rtol=1e-9, atol=1e-9)
    for D, base, positions in _CONV_CASES:
        assert _basis_closed_form_errors(mistake, D, base, positions) > 1e-3
    pos = rng.integers(1, 20000, 4)
    assert np.abs(mistake(x, pos, 10000.0) - _numpy_rotate_half(x, pos, 10000.0)).max() > 1e-3
    # and the oracle itself is not one of them
    assert _basis_closed_form_errors(_oracle_rope(oracle_mod), 32, 10000.0, [3]) < 1e-12


def test_rope_append_rows_and_full_cache(oracle_mod):
    """Each batch uses its own position; V passes through; a full cache is
    reported (code 4)."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((2, 4, 16))
    k = rng.standard_normal((2, 2, 16))
    v = rng.standard_normal((2, 2, 16))
    qo, ko, vo = oracle_mod.rope_append(q, k, v, [0, 9], Lmax=10)
    assert np.array_equal(vo, v)
    assert np.array_equal(qo[0], q[0]) and np.array_equal(ko[0], k[0])
    np.testing.assert_allclose(ko[1], _rope(oracle_mod, k[1], [9, 9]), rtol=0, atol=0)
    with pytest.raises(ValueError):
        oracle_mod.rope_append(q, k, v, [0, 10], Lmax=10)


# ---- paged cache (decode_paged) --------------------------------------------

def test_decode_paged_equals_decode_on_the_gathered_cache(oracle_mod):
    """The paged decode reads exactly the rows the block table names: it equals
    the contiguous decode on the cache the pages were cut from, and on the
    cache gathered back from the pool by numpy indexing (a library routine)."""
    B, Hq, Hkv, D, Lmax, ps = 3, 8, 2, 16, 70, 32
    g = torch.Generator().manual_seed(21)
    q = torch.randn(B, Hq, D, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, Lmax, D, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, Lmax, D, generator=g, dtype=torch.float64)
    sl = np.array([70, 1, 33], dtype=np.int32)
    kp, vp, bt = W.page_cache(k, v, ps, seed=5)
    paged = oracle_mod.decode_paged(q.numpy(), kp.numpy(), vp.numpy(), bt.numpy(), sl, 0.25)
    cont = oracle_mod.decode(q.numpy(), k.numpy(), v.numpy(), sl, 0.25)
    assert np.array_equal(paged, cont)
    kpn, btn = kp.numpy(), bt.numpy()
    t = np.arange(Lmax)
    gathered = kpn[btn[:, t // ps], :, t % ps].transpose(0, 2, 1, 3)   # [B, Hkv, Lmax, D]
    assert np.array_equal(gathered, k.numpy())


def test_decode_paged_rejects_bad_page(oracle_mod):
    q = np.zeros((1, 2, 8))
    kp = np.zeros((2, 1, 4, 8))
    bt = np.array([[0, 7]], dtype=np.int32)
    with pytest.raises(ValueError):
        oracle_mod.decode_paged(q, kp, kp, bt, [6])
    oracle_mod.decode_paged(q, kp, kp, bt, [4])   # page 7 is never needed for 4 keys


# ---- chunked prefill over a cached prefix (prefill_chunk) -------------------

def _chunk_case(seed, B=2, Hq=4, Hkv=2, Lk=23, D=8):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, Lk, D, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, Lk, D, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, Lk, D, generator=g, dtype=torch.float64)
    return q.numpy(), k.numpy(), v.numpy()


@pytest.mark.parametrize("causal", [True, False])
def test_chunk_is_the_tail_of_the_full_prefill(oracle_mod, causal):
    """Prefilling the last Lq queries over all Lk keys gives exactly the last
    Lq rows of the full prefill (the bottom-right alignment of the mask)."""
    q, k, v = _chunk_case(31)
    full = oracle_mod.prefill(q, k, v, causal=causal, scale=0.4)
    for Lq in (1, 5, 23):
        chunk = oracle_mod.prefill_chunk(q[:, :, -Lq:], k, v, causal=causal, scale=0.4)
        assert np.array_equal(chunk, full[:, :, -Lq:])


def test_chunk_of_one_token_is_a_decode_step(oracle_mod):
    q, k, v = _chunk_case(32)
    chunk = oracle_mod.prefill_chunk(q[:, :, -1:], k, v, causal=True, scale=0.3)[:, :, 0]
    dec = oracle_mod.decode(q[:, :, -1], k, v, [k.shape[2]] * k.shape[0], 0.3)
    np.testing.assert_allclose(chunk, dec, rtol=1e-13, atol=1e-13)


def test_chunk_first_row_ignores_the_chunk_after_it(oracle_mod):
    """Row 0 of a causal chunk sees the prefix and itself only: changing the
    later keys of the chunk leaves it unchanged."""
    q, k, v = _chunk_case(33)
    Lq = 9
    a = oracle_mod.prefill_chunk(q[:, :, -Lq:], k, v, causal=True)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, -Lq + 1:] += 5.0
    v2[:, :, -Lq + 1:] -= 3.0
    b = oracle_mod.prefill_chunk(q[:, :, -Lq:], k2, v2, causal=True)
    assert np.array_equal(a[:, :, 0], b[:, :, 0])
    assert not np.allclose(a[:, :, 1], b[:, :, 1])


# ---- MHA -> GQA checkpoint conversion (the GQA paper notes on 51969.com,
# "Uptraining", figures 1 and 4: each group's K/V projection head is the mean
# of the group's heads; "First" takes the group's first head)
def test_meanpool_is_the_group_mean_of_numpy(oracle_mod):
    # a library routine: numpy's mean over the group axis of [Hkv, G, rows, cols]
    w = rnd((12, 5, 7), 81)
    for Hkv in (1, 2, 3, 4, 6, 12):
        out = oracle_mod.meanpool_heads(w, Hkv)
        ref = w.reshape(Hkv, 12 // Hkv, 5, 7).mean(axis=1)
        np.testing.assert_allclose(out, ref, rtol=1e-14, atol=1e-15)


def test_meanpool_constant_heads_closed_form(oracle_mod):
    # head h filled with the value h: group j's block is j G + (G - 1) / 2
    H, Hkv = 32, 8
    G = H // Hkv
    w = np.broadcast_to(np.arange(H, dtype=np.float64)[:, None, None], (H, 4, 6)).copy()
    out = oracle_mod.meanpool_heads(w, Hkv)
    for j in range(Hkv):
        assert np.all(out[j] == j * G + (G - 1) / 2)


def test_meanpool_identity_mqa_and_first(oracle_mod):
    w = rnd((8, 3, 5), 82)
    np.testing.assert_array_equal(oracle_mod.meanpool_heads(w, 8), w)  # G = 1: MHA stays MHA
    np.testing.assert_allclose(oracle_mod.meanpool_heads(w, 1)[0], w.mean(axis=0), rtol=1e-14, atol=1e-15)
    first = oracle_mod.meanpool_heads(w, 2, mode="first")
    np.testing.assert_array_equal(first, w[[0, 4]])


def test_meanpool_keys_are_the_mean_of_the_group_keys(oracle_mod):
    # figure 1's meaning: the converted head projects x to the mean of the
    # group's per-head keys (linearity of the projection)
    H, Hkv, D, dm = 6, 2, 4, 10
    w = rnd((H, D, dm), 83)
    x = rnd((9, dm), 84)
    out = oracle_mod.meanpool_heads(w, Hkv)
    keys = np.einsum("nc,hdc->hnd", x, w)
    for j in range(Hkv):
        np.testing.assert_allclose(x @ out[j].T, keys[j * 3:(j + 1) * 3].mean(axis=0), rtol=1e-12, atol=1e-12)


def test_meanpool_bf16_input_and_bad_args(oracle_mod):
    bits, vals = bf16(rnd((4, 2, 8), 85))
    bits = bits.reshape(4, 2, 8)
    np.testing.assert_array_equal(oracle_mod.meanpool_heads(bits, 2), oracle_mod.meanpool_heads(vals, 2))
    with pytest.raises(ValueError):
        oracle_mod.meanpool_heads(rnd((6, 2, 2), 86), 4)  # 6 heads do not split into 4 groups
