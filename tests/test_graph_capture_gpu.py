"""The device entry points captured into a CUDA graph (stream capture) and
replayed on new inputs, against the fp64 oracle at the bar of
tests/parity.py.

A serving loop captures one decode step and replays it: each replay reads the
current contents of the same buffers, so new query/key/value values and the
grown cache are seen without re-capturing.  The library's split-KV merge
counters return to zero inside every launch, so replays need no reset.
"""
import numpy as np
import pytest
import torch

from grouped_query_attention_09_b300 import workloads as W
from parity import assert_parity

pytestmark = pytest.mark.gpu


def _gen(seed):
    return torch.Generator().manual_seed(seed)


def _bf16(shape, g):
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


def test_decode_step_graph_appends_and_decodes(gqa_lib, oracle_mod, cuda_device):
    """One captured step = rotary embedding + cache append of the new token,
    then decode over the grown cache (G = 4: the warp-level kernel).  Three
    replays on fresh q / k / v values: every replay matches the oracle's
    append followed by its decode, and seqlens advances once per replay."""
    B, Hq, Hkv, D, Lmax = 4, 32, 8, 128, 1024
    lens = [1000, 300, 1, 640]
    g = _gen(5100)
    kc, vc = _bf16((B, Hkv, Lmax, D), g), _bf16((B, Hkv, Lmax, D), g)
    dev = cuda_device
    kcd, vcd = kc.to(dev), vc.to(dev)
    sld = torch.tensor(lens, dtype=torch.int32, device=dev)
    q_in = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    k_new = torch.empty(B, Hkv, D, dtype=torch.bfloat16, device=dev)
    v_new = torch.empty(B, Hkv, D, dtype=torch.bfloat16, device=dev)
    q_rot = torch.empty_like(q_in)
    out = torch.empty_like(q_in)
    # One call of each size outside the capture: the decode workspace exists.
    gqa_lib.gqa_decode(q_rot.zero_(), kcd.clone(), vcd.clone(), sld.clone(), out=out)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gqa_lib.gqa_rope_append(q_in, k_new, v_new, kcd, vcd, sld, q_out=q_rot)
        gqa_lib.gqa_decode(q_rot, kcd, vcd, sld, out=out)
    # Capturing enqueues nothing: the cache and seqlens are untouched.
    torch.cuda.synchronize()
    assert sld.cpu().tolist() == lens

    kref, vref = kc.double().numpy().copy(), vc.double().numpy().copy()
    cur = np.array(lens)
    for step in range(3):
        q, kn, vn = _bf16((B, Hq, D), g), _bf16((B, Hkv, D), g), _bf16((B, Hkv, D), g)
        q_in.copy_(q)
        k_new.copy_(kn)
        v_new.copy_(vn)
        graph.replay()
        torch.cuda.synchronize()
        qo, ko, vo = oracle_mod.rope_append(W.bf16_bits(q), W.bf16_bits(kn), W.bf16_bits(vn), cur, Lmax=Lmax)
        for b, n in enumerate(cur):
            kref[b, :, n] = ko[b]
            vref[b, :, n] = vo[b]
        cur = cur + 1
        ref = oracle_mod.decode(qo, kref, vref, cur, D ** -0.5)
        assert_parity(out.double().cpu().numpy(), ref, f"replay {step}")
        assert sld.cpu().tolist() == cur.tolist()
    assert gqa_lib.gqa_get_device_status() == 0


def test_wide_group_decode_and_prefills_in_one_graph(gqa_lib, oracle_mod, cuda_device):
    """A wide-group decode (G = 32, the tcgen05 kernel with pairs cut across
    CTAs and merged in the launch), the same decode through the no-alloc entry
    point and over FP8 pages, a causal prefill and a chunked prefill captured
    together; two
    replays on fresh inputs both match the oracle (the merge counters a replay
    leaves behind are the zeros the next one needs), the no-alloc output
    equals the other bit for bit, and the FP8-page output equals the
    contiguous FP8 call on the same quantised cache."""
    dev = cuda_device
    # decode: ragged lengths spread over many CTAs, so pairs are cut
    dB, dHq, dHkv, dD, dLmax = 24, 32, 1, 128, 2048
    dl = torch.randint(300, dLmax + 1, (dB,), generator=_gen(5200), dtype=torch.int32)
    dq = torch.empty(dB, dHq, dD, dtype=torch.bfloat16, device=dev)
    dk = torch.empty(dB, dHkv, dLmax, dD, dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    dsl = dl.to(dev)
    dout = torch.empty_like(dq)
    nout = torch.empty_like(dq)
    # the same decode over FP8 pages (128-row pages of E4M3 bytes, unit scales)
    page = 128
    mp = dLmax // page
    f_kp = torch.zeros(dB * mp, dHkv, page, dD, dtype=torch.uint8, device=dev)
    f_vp = torch.zeros_like(f_kp)
    f_bt = torch.randperm(dB * mp, generator=_gen(5210)).to(torch.int32).reshape(dB, mp).to(dev)
    f_ks = torch.ones(dB, dHkv, dtype=torch.float32, device=dev)
    f_vs = torch.ones_like(f_ks)
    f_out = torch.empty_like(dq)
    # prefill (causal, G = 4) and a 100-token chunk after 284 cached ones
    pB, pHq, pHkv, pL, pD = 1, 8, 2, 384, 128
    pq = torch.empty(pB, pHq, pL, pD, dtype=torch.bfloat16, device=dev)
    pk = torch.empty(pB, pHkv, pL, pD, dtype=torch.bfloat16, device=dev)
    pv = torch.empty_like(pk)
    pout = torch.empty_like(pq)
    cLq = 100
    cq = torch.empty(pB, pHq, cLq, pD, dtype=torch.bfloat16, device=dev)
    cout = torch.empty_like(cq)
    for t in (dq, dk, dv, pq, pk, pv, cq):
        t.zero_()
    gqa_lib.gqa_decode(dq, dk, dv, dsl, out=dout)
    gqa_lib.gqa_decode_noalloc(dq, dk, dv, dsl, nout)
    gqa_lib.gqa_decode_fp8_paged(dq, f_kp, f_vp, f_ks, f_vs, f_bt, dsl, out=f_out)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gqa_lib.gqa_decode(dq, dk, dv, dsl, out=dout)
        gqa_lib.gqa_decode_noalloc(dq, dk, dv, dsl, nout)
        gqa_lib.gqa_decode_fp8_paged(dq, f_kp, f_vp, f_ks, f_vs, f_bt, dsl, out=f_out)
        gqa_lib.gqa_prefill(pq, pk, pv, out=pout, causal=True)
        gqa_lib.gqa_prefill_chunk(cq, pk, pv, out=cout, causal=True)

    g = _gen(5300)
    for rep in range(2):
        hq, hk, hv = _bf16(dq.shape, g), _bf16(dk.shape, g), _bf16(dv.shape, g)
        h_pq, h_pk, h_pv, h_cq = _bf16(pq.shape, g), _bf16(pk.shape, g), _bf16(pv.shape, g), _bf16(cq.shape, g)
        for d, h in ((dq, hq), (dk, hk), (dv, hv), (pq, h_pq), (pk, h_pk), (pv, h_pv), (cq, h_cq)):
            d.copy_(h)
        k8, v8, ks8, vs8 = W.quantize_kv_fp8(hk, hv)
        bt_h = f_bt.cpu()
        for b in range(dB):
            for i in range(mp):
                f_kp[int(bt_h[b, i])].copy_(k8[b, :, i * page:(i + 1) * page].to(dev))
                f_vp[int(bt_h[b, i])].copy_(v8[b, :, i * page:(i + 1) * page].to(dev))
        f_ks.copy_(ks8)
        f_vs.copy_(vs8)
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle_mod.decode(W.bf16_bits(hq), W.bf16_bits(hk), W.bf16_bits(hv), dl.numpy(), dD ** -0.5)
        assert_parity(dout.double().cpu().numpy(), ref, f"decode replay {rep}")
        assert torch.equal(nout, dout)
        f_ref = gqa_lib.gqa_decode_fp8(dq, k8.to(dev), v8.to(dev), f_ks, f_vs, dsl)
        assert torch.equal(f_out, f_ref)
        ref = oracle_mod.prefill(W.bf16_bits(h_pq), W.bf16_bits(h_pk), W.bf16_bits(h_pv), causal=True)
        assert_parity(pout.double().cpu().numpy(), ref, f"prefill replay {rep}")
        ref = oracle_mod.prefill_chunk(W.bf16_bits(h_cq), W.bf16_bits(h_pk), W.bf16_bits(h_pv), causal=True)
        assert_parity(cout.double().cpu().numpy(), ref, f"chunk replay {rep}")
    assert gqa_lib.gqa_get_device_status() == 0


def test_capture_that_would_grow_the_workspace_is_refused(gqa_lib, cuda_device):
    """A captured call whose workspace is larger than any call made so far
    returns GQA_ERR_CUDA (naming the capture) and enqueues nothing; the same
    call made outside the capture afterwards works."""
    dev = cuda_device
    gqa_lib.gqa_release()
    small = [torch.zeros(1, 8, 128, dtype=torch.bfloat16, device=dev),
             torch.zeros(1, 2, 128, 128, dtype=torch.bfloat16, device=dev),
             torch.zeros(1, 2, 128, 128, dtype=torch.bfloat16, device=dev),
             torch.full((1,), 128, dtype=torch.int32, device=dev)]
    gqa_lib.gqa_decode(*small)
    torch.cuda.synchronize()
    B, Hq, Hkv, D, Lmax = 64, 32, 8, 128, 4096
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(B, Hkv, Lmax, D, dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    sl = torch.full((B,), Lmax, dtype=torch.int32, device=dev)
    out = torch.full_like(q, 7.0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        with pytest.raises(gqa_lib.GQAError) as ei:
            gqa_lib.gqa_decode(q, k, v, sl, out=out)
        out.add_(0)  # keep the graph non-empty
    assert ei.value.status == gqa_lib.GQA_ERR_CUDA
    assert "capture" in str(ei.value)
    graph.replay()
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    gqa_lib.gqa_decode(q, k, v, sl, out=out)
    assert gqa_lib.gqa_get_device_status() == 0
    assert bool((out == 0).all())
