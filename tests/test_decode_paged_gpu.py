"""Paged-cache decode (gqa_decode_paged through the C ABI) against the fp64
oracle's decode_paged, at the bar of tests/parity.py, and against the
contiguous kernel on the cache the pages were cut from (same plan and tiles,
so the same bits)."""
import numpy as np
import pytest
import torch

from grouped_query_attention_09_b300 import workloads as W
from parity import assert_parity

pytestmark = pytest.mark.gpu


def paged_inputs(w, page_size, seed_off=0):
    q, k, v, sl = W.make_decode_inputs(w)
    kp, vp, bt = W.page_cache(k, v, page_size, seed=w.seed + 50 + seed_off)
    return q, k, v, sl, kp, vp, bt


@pytest.mark.parametrize("name,page_size", [("llama3_8b", 256), ("mqa", 128), ("llama2_70b", 64), ("tiny", 64)])
def test_paged_workload_parity(gqa_lib, oracle_mod, cuda_device, name, page_size):
    w = W.WORKLOADS[name]
    q, k, v, sl, kp, vp, bt = paged_inputs(w, page_size)
    d = cuda_device
    out = gqa_lib.gqa_decode_paged(q.to(d), kp.to(d), vp.to(d), bt.to(d), sl.to(d), scale=w.scale)
    assert gqa_lib.gqa_get_device_status() == 0
    ref = oracle_mod.decode_paged(W.bf16_bits(q), W.bf16_bits(kp), W.bf16_bits(vp), bt.numpy(), sl.numpy(), w.scale)
    assert_parity(out.double().cpu().numpy(), ref, f"paged {name}")
    cont = gqa_lib.gqa_decode(q.to(d), k.to(d), v.to(d), sl.to(d), scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, cont), "paged and contiguous kernels disagree"


def test_paged_nan_tail_ragged_and_bad_pages(gqa_lib, oracle_mod, cuda_device):
    """Ragged lengths with NaN past the end (in the pool), an out-of-range
    entry beyond a sequence's last page (never read: no flag), then a bad
    entry that is needed (flagged; the other sequences stay exact)."""
    w = W.DecodeWorkload("paged_edges", 4, 16, 4, 128, 1000, 1, 1000, 111)
    q, k, v, _ = W.make_decode_inputs(w)
    sl = torch.tensor([1000, 1, 300, 512], dtype=torch.int32)
    W.poison_tail(k, v, sl)
    kp, vp, bt = W.page_cache(k, v, 128, seed=7)
    bt[1, 3] = 10 ** 6  # sequence 1 has 1 key: its page 3 is never needed
    d = cuda_device
    out = gqa_lib.gqa_decode_paged(q.to(d), kp.to(d), vp.to(d), bt.to(d), sl.to(d), scale=w.scale)
    assert gqa_lib.gqa_get_device_status() == 0
    ref = oracle_mod.decode_paged(W.bf16_bits(q), W.bf16_bits(kp), W.bf16_bits(vp), bt.numpy(), sl.numpy(), w.scale)
    assert_parity(out.double().cpu().numpy(), ref, "paged edges")
    bt2 = bt.clone()
    bt2[2, 1] = -3  # needed by sequence 2 (300 keys, page 1 = keys 128..255)
    out2 = gqa_lib.gqa_decode_paged(q.to(d), kp.to(d), vp.to(d), bt2.to(d), sl.to(d), scale=w.scale)
    assert gqa_lib.gqa_get_device_status() == gqa_lib.GQA_DEV_BAD_PAGE
    o2 = out2.double().cpu().numpy()
    assert np.isfinite(o2).all()
    keep = [0, 1, 3]
    assert_parity(o2[keep], ref[keep], "paged edges, other sequences")


def test_paged_one_cta_per_pair_with_bad_entries_in_the_first_pages(gqa_lib, oracle_mod, cuda_device):
    """128 (b, kv head) pairs: one CTA per pair, whose first tiles are
    prefetched into L2 through the block table at launch.  Out-of-pool entries
    in pages that only that prefetch reads (sequences shorter than one page)
    are skipped: no flag, every output exact.  An out-of-pool entry in a page
    the decode needs is flagged, and the other sequences stay exact."""
    B, Hq, Hkv, D, Lmax = 16, 32, 8, 128, 1024
    w = W.DecodeWorkload("paged_pairs", B, Hq, Hkv, D, Lmax, 1, Lmax, 121)
    q, k, v, _ = W.make_decode_inputs(w)
    lens = [Lmax] * B
    lens[3], lens[9] = 100, 1
    sl = torch.tensor(lens, dtype=torch.int32)
    _, num_ctas = gqa_lib.gqa_decode_plan(B, Hq, Hkv, D, Lmax)
    assert num_ctas == B * Hkv  # the one-CTA-per-pair plan
    kp, vp, bt = W.page_cache(k, v, 128, seed=12)
    bt[3, 1], bt[3, 2] = 10 ** 6, -7      # read by the prefetch only: sequence 3 needs page 0
    bt[9, 1], bt[9, 2] = -1, kp.shape[0]  # likewise for sequence 9
    d = cuda_device
    args = (q.to(d), kp.to(d), vp.to(d))
    out = gqa_lib.gqa_decode_paged(*args, bt.to(d), sl.to(d), scale=w.scale)
    assert gqa_lib.gqa_get_device_status() == 0
    ref = oracle_mod.decode_paged(W.bf16_bits(q), W.bf16_bits(kp), W.bf16_bits(vp), bt.numpy(), sl.numpy(), w.scale)
    assert_parity(out.double().cpu().numpy(), ref, "paged, one CTA per pair")
    bt2 = bt.clone()
    bt2[5, 0] = 10 ** 6  # the first page of a full-length sequence
    out2 = gqa_lib.gqa_decode_paged(*args, bt2.to(d), sl.to(d), scale=w.scale)
    assert gqa_lib.gqa_get_device_status() == gqa_lib.GQA_DEV_BAD_PAGE
    o2 = out2.double().cpu().numpy()
    keep = [b for b in range(B) if b != 5]
    assert_parity(o2[keep], ref[keep], "paged, one CTA per pair, other sequences")


def test_paged_page_size_must_match_the_tile(gqa_lib, cuda_device):
    w = W.DecodeWorkload("paged_bad", 2, 8, 2, 128, 256, 1, 256, 5)
    q, k, v, sl = W.make_decode_inputs(w)
    d = cuda_device
    kp, vp, bt = W.page_cache(k, v, 96, seed=3)
    with pytest.raises(gqa_lib.GQAError) as e:
        gqa_lib.gqa_decode_paged(q.to(d), kp.to(d), vp.to(d), bt.to(d), sl.to(d))
    assert e.value.status == gqa_lib.GQA_ERR_UNSUPPORTED
    wm = W.DecodeWorkload("paged_bad_mqa", 2, 32, 1, 128, 256, 1, 256, 6)
    q, k, v, sl = W.make_decode_inputs(wm)
    kp, vp, bt = W.page_cache(k, v, 64, seed=3)   # the wide-group kernel takes 128-key blocks
    with pytest.raises(gqa_lib.GQAError) as e:
        gqa_lib.gqa_decode_paged(q.to(d), kp.to(d), vp.to(d), bt.to(d), sl.to(d))
    assert e.value.status == gqa_lib.GQA_ERR_UNSUPPORTED
