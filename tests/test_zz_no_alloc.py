"""gqa_decode_noalloc: the allocation-free decode entry point.

It serves callers that cannot let the library allocate device memory (a
serving engine that owns all HBM through its own pool; a latency-critical
loop that may not call cudaMalloc after start-up).  Its workspace is a fixed
array inside libgqa.so.  These tests call it through the C ABI, two calls in
a row, and check each call against gqa_decode and against the fp64 oracle with
the tolerance of the decode parity tests; they also check that once the first
call has set the array up, later calls change no device-memory total.  The
file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from grouped_query_attention_09_b300 import workloads as W
from parity import ATOL, RTOL, assert_parity

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def call_noalloc(lib, q, k, v, sl, out, scale, stream):
    B, Hq, D = q.shape
    Hkv, Lmax = k.shape[1], k.shape[2]
    return lib.gqa_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(sl), _ptr(out), B, Hq, Hkv, D, Lmax,
                                  ctypes.c_float(scale), ctypes.c_void_p(stream.cuda_stream))


def _oracle(oracle_mod, q, k, v, sl, scale):
    return oracle_mod.decode(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), sl.numpy(), scale)


@pytest.mark.parametrize("name", ["mqa", "llama3_8b", "llama2_70b"])
def test_noalloc_matches_gqa_decode_twice(gqa_lib, oracle_mod, cuda_device, name):
    lib = gqa_lib.load_library()
    w = W.WORKLOADS[name]
    q, k, v, sl = W.make_decode_inputs(w)
    qd, kd, vd, sld = (t.to(cuda_device) for t in (q, k, v, sl))
    stream = torch.cuda.current_stream(cuda_device)
    ref = gqa_lib.gqa_decode(qd, kd, vd, sld, scale=w.scale).double()
    exact = _oracle(oracle_mod, q, k, v, sl, w.scale)
    outs = [torch.full_like(qd, float("nan")) for _ in range(2)]
    free = []
    for call in range(2):
        # device memory free before and after the call, with nothing else
        # allocating in between (torch's allocator works between the calls)
        torch.cuda.synchronize()
        before = torch.cuda.mem_get_info(cuda_device)[0]
        st = call_noalloc(lib, qd, kd, vd, sld, outs[call], w.scale, stream)
        assert st == 0, gqa_lib.gqa_status_string(st)
        torch.cuda.synchronize()
        free.append((before, torch.cuda.mem_get_info(cuda_device)[0]))
        got = outs[call].double()
        assert torch.isfinite(got).all(), f"call {call}: non-finite output"
        bad = (got - ref).abs() > ATOL + RTOL * ref.abs()
        assert not bad.any(), f"call {call}: {int(bad.sum())} elements differ from gqa_decode"
        assert_parity(got.cpu().numpy(), exact, f"{name} no-alloc call {call}")
    # the first call on this device may have set the array up; the second
    # changed no device-memory total
    assert free[1][0] == free[1][1]
    assert gqa_lib.gqa_get_device_status() == 0


def test_noalloc_second_call_with_other_lengths(gqa_lib, oracle_mod, cuda_device):
    """The array keeps the last call's contents; a following call with other
    sizes must not see them."""
    lib = gqa_lib.load_library()
    stream = torch.cuda.current_stream(cuda_device)
    for w in (W.DecodeWorkload("a", 6, 16, 2, 128, 900, 1, 900, 5),
              W.DecodeWorkload("b", 3, 8, 2, 64, 300, 1, 300, 6)):
        q, k, v, sl = W.make_decode_inputs(w)
        qd, kd, vd, sld = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device), sl.to(cuda_device)
        out = torch.empty_like(qd)
        assert call_noalloc(lib, qd, kd, vd, sld, out, w.scale, stream) == 0
        ref = gqa_lib.gqa_decode(qd, kd, vd, sld, scale=w.scale)
        torch.cuda.synchronize()
        diff = (out.double() - ref.double()).abs()
        assert (diff <= ATOL + RTOL * ref.double().abs()).all()
        assert_parity(out.double().cpu().numpy(), _oracle(oracle_mod, q, k, v, sl, w.scale), w.name)


def test_noalloc_device_status_is_reported(gqa_lib, cuda_device):
    """The call keeps its status word in the fixed array; gqa_get_device_status
    reports (and clears) it: a length above the cache capacity is clamped and
    flagged."""
    lib = gqa_lib.load_library()
    stream = torch.cuda.current_stream(cuda_device)
    w = W.DecodeWorkload("clamp", 2, 8, 2, 128, 256, 256, 256, 8)
    q, k, v, _ = W.make_decode_inputs(w)
    sl = torch.tensor([300, 10], dtype=torch.int32)
    qd, kd, vd, sld = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device), sl.to(cuda_device)
    out = torch.empty_like(qd)
    assert gqa_lib.gqa_get_device_status() == 0
    assert call_noalloc(lib, qd, kd, vd, sld, out, w.scale, stream) == 0
    assert gqa_lib.gqa_get_device_status() == gqa_lib.GQA_DEV_SEQLEN_CLAMPED
    assert gqa_lib.gqa_get_device_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(gqa_lib, cuda_device):
    """B * Hkv above the fixed maximum comes back as GQA_ERR_TOO_LARGE before
    any work is enqueued."""
    lib = gqa_lib.load_library()
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: the call returns first
    torch.cuda.set_device(cuda_device)
    st = lib.gqa_decode_noalloc(fake, fake, fake, fake, fake, 1000, 9 * 2, 9, 128, 64, ctypes.c_float(0.1), None)
    assert st == gqa_lib.GQA_ERR_TOO_LARGE
    assert "fixed scratch" in gqa_lib.gqa_status_string(st)
