"""gqa_decode_noalloc: the allocation-free decode entry point.

It serves callers that cannot let the library allocate device memory (a
serving engine that owns all HBM through its own pool; a latency-critical
loop that may not call cudaMalloc after start-up).  Its workspace is a fixed
array inside libgqa.so.  These tests call it through the C ABI and check it
against gqa_decode, on two calls in a row, with the tolerance of the decode
parity tests.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from grouped_query_attention_09_b300 import workloads as W

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def call_noalloc(lib, q, k, v, sl, out, scale, stream):
    B, Hq, D = q.shape
    Hkv, Lmax = k.shape[1], k.shape[2]
    return lib.gqa_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(sl), _ptr(out), B, Hq, Hkv, D, Lmax,
                                  ctypes.c_float(scale), ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("name", ["mqa", "llama3_8b"])
def test_noalloc_matches_gqa_decode_twice(gqa_lib, cuda_device, name):
    lib = gqa_lib.load_library()
    w = W.WORKLOADS[name]
    q, k, v, sl = [t.to(cuda_device) for t in W.make_decode_inputs(w)]
    stream = torch.cuda.current_stream(cuda_device)
    ref = gqa_lib.gqa_decode(q, k, v, sl, scale=w.scale).double()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        st = call_noalloc(lib, q, k, v, sl, out, w.scale, stream)
        assert st == 0, gqa_lib.gqa_status_string(st)
        torch.cuda.synchronize()
        got = out.double()
        assert torch.isfinite(got).all(), f"call {call}: non-finite output"
        bad = (got - ref).abs() > ATOL + RTOL * ref.abs()
        assert not bad.any(), f"call {call}: {int(bad.sum())} elements differ from gqa_decode"


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


def test_noalloc_rejects_sizes_beyond_its_scratch(gqa_lib, cuda_device):
    """B * Hkv above the fixed maximum comes back as GQA_ERR_TOO_LARGE before
    any work is enqueued."""
    lib = gqa_lib.load_library()
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: the call returns first
    torch.cuda.set_device(cuda_device)
    st = lib.gqa_decode_noalloc(fake, fake, fake, fake, fake, 1000, 9 * 2, 9, 128, 64, ctypes.c_float(0.1), None)
    assert st == gqa_lib.GQA_ERR_TOO_LARGE
    assert "fixed scratch" in gqa_lib.gqa_status_string(st)
