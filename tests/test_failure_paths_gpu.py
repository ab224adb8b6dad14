"""Failure paths on the GPU, made to happen without a fault: a pipeline wait
that runs out, and a workspace allocation that fails.

The waits: gqa_test_set_wait_limit_ns(ns) makes the next launches issue no
pipeline loads and give up every pipeline wait after ns, so the waits for
data that never comes run out and the call takes the kernels' abort path
(flag GQA_DEV_WAIT_TIMEOUT, every role leaves its loop, in-flight MMAs are
drained with the normal limit, TMEM is freed, the kernel returns).  The tests
check that the call returns, that the status comes back, that reading it
resets the decode workspace's arrival counters, and that the next normal call
is parity-green against the oracle.

The allocation: gqa_test_fail_workspace_allocs(1) makes the next decode
workspace allocation fail as out of memory; the call must return
GQA_ERR_CUDA with the CUDA error named, and the next call must work.
(No counterpart on the paper pages: these are the library's error paths.)
"""
import pytest
import torch

from grouped_query_attention_09_b300 import workloads as W
from parity import assert_parity

pytestmark = pytest.mark.gpu

LIMIT_NS = 5_000_000  # 5 ms: each timed-out launch ends in about this long


@pytest.fixture
def short_waits(gqa_lib):
    gqa_lib.gqa_test_set_wait_limit_ns(LIMIT_NS)
    try:
        yield
    finally:
        gqa_lib.gqa_test_set_wait_limit_ns(0)


def _decode_case(name):
    w = W.WORKLOADS[name]
    q, k, v, sl = W.make_decode_inputs(w)
    return w, q, k, v, sl


@pytest.mark.parametrize("name", ["llama3_8b", "mqa"])
def test_decode_wait_timeout_then_recovers(gqa_lib, oracle_mod, cuda_device, name):
    """llama3_8b runs the warp-level kernel (G = 4), mqa the tcgen05 kernel
    (G = 32)."""
    w, q, k, v, sl = _decode_case(name)
    d = cuda_device
    qd, kd, vd, sld = q.to(d), k.to(d), v.to(d), sl.to(d)
    assert gqa_lib.gqa_get_device_status() == 0
    gqa_lib.gqa_test_set_wait_limit_ns(LIMIT_NS)
    try:
        for _ in range(2):
            gqa_lib.gqa_decode(qd, kd, vd, sld, scale=w.scale)
        torch.cuda.synchronize()
    finally:
        gqa_lib.gqa_test_set_wait_limit_ns(0)
    flags = gqa_lib.gqa_get_device_status()
    assert flags & gqa_lib.GQA_DEV_WAIT_TIMEOUT, f"no timeout reported (flags {flags:#x})"
    # the status read reset the counters: a normal call is correct again
    out = gqa_lib.gqa_decode(qd, kd, vd, sld, scale=w.scale)
    assert gqa_lib.gqa_get_device_status() == 0
    ref = oracle_mod.decode(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), sl.numpy(), w.scale)
    assert_parity(out.double().cpu().numpy(), ref, f"{name} after timeout")


def test_fp8_and_paged_decode_wait_timeout(gqa_lib, cuda_device, short_waits):
    """FP8 caches on both kernels (the tcgen05 one waits in its converter
    warps), and a paged cache."""
    d = cuda_device
    for name in ("llama3_8b", "mqa"):
        w = W.WORKLOADS[name]
        q, k8, v8, ks, vs, sl = W.make_decode_fp8_inputs(w)
        gqa_lib.gqa_decode_fp8(q.to(d), k8.to(d), v8.to(d), ks.to(d), vs.to(d), sl.to(d), scale=w.scale)
        assert gqa_lib.gqa_get_device_status() & gqa_lib.GQA_DEV_WAIT_TIMEOUT
    w = W.WORKLOADS["llama3_8b"]
    q, k, v, sl = W.make_decode_inputs(w)
    kp, vp, bt = W.page_cache(k, v, 256, seed=3)
    gqa_lib.gqa_decode_paged(q.to(d), kp.to(d), vp.to(d), bt.to(d), sl.to(d), scale=w.scale)
    assert gqa_lib.gqa_get_device_status() & gqa_lib.GQA_DEV_WAIT_TIMEOUT


def test_prefill_wait_timeout_then_recovers(gqa_lib, oracle_mod, cuda_device):
    w = W.PrefillWorkload("timeout", 2, 1024, 8, 2, 128, True, 17)
    q, k, v = W.make_prefill_inputs(w)
    d = cuda_device
    qd, kd, vd = q.to(d), k.to(d), v.to(d)
    gqa_lib.gqa_test_set_wait_limit_ns(LIMIT_NS)
    try:
        gqa_lib.gqa_prefill(qd, kd, vd, causal=True)
        gqa_lib.gqa_prefill_chunk(qd[:, :, 512:].contiguous(), kd, vd, causal=True)
        torch.cuda.synchronize()
    finally:
        gqa_lib.gqa_test_set_wait_limit_ns(0)
    assert gqa_lib.gqa_get_device_status() & gqa_lib.GQA_DEV_WAIT_TIMEOUT
    out = gqa_lib.gqa_prefill(qd, kd, vd, causal=True)
    assert gqa_lib.gqa_get_device_status() == 0
    ref = oracle_mod.prefill(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), causal=True)
    assert_parity(out.double().cpu().numpy(), ref, "prefill after timeout")


def test_workspace_allocation_failure_is_reported(gqa_lib, oracle_mod, cuda_device):
    """With the workspace released, the next decode must allocate one; the
    injected failure comes back as GQA_ERR_CUDA naming the CUDA error, and the
    call after it allocates and is correct."""
    w, q, k, v, sl = _decode_case("llama2_70b")  # cut pairs: the workspace is used
    d = cuda_device
    qd, kd, vd, sld = q.to(d), k.to(d), v.to(d), sl.to(d)
    torch.cuda.synchronize()
    gqa_lib.gqa_release()
    gqa_lib.gqa_test_fail_workspace_allocs(1)
    try:
        with pytest.raises(gqa_lib.GQAError) as e:
            gqa_lib.gqa_decode(qd, kd, vd, sld, scale=w.scale)
    finally:
        gqa_lib.gqa_test_fail_workspace_allocs(0)
    assert e.value.status == gqa_lib.GQA_ERR_CUDA
    assert "cudaErrorMemoryAllocation" in str(e.value)
    out = gqa_lib.gqa_decode(qd, kd, vd, sld, scale=w.scale)
    assert gqa_lib.gqa_get_device_status() == 0
    ref = oracle_mod.decode(W.bf16_bits(q), W.bf16_bits(k), W.bf16_bits(v), sl.numpy(), w.scale)
    assert_parity(out.double().cpu().numpy(), ref, "decode after a failed allocation")
