"""Grouped-query attention on NVIDIA B300 (sm_103a).

A thin ctypes binding of libgqa.so: every function here only marshals
arguments (torch tensors -> raw pointers and sizes) and raises on a non-zero
status.  All arithmetic runs in the library's CUDA kernels; there is no CPU
or PyTorch fallback, and a missing or unloadable library raises.

Names and semantics follow include/gqa.h:
  gqa_decode, gqa_decode_fp8, gqa_decode_paged, gqa_decode_fp8_paged, gqa_decode_noalloc, gqa_rope_append,
  gqa_meanpool_kv_heads, gqa_prefill, gqa_prefill_chunk, gqa_decode_host, gqa_prefill_host,
  gqa_status_string, gqa_get_device_status, gqa_decode_plan, gqa_release,
  and the failure-injection hooks gqa_test_set_wait_limit_ns,
  gqa_test_fail_workspace_allocs.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgqa.so")

GQA_OK = 0
GQA_ERR_INVALID_ARG = 1
GQA_ERR_UNSUPPORTED = 2
GQA_ERR_NULL = 3
GQA_ERR_MISALIGNED = 4
GQA_ERR_CUDA = 5
GQA_ERR_NO_DEVICE = 6
GQA_ERR_TOO_LARGE = 7

GQA_DEV_SEQLEN_CLAMPED = 0x1
GQA_DEV_EMPTY_CONTEXT = 0x2
GQA_DEV_WAIT_TIMEOUT = 0x4
GQA_DEV_CACHE_FULL = 0x8
GQA_DEV_BAD_PAGE = 0x10

EXPORTED = ("gqa_decode", "gqa_prefill", "gqa_decode_host", "gqa_prefill_host",
            "gqa_status_string", "gqa_get_device_status", "gqa_decode_plan", "gqa_release",
            "gqa_decode_noalloc", "gqa_decode_fp8", "gqa_rope_append", "gqa_decode_paged", "gqa_decode_fp8_paged",
            "gqa_prefill_chunk",
            "gqa_meanpool_kv_heads", "gqa_test_set_wait_limit_ns", "gqa_test_fail_workspace_allocs")

_lib = None


class GQAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gqa_status_string(status)}")


def load_library():
    """Loads libgqa.so (built by grouped_query_attention_09_b300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: run `python -m grouped_query_attention_09_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.gqa_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.gqa_prefill.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, vp]
    lib.gqa_decode_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.gqa_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.gqa_prefill_host.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, vp]
    lib.gqa_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.gqa_rope_append.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_double, vp]
    lib.gqa_rope_append.restype = i
    lib.gqa_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.gqa_decode_paged.restype = i
    lib.gqa_decode_fp8_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.gqa_decode_fp8_paged.restype = i
    lib.gqa_prefill_chunk.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
    lib.gqa_prefill_chunk.restype = i
    lib.gqa_meanpool_kv_heads.argtypes = [vp, vp, i, i, i, i, i, vp]
    lib.gqa_meanpool_kv_heads.restype = i
    for fn in ("gqa_decode", "gqa_prefill", "gqa_decode_host", "gqa_prefill_host", "gqa_decode_noalloc",
               "gqa_decode_fp8"):
        getattr(lib, fn).restype = i
    lib.gqa_status_string.argtypes = [i]
    lib.gqa_status_string.restype = ctypes.c_char_p
    lib.gqa_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.gqa_get_device_status.restype = i
    lib.gqa_decode_plan.argtypes = [i, i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
    lib.gqa_decode_plan.restype = i
    lib.gqa_release.argtypes = []
    lib.gqa_release.restype = None
    lib.gqa_test_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.gqa_test_set_wait_limit_ns.restype = None
    lib.gqa_test_fail_workspace_allocs.argtypes = [i]
    lib.gqa_test_fail_workspace_allocs.restype = None
    _lib = lib
    return lib


def gqa_status_string(status: int) -> str:
    return load_library().gqa_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != GQA_OK:
        raise GQAError(status, where)


def _stream_ptr(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _dev_ptr(t, name, dtype):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def gqa_decode(q, k_cache, v_cache, seqlens, out=None, scale=None, stream=None):
    """One decode step.  q [B, Hq, D] bf16; k_cache/v_cache [B, Hkv, Lmax, D]
    bf16; seqlens [B] int32 (device); returns out [B, Hq, D] bf16."""
    import torch
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if scale is None:
        scale = D ** -0.5
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.gqa_decode(_dev_ptr(q, "q", torch.bfloat16), _dev_ptr(k_cache, "k_cache", torch.bfloat16),
                            _dev_ptr(v_cache, "v_cache", torch.bfloat16), _dev_ptr(seqlens, "seqlens", torch.int32),
                            _dev_ptr(out, "out", torch.bfloat16), B, Hq, Hkv, D, Lmax, float(scale),
                            _stream_ptr(stream, q.device))
    _check(st, "gqa_decode")
    return out


def gqa_decode_noalloc(q, k_cache, v_cache, seqlens, out, scale=None, stream=None):
    """gqa_decode with its workspace in the library's fixed device array: the
    call allocates nothing (out must be given).  Overlapping calls race."""
    import torch
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    if scale is None:
        scale = D ** -0.5
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.gqa_decode_noalloc(_dev_ptr(q, "q", torch.bfloat16), _dev_ptr(k_cache, "k_cache", torch.bfloat16),
                                    _dev_ptr(v_cache, "v_cache", torch.bfloat16),
                                    _dev_ptr(seqlens, "seqlens", torch.int32), _dev_ptr(out, "out", torch.bfloat16),
                                    B, Hq, Hkv, D, Lmax, float(scale), _stream_ptr(stream, q.device))
    _check(st, "gqa_decode_noalloc")
    return out


def gqa_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, seqlens, out=None, scale=None, stream=None):
    """Decode over an FP8 E4M3 cache.  q [B, Hq, D] bf16; k_cache/v_cache
    [B, Hkv, Lmax, D] uint8 (E4M3 bytes); k_scale/v_scale [B, Hkv] fp32;
    seqlens [B] int32 (device); returns out [B, Hq, D] bf16."""
    import torch
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if scale is None:
        scale = D ** -0.5
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.gqa_decode_fp8(_dev_ptr(q, "q", torch.bfloat16), _dev_ptr(k_cache, "k_cache", torch.uint8),
                                _dev_ptr(v_cache, "v_cache", torch.uint8), _dev_ptr(k_scale, "k_scale", torch.float32),
                                _dev_ptr(v_scale, "v_scale", torch.float32), _dev_ptr(seqlens, "seqlens", torch.int32),
                                _dev_ptr(out, "out", torch.bfloat16), B, Hq, Hkv, D, Lmax, float(scale),
                                _stream_ptr(stream, q.device))
    _check(st, "gqa_decode_fp8")
    return out


def gqa_decode_paged(q, k_pages, v_pages, block_table, seqlens, out=None, scale=None, stream=None):
    """Decode over a paged cache.  q [B, Hq, D] bf16; k_pages/v_pages
    [num_pages, Hkv, page_size, D] bf16; block_table [B, max_pages] int32;
    seqlens [B] int32 (all device); returns out [B, Hq, D] bf16."""
    import torch
    B, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = k_pages.shape
    max_pages = block_table.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if scale is None:
        scale = D ** -0.5
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.gqa_decode_paged(_dev_ptr(q, "q", torch.bfloat16), _dev_ptr(k_pages, "k_pages", torch.bfloat16),
                                  _dev_ptr(v_pages, "v_pages", torch.bfloat16),
                                  _dev_ptr(block_table, "block_table", torch.int32),
                                  _dev_ptr(seqlens, "seqlens", torch.int32), _dev_ptr(out, "out", torch.bfloat16),
                                  B, Hq, Hkv, D, num_pages, page_size, max_pages, float(scale),
                                  _stream_ptr(stream, q.device))
    _check(st, "gqa_decode_paged")
    return out


def gqa_decode_fp8_paged(q, k_pages, v_pages, k_scale, v_scale, block_table, seqlens, out=None, scale=None,
                         stream=None):
    """Decode over a paged FP8 E4M3 cache.  q [B, Hq, D] bf16; k_pages/v_pages
    [num_pages, Hkv, page_size, D] uint8; k_scale/v_scale [B, Hkv] fp32;
    block_table [B, max_pages] int32; seqlens [B] int32 (all device); returns
    out [B, Hq, D] bf16."""
    import torch
    B, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = k_pages.shape
    max_pages = block_table.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if scale is None:
        scale = D ** -0.5
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.gqa_decode_fp8_paged(_dev_ptr(q, "q", torch.bfloat16), _dev_ptr(k_pages, "k_pages", torch.uint8),
                                      _dev_ptr(v_pages, "v_pages", torch.uint8),
                                      _dev_ptr(k_scale, "k_scale", torch.float32),
                                      _dev_ptr(v_scale, "v_scale", torch.float32),
                                      _dev_ptr(block_table, "block_table", torch.int32),
                                      _dev_ptr(seqlens, "seqlens", torch.int32), _dev_ptr(out, "out", torch.bfloat16),
                                      B, Hq, Hkv, D, num_pages, page_size, max_pages, float(scale),
                                      _stream_ptr(stream, q.device))
    _check(st, "gqa_decode_fp8_paged")
    return out


def gqa_rope_append(q, k_new, v_new, k_cache, v_cache, seqlens, q_out=None, base=10000.0, stream=None):
    """Rotary embedding of the new token at position seqlens[b] and the append
    of its K/V heads as cache row seqlens[b]; seqlens advances by one.
    q [B, Hq, D]; k_new, v_new [B, Hkv, D]; caches [B, Hkv, Lmax, D] (bf16,
    device); seqlens [B] int32 (device, updated).  Returns q_out (rotated q;
    pass q_out=q to rotate in place)."""
    import torch
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    if q_out is None:
        q_out = torch.empty_like(q)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.gqa_rope_append(_dev_ptr(q, "q", torch.bfloat16), _dev_ptr(k_new, "k_new", torch.bfloat16),
                                 _dev_ptr(v_new, "v_new", torch.bfloat16), _dev_ptr(q_out, "q_out", torch.bfloat16),
                                 _dev_ptr(k_cache, "k_cache", torch.bfloat16),
                                 _dev_ptr(v_cache, "v_cache", torch.bfloat16), _dev_ptr(seqlens, "seqlens", torch.int32),
                                 B, Hq, Hkv, D, Lmax, float(base), _stream_ptr(stream, q.device))
    _check(st, "gqa_rope_append")
    return q_out


def gqa_meanpool_kv_heads(w, Hkv, mode="mean", out=None, stream=None):
    """MHA -> GQA checkpoint conversion of a key or value projection.
    w [H, rows, cols] bf16 (device; head h's block, e.g. an nn.Linear weight
    [H * head_dim, d_model] viewed as [H, head_dim, d_model]); returns
    [Hkv, rows, cols]: group j's block is the mean of heads j*G .. j*G + G - 1
    (mode "mean") or head j*G (mode "first")."""
    import torch
    H, rows, cols = w.shape
    if out is None:
        out = torch.empty((int(Hkv), rows, cols), dtype=w.dtype, device=w.device)
    m = {"mean": 0, "first": 1}[mode]
    lib = load_library()
    with torch.cuda.device(w.device):
        st = lib.gqa_meanpool_kv_heads(_dev_ptr(w, "w", torch.bfloat16), _dev_ptr(out, "out", torch.bfloat16),
                                       H, int(Hkv), rows, cols, m, _stream_ptr(stream, w.device))
    _check(st, "gqa_meanpool_kv_heads")
    return out


def gqa_prefill(q, k, v, out=None, causal=True, stream=None):
    """Prefill.  q [B, Hq, L, D], k/v [B, Hkv, L, D] bf16; returns out like q."""
    import torch
    B, Hq, L, D = q.shape
    Hkv = k.shape[1]
    if out is None:
        out = torch.empty_like(q)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.gqa_prefill(_dev_ptr(q, "q", torch.bfloat16), _dev_ptr(k, "k", torch.bfloat16),
                             _dev_ptr(v, "v", torch.bfloat16), _dev_ptr(out, "out", torch.bfloat16),
                             B, L, Hq, Hkv, D, int(bool(causal)), _stream_ptr(stream, q.device))
    _check(st, "gqa_prefill")
    return out


def gqa_prefill_chunk(q, k, v, out=None, causal=True, stream=None):
    """Chunked prefill: q [B, Hq, Lq, D] (the chunk), k/v [B, Hkv, Lk, D] (the
    cached prefix then the chunk, Lk >= Lq), bf16 on the device; causal row i
    sees keys t <= Lk - Lq + i.  Returns out like q."""
    import torch
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.gqa_prefill_chunk(_dev_ptr(q, "q", torch.bfloat16), _dev_ptr(k, "k", torch.bfloat16),
                                   _dev_ptr(v, "v", torch.bfloat16), _dev_ptr(out, "out", torch.bfloat16),
                                   B, Lq, Lk, Hq, Hkv, D, int(bool(causal)), _stream_ptr(stream, q.device))
    _check(st, "gqa_prefill_chunk")
    return out


def _host_ptr(t, name, dtype):
    import torch
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a CPU tensor")
    if t.dtype != dtype or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous {dtype} tensor")
    return ctypes.c_void_p(t.data_ptr())


def gqa_decode_host(q, k_cache, v_cache, seqlens, out=None, scale=None, stream=None, device=None):
    """gqa_decode on host (CPU, ideally pinned) tensors; returns a host out."""
    import torch
    B, Hq, D = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if scale is None:
        scale = D ** -0.5
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        st = load_library().gqa_decode_host(
            _host_ptr(q, "q", torch.bfloat16), _host_ptr(k_cache, "k_cache", torch.bfloat16),
            _host_ptr(v_cache, "v_cache", torch.bfloat16), _host_ptr(seqlens, "seqlens", torch.int32),
            _host_ptr(out, "out", torch.bfloat16), B, Hq, Hkv, D, Lmax, float(scale), _stream_ptr(stream, device))
    _check(st, "gqa_decode_host")
    return out


def gqa_prefill_host(q, k, v, out=None, causal=True, stream=None, device=None):
    """gqa_prefill on host tensors; returns a host out."""
    import torch
    B, Hq, L, D = q.shape
    Hkv = k.shape[1]
    if out is None:
        out = torch.empty_like(q)
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        st = load_library().gqa_prefill_host(
            _host_ptr(q, "q", torch.bfloat16), _host_ptr(k, "k", torch.bfloat16), _host_ptr(v, "v", torch.bfloat16),
            _host_ptr(out, "out", torch.bfloat16), B, L, Hq, Hkv, D, int(bool(causal)), _stream_ptr(stream, device))
    _check(st, "gqa_prefill_host")
    return out


def gqa_get_device_status(stream=None, device=None) -> int:
    """Synchronises the stream and returns (and clears) the GQA_DEV_* bits."""
    import torch
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    flags = ctypes.c_uint32(0)
    with torch.cuda.device(device):
        st = load_library().gqa_get_device_status(_stream_ptr(stream, device), ctypes.byref(flags))
    _check(st, "gqa_get_device_status")
    return int(flags.value)


def gqa_decode_plan(B, Hq, Hkv, D, Lmax):
    """(tile_keys, num_ctas) of the split gqa_decode would use."""
    tk, nc = ctypes.c_int(0), ctypes.c_int(0)
    st = load_library().gqa_decode_plan(B, Hq, Hkv, D, Lmax, ctypes.byref(tk), ctypes.byref(nc))
    _check(st, "gqa_decode_plan")
    return tk.value, nc.value


def gqa_release():
    load_library().gqa_release()


def gqa_test_set_wait_limit_ns(ns: int):
    """Test hook: with ns > 0, later launches issue no pipeline loads and their
    pipeline waits give up after ns nanoseconds (0 restores normal operation)."""
    load_library().gqa_test_set_wait_limit_ns(int(ns))


def gqa_test_fail_workspace_allocs(n: int):
    """Test hook: the next n decode-workspace allocations fail as out of memory."""
    load_library().gqa_test_fail_workspace_allocs(int(n))
