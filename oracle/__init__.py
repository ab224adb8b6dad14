"""fp64 CPU oracle for grouped-query attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` import this package.  The product library never does, and
this package imports nothing from it.

The arithmetic lives in ``gqa_oracle.c`` (plain C, OpenMP over output rows);
this module only compiles it with gcc and marshals numpy arrays through ctypes.
Every function follows the steps stated in that file's header:

* widen bf16 to fp64 exactly;
* expand K/V per group (query head h reads KV head h // (Hq // Hkv)), the
  ``repeat_interleave`` of "手把手教你用PyTorch实现GQA" section 1.3 and the
  ``repeat_kv`` of the GQA paper notes ("QA 相关", inference);
* scores = q.k * scale, causal removal of future keys, softmax, @ V
  (the Huawei Cloud post "多头注意力机制的代码实现（MQA和GQA）", section 5).

Inputs are numpy arrays: ``np.uint16`` holding bf16 bit patterns, or
``np.float64``.  Outputs are ``np.float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

EMPTY_CONTEXT = 3


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (-O2, OpenMP) if missing or stale."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        p = ctypes.c_void_p
        i = ctypes.c_int
        lib.gqa_oracle_decode.argtypes = [p, p, p, i, p, i, i, i, i, i, ctypes.c_double, p, i, p]
        lib.gqa_oracle_decode.restype = i
        lib.gqa_oracle_prefill.argtypes = [p, p, p, i, i, i, i, i, i, i, ctypes.c_double, p, i, p]
        lib.gqa_oracle_prefill.restype = i
        lib.gqa_oracle_decode_fp8.argtypes = [p, i, p, p, p, p, p, i, i, i, i, i, ctypes.c_double, p, i, p]
        lib.gqa_oracle_decode_fp8.restype = i
        lib.gqa_oracle_e4m3_values.argtypes = [p, i, p]
        lib.gqa_oracle_e4m3_values.restype = None
        lib.gqa_oracle_rope_append.argtypes = [p, p, p, i, p, i, i, i, i, i, ctypes.c_double, p, p, p]
        lib.gqa_oracle_rope_append.restype = i
        lib.gqa_oracle_decode_paged.argtypes = [p, p, p, i, p, i, i, i, p, i, i, i, i, ctypes.c_double, p, i, p]
        lib.gqa_oracle_decode_paged.restype = i
        lib.gqa_oracle_prefill_chunk.argtypes = [p, p, p, i, i, i, i, i, i, i, i, ctypes.c_double, p, i, p]
        lib.gqa_oracle_meanpool_heads.argtypes = [p, i, i, i, i, i, i, p]
        lib.gqa_oracle_meanpool_heads.restype = i
        lib.gqa_oracle_prefill_chunk.restype = i
        lib.gqa_oracle_num_threads.restype = i
        _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle runs on (OMP_NUM_THREADS, else all cores)."""
    return int(_load().gqa_oracle_num_threads())


def _prep(*arrays):
    dtypes = {a.dtype for a in arrays}
    if len(dtypes) != 1 or next(iter(dtypes)) not in (np.dtype(np.uint16), np.dtype(np.float64)):
        raise TypeError("oracle inputs must all be uint16 (bf16 bits) or all float64")
    etype = 0 if arrays[0].dtype == np.uint16 else 1
    return [np.ascontiguousarray(a) for a in arrays], etype


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def decode(q, k_cache, v_cache, seqlens, scale=None, rows=None, check=True):
    """Decode attention of one new query token per (b, h).

    q [B, Hq, D]; k_cache, v_cache [B, Hkv, Lmax, D]; seqlens [B] (int).
    rows: optional int array [n, 2] of (b, h) to evaluate (default: all, b-major).
    Returns fp64 [B, Hq, D] (rows=None) or [n, D].
    """
    (q, k_cache, v_cache), etype = _prep(q, k_cache, v_cache)
    B, Hq, D = q.shape
    _, Hkv, Lmax, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape or k_cache.shape[0] != B:
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32).reshape(B))
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
    n = B * Hq if r is None else r.shape[0]
    out = np.empty((n, D), dtype=np.float64)
    rc = _load().gqa_oracle_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), etype, _ptr(sl),
                                   B, Hq, Hkv, D, Lmax, float(scale), _ptr(r), n, _ptr(out))
    if check and rc not in (0,):
        raise ValueError(f"oracle decode returned {rc}")
    return out.reshape(B, Hq, D) if r is None else out


def e4m3_values(bytes_u8):
    """Exact fp64 values of OCP FP8 E4M3 bytes (uint8 array)."""
    b = np.ascontiguousarray(np.asarray(bytes_u8, dtype=np.uint8).reshape(-1))
    out = np.empty(b.size, dtype=np.float64)
    _load().gqa_oracle_e4m3_values(_ptr(b), b.size, _ptr(out))
    return out.reshape(np.shape(bytes_u8))


def decode_fp8(q, k8, v8, k_scale, v_scale, seqlens, scale=None, rows=None, check=True):
    """Decode over an FP8 E4M3 cache: real K = e4m3(k8) * k_scale[b, j] (same
    for V).  q [B, Hq, D] (bf16 bits or fp64); k8, v8 uint8 [B, Hkv, Lmax, D];
    k_scale, v_scale [B, Hkv] (or [B * Hkv]).  Returns fp64 like decode()."""
    (q,), etype = _prep(q)
    k8 = np.ascontiguousarray(np.asarray(k8, dtype=np.uint8))
    v8 = np.ascontiguousarray(np.asarray(v8, dtype=np.uint8))
    B, Hq, D = q.shape
    _, Hkv, Lmax, D2 = k8.shape
    if D2 != D or v8.shape != k8.shape or k8.shape[0] != B:
        raise ValueError("shape mismatch")
    ks = np.ascontiguousarray(np.asarray(k_scale, dtype=np.float64).reshape(B * Hkv))
    vs = np.ascontiguousarray(np.asarray(v_scale, dtype=np.float64).reshape(B * Hkv))
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32).reshape(B))
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
    n = B * Hq if r is None else r.shape[0]
    out = np.empty((n, D), dtype=np.float64)
    rc = _load().gqa_oracle_decode_fp8(_ptr(q), etype, _ptr(k8), _ptr(v8), _ptr(ks), _ptr(vs), _ptr(sl),
                                       B, Hq, Hkv, D, Lmax, float(scale), _ptr(r), n, _ptr(out))
    if check and rc not in (0,):
        raise ValueError(f"oracle decode_fp8 returned {rc}")
    return out.reshape(B, Hq, D) if r is None else out


def decode_paged(q, k_pages, v_pages, block_table, seqlens, scale=None, rows=None, check=True):
    """Decode over a paged cache: k_pages, v_pages [num_pages, Hkv, page_size, D];
    block_table [B, max_pages] int (row t of sequence b is row t % page_size
    of page block_table[b, t // page_size]); otherwise like decode()."""
    (q, k_pages, v_pages), etype = _prep(q, k_pages, v_pages)
    B, Hq, D = q.shape
    num_pages, Hkv, page_size, D2 = k_pages.shape
    if D2 != D or v_pages.shape != k_pages.shape:
        raise ValueError("shape mismatch")
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    if bt.ndim != 2 or bt.shape[0] != B:
        raise ValueError("block_table must be [B, max_pages]")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32).reshape(B))
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
    n = B * Hq if r is None else r.shape[0]
    out = np.empty((n, D), dtype=np.float64)
    rc = _load().gqa_oracle_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), etype, _ptr(bt), num_pages, page_size,
                                         bt.shape[1], _ptr(sl), B, Hq, Hkv, D, float(scale), _ptr(r), n, _ptr(out))
    if check and rc != 0:
        raise ValueError(f"oracle decode_paged returned {rc}")
    return out.reshape(B, Hq, D) if r is None else out


def rope_append(q, k_new, v_new, seqlens, Lmax, base=10000.0, check=True):
    """The new token of sequence b at position p = seqlens[b]: rotary embedding
    of its query and key heads at p (Llama rotate-half form, angle
    p * base^(-2i/D) for the pair (i, i + D/2)).  q [B, Hq, D]; k_new, v_new
    [B, Hkv, D] (bf16 bits or fp64).  Returns fp64 (q_out, k_row, v_row):
    the rotated query, and the key / value rows that become cache row p."""
    (q, k_new, v_new), etype = _prep(q, k_new, v_new)
    B, Hq, D = q.shape
    _, Hkv, D2 = k_new.shape
    if D2 != D or v_new.shape != k_new.shape or k_new.shape[0] != B:
        raise ValueError("shape mismatch")
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32).reshape(B))
    q_out = np.empty((B, Hq, D), dtype=np.float64)
    k_row = np.empty((B, Hkv, D), dtype=np.float64)
    v_row = np.empty((B, Hkv, D), dtype=np.float64)
    rc = _load().gqa_oracle_rope_append(_ptr(q), _ptr(k_new), _ptr(v_new), etype, _ptr(sl), B, Hq, Hkv, D,
                                        int(Lmax), float(base), _ptr(q_out), _ptr(k_row), _ptr(v_row))
    if check and rc != 0:
        raise ValueError(f"oracle rope_append returned {rc}")
    return q_out, k_row, v_row


def prefill(q, k, v, causal=True, scale=None, rows=None, check=True):
    """Prefill attention.

    q [B, Hq, L, D]; k, v [B, Hkv, L, D].  rows: optional int array [n, 3] of
    (b, h, i).  Returns fp64 [B, Hq, L, D] (rows=None) or [n, D].
    """
    (q, k, v), etype = _prep(q, k, v)
    B, Hq, L, D = q.shape
    _, Hkv, L2, D2 = k.shape
    if L2 != L or D2 != D or v.shape != k.shape or k.shape[0] != B:
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = B * Hq * L if r is None else r.shape[0]
    out = np.empty((n, D), dtype=np.float64)
    rc = _load().gqa_oracle_prefill(_ptr(q), _ptr(k), _ptr(v), etype, B, L, Hq, Hkv, D,
                                    int(bool(causal)), float(scale), _ptr(r), n, _ptr(out))
    if check and rc != 0:
        raise ValueError(f"oracle prefill returned {rc}")
    return out.reshape(B, Hq, L, D) if r is None else out


def prefill_chunk(q, k, v, causal=True, scale=None, rows=None, check=True):
    """Prefill of the last Lq of Lk tokens: q [B, Hq, Lq, D]; k, v [B, Hkv, Lk, D]
    (Lk >= Lq).  Causal row i is token Lk - Lq + i and sees keys t <= Lk - Lq + i.
    rows: optional (b, h, i) triples.  Returns fp64 [B, Hq, Lq, D] or [n, D]."""
    (q, k, v), etype = _prep(q, k, v)
    B, Hq, Lq, D = q.shape
    _, Hkv, Lk, D2 = k.shape
    if D2 != D or v.shape != k.shape or k.shape[0] != B or Lk < Lq:
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = B * Hq * Lq if r is None else r.shape[0]
    out = np.empty((n, D), dtype=np.float64)
    rc = _load().gqa_oracle_prefill_chunk(_ptr(q), _ptr(k), _ptr(v), etype, B, Lq, Lk, Hq, Hkv, D,
                                          int(bool(causal)), float(scale), _ptr(r), n, _ptr(out))
    if check and rc != 0:
        raise ValueError(f"oracle prefill_chunk returned {rc}")
    return out.reshape(B, Hq, Lq, D) if r is None else out


def meanpool_heads(w, Hkv, mode="mean", check=True):
    """MHA -> GQA checkpoint conversion of a key or value projection: w
    [H, rows, cols] (bf16 bits or fp64; the per-head blocks of the weight)
    becomes [Hkv, rows, cols] fp64, group j's block being the mean of heads
    j*G .. j*G + G - 1 (mode "mean") or head j*G (mode "first")."""
    (w,), etype = _prep(w)
    if w.ndim != 3:
        raise ValueError("w must be [H, rows, cols]")
    H, rows, cols = w.shape
    out = np.empty((int(Hkv), rows, cols), dtype=np.float64)
    m = {"mean": 0, "first": 1}[mode]
    rc = _load().gqa_oracle_meanpool_heads(_ptr(w), etype, H, int(Hkv), rows, cols, m, _ptr(out))
    if check and rc != 0:
        raise ValueError(f"oracle meanpool_heads returned {rc}")
    return out
