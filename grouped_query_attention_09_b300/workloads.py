"""Seeded synthetic workloads and the work counts used to measure them.

This module holds input generation and byte/flop accounting only -- none of
the attention arithmetic -- so that both the CUDA path and the fp64 oracle
can be fed the very same bytes.

Inputs: a CPU ``torch.Generator`` seeded per workload draws, in this order,
q, then k, then v as fp32 N(0, 1) and rounds them to bf16 (round to nearest
even); decode workloads with ragged lengths then draw seqlens with
``torch.randint(lo, hi + 1)``.  Cache rows at or beyond seqlens[b] hold N(0, 1)
values too (``tail="randn"``) or NaN (``tail="nan"``, the poison test).

The five workloads are synthetic stand-ins with the shapes of Llama-class
serving (no weights or datasets are involved):

  tiny       decode  B=2,  Hq=8,  Hkv=2, D=64,  L=128 for both sequences
  llama3_8b  decode  B=16, Hq=32, Hkv=8, D=128, L=4096 for every sequence
  llama2_70b decode  B=8,  Hq=64, Hkv=8, D=128, L_b ~ U[4096, 16384], Lmax=16384
  mqa        decode  B=64, Hq=32, Hkv=1, D=128, L_b ~ U[512, 2048],  Lmax=2048
  prefill    causal  B=4,  L=2048, Hq=32, Hkv=8, D=128
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

LOG2E = 1.4426950408889634


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    Lmax: int
    len_lo: int
    len_hi: int
    seed: int

    @property
    def scale(self) -> float:
        return self.D ** -0.5


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    L: int
    Hq: int
    Hkv: int
    D: int
    causal: bool
    seed: int


WORKLOADS = {
    "tiny": DecodeWorkload("tiny", 2, 8, 2, 64, 128, 128, 128, 1),
    "llama3_8b": DecodeWorkload("llama3_8b", 16, 32, 8, 128, 4096, 4096, 4096, 2),
    "llama2_70b": DecodeWorkload("llama2_70b", 8, 64, 8, 128, 16384, 4096, 16384, 3),
    "mqa": DecodeWorkload("mqa", 64, 32, 1, 128, 2048, 512, 2048, 4),
    "prefill": PrefillWorkload("prefill", 4, 2048, 32, 8, 128, True, 5),
}


def _randn_bf16(shape, g):
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def make_decode_inputs(w: DecodeWorkload, tail: str = "randn", q_mult: float = 1.0):
    """Returns CPU tensors (q, k_cache, v_cache, seqlens) of workload w.

    q_mult scales q before its bf16 rounding (the "peaky" variant, q x 8)."""
    g = torch.Generator("cpu").manual_seed(w.seed)
    q = (torch.randn((w.B, w.Hq, w.D), generator=g, dtype=torch.float32) * q_mult).to(torch.bfloat16)
    k = _randn_bf16((w.B, w.Hkv, w.Lmax, w.D), g)
    v = _randn_bf16((w.B, w.Hkv, w.Lmax, w.D), g)
    if w.len_lo == w.len_hi:
        seqlens = torch.full((w.B,), w.len_lo, dtype=torch.int32)
    else:
        seqlens = torch.randint(w.len_lo, w.len_hi + 1, (w.B,), generator=g, dtype=torch.int32)
    if tail == "nan":
        poison_tail(k, v, seqlens)
    elif tail != "randn":
        raise ValueError(tail)
    return q, k, v, seqlens


E4M3_MAX = 448.0
E4M3_NAN = 0x7F


def quantize_kv_fp8(k, v):
    """FP8 E4M3 cache of bf16/fp32 K, V [B, Hkv, L, D]: one scale per (b, kv
    head) for K and one for V, scale = max|x| / 448 over that head's rows, and
    bytes = round-to-nearest-even E4M3 of x / scale (torch's float8_e4m3fn
    conversion).  Returns (k8, v8) uint8 tensors and (k_scale, v_scale) fp32
    [B, Hkv] tensors; the real cache entries are e4m3(byte) * scale."""
    def one(x):
        x = x.float()
        amax = x.abs().amax(dim=(2, 3)).clamp(min=1e-30)
        scale = amax / E4M3_MAX
        q8 = (x / scale[:, :, None, None]).to(torch.float8_e4m3fn)
        return q8.view(torch.uint8), scale.float()
    k8, ks = one(k)
    v8, vs = one(v)
    return k8, v8, ks, vs


def make_decode_fp8_inputs(w: DecodeWorkload, tail: str = "randn", q_mult: float = 1.0):
    """q (bf16), k8, v8 (E4M3 bytes), k_scale, v_scale, seqlens of workload w:
    the bf16 workload's draws (same seed and order), then quantize_kv_fp8.
    tail="nan" writes the E4M3 NaN byte into cache rows t >= seqlens[b]."""
    q, k, v, seqlens = make_decode_inputs(w, q_mult=q_mult)
    k8, v8, ks, vs = quantize_kv_fp8(k, v)
    if tail == "nan":
        for b in range(k8.shape[0]):
            n = max(int(seqlens[b]), 0)
            k8[b, :, n:, :] = E4M3_NAN
            v8[b, :, n:, :] = E4M3_NAN
    elif tail != "randn":
        raise ValueError(tail)
    return q, k8, v8, ks, vs, seqlens


def page_cache(k, v, page_size: int, seed: int, spare_pages: int = 3):
    """Paged copy of a contiguous cache [B, Hkv, Lmax, D]: a pool of pages
    [num_pages, Hkv, page_size, D] (num_pages = B * ceil(Lmax / page_size) +
    spare_pages, pages handed out in a seeded random order, spare pages left
    as noise) and a block table [B, ceil(Lmax / page_size)] int32 with row t of
    sequence b in page block_table[b, t // page_size], row t % page_size.
    Rows past Lmax in a sequence's last page are padding (noise)."""
    B, Hkv, Lmax, D = k.shape
    mp = -(-Lmax // page_size)
    num_pages = B * mp + spare_pages
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g)[: B * mp].to(torch.int32)
    bt = perm.reshape(B, mp).contiguous()
    kp = torch.randn(num_pages, Hkv, page_size, D, generator=g).to(k.dtype)
    vp = torch.randn(num_pages, Hkv, page_size, D, generator=g).to(v.dtype)
    for b in range(B):
        for i in range(mp):
            t0, t1 = i * page_size, min((i + 1) * page_size, Lmax)
            kp[bt[b, i], :, : t1 - t0] = k[b, :, t0:t1]
            vp[bt[b, i], :, : t1 - t0] = v[b, :, t0:t1]
    return kp, vp, bt


def poison_tail(k, v, seqlens):
    """Fills cache rows t >= seqlens[b] with NaN (in place)."""
    for b in range(k.shape[0]):
        n = int(seqlens[b])
        k[b, :, max(n, 0):, :] = float("nan")
        v[b, :, max(n, 0):, :] = float("nan")


def make_prefill_inputs(w: PrefillWorkload, q_mult: float = 1.0):
    g = torch.Generator("cpu").manual_seed(w.seed)
    q = (torch.randn((w.B, w.Hq, w.L, w.D), generator=g, dtype=torch.float32) * q_mult).to(torch.bfloat16)
    k = _randn_bf16((w.B, w.Hkv, w.L, w.D), g)
    v = _randn_bf16((w.B, w.Hkv, w.L, w.D), g)
    return q, k, v


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a CPU bf16 tensor (the bytes the oracle reads)."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------ work accounting
def kv_cache_bytes(b: int, s: int, h: int, l: int, elem_bytes: int = 2) -> int:
    """Bytes of a K plus V cache: 2 tensors x elem_bytes x b x s x h x l.

    For fp16 this is the 4bshl of the GQA paper notes ("QA 相关", the
    Llama2-7B example: b=1, s=4000, h=4096, l=32 -> 2,097,152,000 B)."""
    return 2 * elem_bytes * b * s * h * l


def decode_kv_bytes(seqlens, Hkv: int, D: int, elem_bytes: int = 2) -> int:
    """Algorithmic K/V bytes one decode step must read: the visible rows only,
    once per KV head (sum_b seqlens[b] * Hkv * D * 2 tensors * elem_bytes)."""
    total = int(torch.as_tensor(seqlens).clamp(min=0).sum())
    return kv_cache_bytes(1, total, Hkv * D, 1, elem_bytes)


def decode_kv_bytes_fp8(seqlens, Hkv: int, D: int) -> int:
    """Algorithmic bytes of a decode step over an FP8 cache: one byte per K/V
    element of the visible rows (the per-head scales are negligible)."""
    return decode_kv_bytes(seqlens, Hkv, D, elem_bytes=1)


def decode_flops(seqlens, Hq: int, D: int) -> int:
    """Multiply-add work of a decode step: QK^T and PV, 2 flops per MAC."""
    total = int(torch.as_tensor(seqlens).clamp(min=0).sum())
    return 4 * Hq * D * total


def prefill_flops(B: int, Hq: int, L: int, D: int, causal: bool) -> int:
    """Flops of QK^T and PV over the visible (query, key) pairs: 4*D per pair;
    the causal triangle including the diagonal has L(L+1)/2 pairs per head."""
    pairs = L * (L + 1) // 2 if causal else L * L
    return 4 * B * Hq * D * pairs


def prefill_chunk_flops(B: int, Hq: int, Lq: int, Lk: int, D: int, causal: bool) -> int:
    """Flops of a chunk of Lq queries after Lk - Lq cached tokens: 4*D per
    visible (query, key) pair; causal row i sees Lk - Lq + i + 1 keys."""
    pairs = Lq * (Lk - Lq) + Lq * (Lq + 1) // 2 if causal else Lq * Lk
    return 4 * B * Hq * D * pairs
