"""The C ABI of libgqa.so on a machine without a GPU: the library loads, it
exports every function include/gqa.h declares, and argument errors come back
as status codes before anything touches a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "gqa.h")).read()
    return sorted(set(re.findall(r"GQA_API\s+[\w\s\*]*?\b(gqa_\w+)\s*\(", text)))


def test_header_declarations_are_exported(gqa_lib):
    names = declared_functions()
    assert len(names) >= 8
    lib = ctypes.CDLL(gqa_lib.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(gqa_lib.EXPORTED)


def test_library_has_no_driver_link_dependency(gqa_lib):
    """The driver API is reached through the runtime's entry-point query, so the
    library loads where libcuda.so.1 is absent (this test machine)."""
    import subprocess
    out = subprocess.run(["ldd", gqa_lib.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


def test_status_strings(gqa_lib):
    for st in range(0, 7):
        s = gqa_lib.gqa_status_string(st)
        assert s.startswith("GQA_")
    assert gqa_lib.gqa_status_string(99) == "unknown gqa status"


P = ctypes.c_void_p(4096)  # aligned, never dereferenced: every call below fails validation first


@pytest.mark.parametrize("args,status", [
    ((None, P, P, P, P, 2, 8, 2, 64, 128, 0.125), 3),            # NULL q
    ((P, P, P, None, P, 2, 8, 2, 64, 128, 0.125), 3),            # NULL seqlens
    ((P, P, P, P, P, 0, 8, 2, 64, 128, 0.125), 1),               # B = 0
    ((P, P, P, P, P, 2, 8, 3, 64, 128, 0.125), 1),               # Hq % Hkv != 0
    ((P, P, P, P, P, 2, 8, 2, 64, 0, 0.125), 1),                 # Lmax = 0
    ((P, P, P, P, P, 2, 8, 2, 64, 128, 0.0), 1),                 # scale = 0
    ((P, P, P, P, P, 2, 8, 2, 64, 128, float("nan")), 1),        # scale NaN
    ((P, P, P, P, P, 2, 8, 2, 96, 128, 0.125), 2),               # D = 96
    ((P, P, P, P, P, 2, 24, 2, 64, 128, 0.125), 2),              # G = 12
    ((P, P, P, P, P, 2000, 8, 2, 64, 128, 0.125), 2),            # B > 1024
    ((ctypes.c_void_p(4104), P, P, P, P, 2, 8, 2, 64, 128, 0.125), 4),  # q misaligned
    ((P, P, P, ctypes.c_void_p(4098), P, 2, 8, 2, 64, 128, 0.125), 4),  # seqlens misaligned
])
def test_decode_argument_errors(gqa_lib, args, status):
    lib = gqa_lib.load_library()
    assert lib.gqa_decode(*args, None) == status


@pytest.mark.parametrize("args,status", [
    ((None, P, P, P, 1, 16, 4, 2, 128, 1), 3),
    ((P, P, P, P, 1, 0, 4, 2, 128, 1), 1),
    ((P, P, P, P, 1, 16, 4, 3, 128, 1), 1),
    ((P, P, P, P, 1, 16, 4, 2, 128, 2), 1),
    ((P, P, P, P, 1, 16, 4, 2, 80, 1), 2),
    ((P, P, ctypes.c_void_p(4100), P, 1, 16, 4, 2, 128, 1), 4),
])
def test_prefill_argument_errors(gqa_lib, args, status):
    lib = gqa_lib.load_library()
    assert lib.gqa_prefill(*args, None) == status


@pytest.mark.parametrize("args,status", [
    ((None, P, 8, 2, 4, 8, 0), 3),                                 # NULL w
    ((P, ctypes.c_void_p(1 << 20), 8, 3, 4, 8, 0), 1),             # 8 heads into 3 groups
    ((P, ctypes.c_void_p(1 << 20), 8, 2, 0, 8, 0), 1),             # rows = 0
    ((P, ctypes.c_void_p(1 << 20), 8, 2, 4, 8, 2), 1),             # unknown mode
    ((P, ctypes.c_void_p(4096 + 64), 8, 2, 4, 8, 0), 1),           # output overlaps the input
    ((ctypes.c_void_p(4098), ctypes.c_void_p(1 << 20), 8, 2, 4, 8, 0), 4),  # w misaligned
])
def test_meanpool_argument_errors(gqa_lib, args, status):
    lib = gqa_lib.load_library()
    assert lib.gqa_meanpool_kv_heads(*args, None) == status


def test_host_entry_points_validate_first(gqa_lib):
    lib = gqa_lib.load_library()
    assert lib.gqa_decode_host(None, P, P, P, P, 2, 8, 2, 64, 128, 0.125, None) == 3
    assert lib.gqa_decode_host(P, P, P, P, P, 2, 8, 3, 64, 128, 0.125, None) == 1
    assert lib.gqa_prefill_host(P, P, P, P, 1, 16, 4, 2, 96, 1, None) == 2


@pytest.mark.parametrize("shape,tile_keys,ctas", [
    ((2, 8, 2, 64, 128), 64, 4),          # 4 short pairs (2 tiles of 64 keys): one CTA each, no cut
    ((16, 32, 8, 128, 4096), 64, 128),    # 128 pairs nearly fill 148 SMs: one CTA per pair
    ((8, 64, 8, 128, 16384), 64, 148),
    ((64, 32, 1, 128, 2048), 128, 148),   # G = 32: tcgen05 kernel, 128-key blocks
    ((2, 32, 1, 128, 300), 128, 6),       # 2 pairs x 3 blocks
])
def test_decode_plan(gqa_lib, shape, tile_keys, ctas):
    """Split plan: 64-key tiles for G <= 8 (warp-level MMA kernel), 128-key
    blocks for wide groups at D = 128 (tcgen05 kernel); at most one persistent
    CTA per SM (148 on a B300), never more CTAs than tiles, and one CTA per
    (b, kv head) pair when the pairs fill at least three quarters of the SMs."""
    tile, n = gqa_lib.gqa_decode_plan(*shape)
    assert tile == tile_keys
    assert n == ctas


def test_device_status_without_gpu_is_an_error(gqa_lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    flags = ctypes.c_uint32(0)
    st = gqa_lib.load_library().gqa_get_device_status(None, ctypes.byref(flags))
    assert st == gqa_lib.GQA_ERR_NO_DEVICE
