"""The parity bar shared by the GPU tests.

|gpu - oracle| <= 1e-2 + 1e-2 |oracle|, element-wise, on the same seeded bf16
inputs.  The kernels accumulate in fp32, round the softmax weights to bf16
before P V and round the output to bf16; at |out| <= ~4 the bf16 output
rounding alone is up to 2^-9 |out|, well inside the bar.
"""
import numpy as np

ATOL = 1e-2
RTOL = 1e-2


def assert_parity(gpu, ref, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, f"{what}: shape {gpu.shape} vs {ref.shape}"
    assert np.isfinite(gpu).all(), f"{what}: non-finite output"
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; worst at {idx}: "
                             f"gpu={gpu[idx]!r} oracle={ref[idx]!r}")
