"""Error of fast_exp, the exponential the tensor-core kernels use for the decay factors.

fast_exp(x) evaluates exp(x) as 2^(x log2 e) with the hardware base-2 exponential
(ex2.approx.ftz), which flushes results below the smallest normal float to zero. The
kernels feed it the cumulative log-decays g_t and -g_t of a chunk in the ratio form
(|g| <= 80) and differences g_t - g_i <= 0 in the exponential form. Two rounding steps
bound its relative error: the product x log2 e rounded to fp32 (|x| 2^-24 relative in
the result) and the approximation of 2^y (about 2^-22 relative). Over |x| <= 87, where
exp(x) is a normal float, that is below 8e-6, far under the 2^-9 of the bf16 operands
the factors scale. Below the normal range the result is flushed to zero.

The probe kernel is compiled from tests/fast_exp_probe.cu with nvcc and compared with
CUDA's expf on a dense grid of the input range.
"""
import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = tempfile.mkdtemp(prefix="fast_exp_probe_")
    lib = os.path.join(tmp, "probe.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-shared", "-Xcompiler", "-fPIC", "-I", os.path.join(HERE, "..", "include"),
                    os.path.join(HERE, "fast_exp_probe.cu"), "-o", lib], check=True)
    fn = ctypes.CDLL(lib).fast_exp_probe
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int]
    fn.restype = ctypes.c_int
    return fn


def evaluate(fn, x):
    xd = torch.tensor(x, dtype=torch.float32, device="cuda")
    fast, ref = torch.empty_like(xd), torch.empty_like(xd)
    assert fn(xd.data_ptr(), fast.data_ptr(), ref.data_ptr(), xd.numel()) == 0
    return fast.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)


def test_relative_error_over_the_normal_range(probe):
    # every float32 in [-87, 0] at a stride of ~1e-4, plus the ends and integers
    x = np.concatenate([np.linspace(-87.0, 0.0, 870_001, dtype=np.float32),
                        np.arange(-87, 1, dtype=np.float32)])
    fast, ref = evaluate(probe, x)
    exact = np.exp(x.astype(np.float64))
    rel_fast = np.abs(fast - exact) / exact
    rel_ref = np.abs(ref - exact) / exact
    assert rel_fast.max() < 8e-6, (rel_fast.max(), x[rel_fast.argmax()])
    # CUDA's expf, on the same grid, for scale (it is correctly rounded to within 2 ulp)
    assert rel_ref.max() < 3e-7
    # the range the ratio form uses, |g| <= 80, both signs
    xr = np.linspace(-80.0, 80.0, 160_001, dtype=np.float32)
    fast, _ = evaluate(probe, xr)
    exact = np.exp(xr.astype(np.float64))
    assert (np.abs(fast - exact) / exact).max() < 8e-6
    assert fast[0] == fast[0] and fast[-1] < np.finfo(np.float32).max  # finite at both ends


def test_flush_below_the_normal_range(probe):
    x = np.linspace(-120.0, -88.0, 1001, dtype=np.float32)
    fast, _ = evaluate(probe, x)
    smallest_normal = np.finfo(np.float32).tiny
    assert np.all((fast == 0.0) | (fast >= smallest_normal * 0.999))
    assert np.all(fast < 2.0 * np.exp(-87.0))
    assert fast[0] == 0.0  # exp(-120) is far below the normal range: flushed


def test_exact_points(probe):
    fast, _ = evaluate(probe, np.array([0.0, -np.log(2.0)], dtype=np.float32))
    assert fast[0] == 1.0
    assert abs(fast[1] - 0.5) < 1e-6
