"""The FMA-pipe exp2 used for part of the softmax exponentials: relative error against the
exact value (fp64) and against CUDA's exp2f, over the range the kernels feed it."""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe():
    d = tempfile.mkdtemp(prefix="exp2probe_")
    so = os.path.join(d, "exp2_probe.so")
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                           "-Xcompiler", "-fPIC", os.path.join(HERE, "kernels", "exp2_probe.cu"),
                           "-o", so])
    lib = ctypes.CDLL(so)
    lib.exp2_probe.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int]
    return lib


def test_exp2_poly_error_bound(probe):
    x = torch.cat([torch.linspace(-125.0, 9.0, 1 << 20), torch.linspace(-1.0, 1.0, 1 << 16),
                   torch.tensor([0.0, -0.5, 0.5, -1.5, 8.0, -124.5])]).float().cuda()
    poly, ref = torch.empty_like(x), torch.empty_like(x)
    assert probe.exp2_probe(x.data_ptr(), poly.data_ptr(), ref.data_ptr(), x.numel()) == 0
    xs = x.cpu().double().numpy()
    exact = np.exp2(xs)
    rel = np.abs(poly.cpu().double().numpy() - exact) / exact
    assert rel.max() <= 1.0e-4, rel.max()
    rel_cuda = np.abs(poly.cpu().double().numpy() - ref.cpu().double().numpy()) / exact
    assert rel_cuda.max() <= 1.1e-4, rel_cuda.max()
    # clamped below -125
    y = torch.tensor([-200.0, -1e30], device="cuda")
    py, ry = torch.empty_like(y), torch.empty_like(y)
    assert probe.exp2_probe(y.data_ptr(), py.data_ptr(), ry.data_ptr(), 2) == 0
    assert (py.cpu() >= 0).all() and (py.cpu() <= 2.0 ** -124).all()
