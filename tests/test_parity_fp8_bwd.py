"""GPU parity of the FP8 backward pass (HYBRID recipe: E4M3 Q, K, V; E5M2 dO) against the
fp64 oracle on the decoded inputs.

Isolated check: O and LSE come from the oracle (rounded to the output dtype / fp32), so the
only difference from the oracle's gradients is the kernels' own 16-bit arithmetic on the
exactly widened FP8 values — the tolerance is the 16-bit one.  End-to-end check: O and LSE
come from the FP8 forward kernel, whose E4M3 rounding of P enters Delta = rowsum(dO∘O); the
tolerance there is the FP8 one."""
import numpy as np
import pytest
import torch

import oracle
from sdpa_workloads import Workload, make_inputs
from sdpa_testlib import FP8_REL_L2, assert_grad_close, f64, rel_l2, run_bwd_fp8, run_fwd

pytestmark = pytest.mark.gpu


def _fp8_bwd(w, x, o, lse, out_dtype):
    return run_bwd_fp8(w, x, o, lse, out_dtype)


def _decoded(x):
    return (f64(x.q, x.descale_q), f64(x.k, x.descale_k), f64(x.v, x.descale_v),
            f64(x.do, x.descale_do))


def _isolated(w, out_dtype=torch.bfloat16, seed=0, dout=None):
    x = make_inputs(w, seed=seed, with_do=True)
    if dout is not None:
        x.do, x.descale_do = dout(x)
    q64, k64, v64, do64 = _decoded(x)
    O, L = oracle.forward(q64, k64, v64, w.scale, w.causal)
    o = torch.empty_strided(x.q.shape, x.q.stride(), dtype=out_dtype, device="cuda")
    o.copy_(torch.from_numpy(O).to(out_dtype))
    lse = torch.from_numpy(L).float().cuda()
    dq, dk, dv = _fp8_bwd(w, x, o, lse, out_dtype)
    dQ, dK, dV = oracle.backward(q64, k64, v64, do64, w.scale, w.causal)
    assert_grad_close(f64(dq), dQ, "dQ")
    assert_grad_close(f64(dk), dK, "dK")
    assert_grad_close(f64(dv), dV, "dV")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_isolated_head_dims_and_masks(d, causal):
    _isolated(Workload("t", 2, 4, 2, 260, 300, d, "e4m3", causal=causal, backward=True), seed=d)


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_isolated_output_dtypes_bshd_gqa(out_dtype):
    _isolated(Workload("t", 2, 8, 2, 333, 333, 128, "e4m3", layout="bshd", causal=True, backward=True),
              out_dtype=out_dtype, seed=5)


def test_isolated_e4m3_gradient_input():
    """dO may also come as E4M3 (more mantissa, less range)."""
    from sdpa_workloads import quantize_e4m3

    def as_e4m3(x):
        full = torch.from_numpy(f64(x.do, x.descale_do)).float()
        q8, dsc = quantize_e4m3(full)
        return q8, dsc
    _isolated(Workload("t", 1, 4, 4, 256, 256, 128, "e4m3", causal=True, backward=True), seed=9,
              dout=as_e4m3)


def test_isolated_split_groups():
    _isolated(Workload("t", 1, 16, 1, 512, 512, 64, "e4m3", causal=True, backward=True), seed=3)


@pytest.mark.parametrize("d", [128, 256])
def test_end_to_end_with_the_fp8_forward(d):
    """O and LSE from the E4M3 forward kernel (bf16 O), then the FP8 backward."""
    w = Workload("t", 2, 4, 4, 384, 384, d, "e4m3", causal=True, backward=True)
    x = make_inputs(w, seed=d + 1, with_do=True)
    o, lse, _ = run_fwd(w, x)
    dq, dk, dv = _fp8_bwd(w, x, o, lse, torch.bfloat16)
    q64, k64, v64, do64 = _decoded(x)
    dQ, dK, dV = oracle.backward(q64, k64, v64, do64, w.scale, w.causal)
    for g, r, n in ((dq, dQ, "dQ"), (dk, dK, "dK"), (dv, dV, "dV")):
        err = rel_l2(f64(g), r)
        assert err <= FP8_REL_L2, f"{n}: rel L2 {err:.3e}"
