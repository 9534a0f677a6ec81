"""GPU parity of the forward pass against the fp64 oracle (full outputs, small shapes).

Shapes span several 128-row tiles and ragged tails, both masks, every head dim, both
16-bit dtypes, grouped heads, BSHD strides, s_q != s_kv, single rows, and the degenerate
scales.  Tolerances: max |O - O_ref| <= 2e-2 and mean <= 2e-3; |LSE - LSE_ref| <= 1e-3."""
import pytest
import torch

import oracle
from sdpa_workloads import Workload, make_inputs, tiny
from sdpa_testlib import (assert_fwd_close, assert_lse_close, f64, run_fwd)

pytestmark = pytest.mark.gpu


def _check(w: Workload, seed: int = 0, with_lse: bool = True):
    x = make_inputs(w, seed=seed, with_do=False)
    o, lse, _ = run_fwd(w, x, with_lse=with_lse)
    O, L = oracle.forward(f64(x.q), f64(x.k), f64(x.v), w.scale, w.causal)
    assert_fwd_close(f64(o), O)
    if with_lse:
        assert_lse_close(lse.cpu().double().numpy(), L)


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_config(causal):
    _check(tiny(causal))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("s", [256, 333])
def test_head_dims_dtypes_masks(dtype, d, causal, s):
    _check(Workload("t", 2, 2, 2, s, s, d, dtype, causal=causal), seed=d + s)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("s_q,s_kv", [(100, 300), (300, 130), (1, 1), (1, 257), (129, 1)])
def test_unequal_lengths(causal, s_q, s_kv):
    _check(Workload("t", 1, 2, 2, s_q, s_kv, 128, "bf16", causal=causal), seed=s_q * 7 + s_kv)


@pytest.mark.parametrize("h_q,h_kv", [(4, 2), (8, 1), (6, 3)])
@pytest.mark.parametrize("d", [64, 128])
def test_grouped_heads(h_q, h_kv, d):
    _check(Workload("t", 2, h_q, h_kv, 192, 192, d, "bf16", causal=True), seed=h_q * h_kv)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_bshd_strides(d, causal):
    _check(Workload("t", 2, 3, 3, 200, 200, d, "f16", layout="bshd", causal=causal), seed=5)


def test_bshd_equals_bhsd_bit_for_bit():
    w1 = Workload("t", 2, 3, 3, 300, 300, 64, "f16", layout="bshd", causal=True)
    x = make_inputs(w1, seed=9, with_do=False)
    o1, l1, _ = run_fwd(w1, x)
    x.q, x.k, x.v = x.q.contiguous(), x.k.contiguous(), x.v.contiguous()
    o2, l2, _ = run_fwd(w1, x)
    assert torch.equal(o1.cpu(), o2.cpu())
    assert torch.equal(l1.cpu(), l2.cpu())


def test_inference_without_stats():
    _check(Workload("t", 1, 2, 2, 300, 300, 128, "bf16", causal=True), with_lse=False)


@pytest.mark.parametrize("scale", [0.0, -0.09, 0.5])
def test_scale_values(scale):
    _check(Workload("t", 1, 2, 2, 200, 260, 128, "bf16", causal=False, attn_scale=scale), seed=3)
    _check(Workload("t", 1, 2, 2, 200, 200, 64, "f16", causal=True, attn_scale=scale), seed=4)


@pytest.mark.parametrize("causal", [False, True])
def test_longer_sequence(causal):
    _check(Workload("t", 1, 2, 1, 1280, 1280, 128, "bf16", causal=causal), seed=11)


def test_causal_first_and_last_rows_on_gpu():
    """Row 0 returns V_0 exactly up to rounding; the last causal row equals the full one."""
    w = Workload("t", 1, 2, 2, 256, 256, 128, "bf16", causal=True)
    x = make_inputs(w, seed=21, with_do=False)
    oc, _, _ = run_fwd(w, x)
    of, _, _ = run_fwd(Workload("t", 1, 2, 2, 256, 256, 128, "bf16", causal=False), x)
    assert torch.equal(oc[:, :, 0].cpu(), x.v[:, :, 0])
    assert (oc[:, :, -1].float() - of[:, :, -1].float()).abs().max().item() <= 1e-2
