"""GPU parity of the backward pass against the fp64 oracle (full gradients, small shapes).

The CUDA forward pass supplies O and LSE (as in training), then dQ, dK, dV must match
the oracle's analytic gradients within relative L2 <= 1e-2."""
import numpy as np
import pytest
import torch

import oracle
from sdpa_workloads import Workload, make_inputs, tiny
from sdpa_testlib import assert_grad_close, f64, run_bwd, run_fwd

pytestmark = pytest.mark.gpu


def _check(w: Workload, seed: int = 0):
    x = make_inputs(w, seed=seed, with_do=True)
    o, lse, dev = run_fwd(w, x)
    dq, dk, dv = run_bwd(w, dev, o, lse, x.do)
    q64, k64, v64, do64 = f64(x.q), f64(x.k), f64(x.v), f64(x.do)
    dQ, dK, dV = oracle.backward(q64, k64, v64, do64, w.scale, w.causal)
    assert_grad_close(f64(dq), dQ, "dQ")
    assert_grad_close(f64(dk), dK, "dK")
    assert_grad_close(f64(dv), dV, "dV")
    return dq, dk, dv


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_config(causal):
    _check(tiny(causal))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("s", [256, 333])
def test_head_dims_dtypes_masks(dtype, d, causal, s):
    _check(Workload("t", 2, 2, 2, s, s, d, dtype, causal=causal, backward=True), seed=d + s)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("s_q,s_kv", [(100, 300), (300, 130), (1, 1), (129, 1), (1, 200)])
def test_unequal_lengths(causal, s_q, s_kv):
    _check(Workload("t", 1, 2, 2, s_q, s_kv, 128, "bf16", causal=causal, backward=True),
           seed=s_q + 3 * s_kv)


@pytest.mark.parametrize("h_q,h_kv", [(4, 2), (8, 1), (6, 3)])
@pytest.mark.parametrize("d", [64, 128])
def test_grouped_heads(h_q, h_kv, d):
    _check(Workload("t", 2, h_q, h_kv, 192, 192, d, "bf16", causal=True, backward=True),
           seed=h_q + h_kv)


@pytest.mark.parametrize("d", [64, 128])
def test_bshd_strides(d):
    _check(Workload("t", 2, 3, 3, 200, 200, d, "f16", layout="bshd", causal=True, backward=True),
           seed=8)


@pytest.mark.parametrize("scale", [0.0, -0.09])
def test_scale_values(scale):
    _check(Workload("t", 1, 2, 2, 200, 200, 64, "bf16", causal=True, backward=True,
                    attn_scale=scale), seed=2)


def test_longer_sequence_and_invariants():
    w = Workload("t", 1, 4, 2, 1280, 1280, 128, "bf16", causal=True, backward=True)
    dq, dk, dv = _check(w, seed=13)
    x = make_inputs(w, seed=13, with_do=True)
    # Σ_j dK_j = 0 per KV head; Σ_j dV_j = Σ over the group's rows of dO
    sk = dk.float().sum(dim=2).cpu().numpy()
    assert np.abs(sk).max() <= 2e-2 * max(1.0, np.abs(dk.float().cpu().numpy()).sum(2).max())
    sv = dv.float().sum(dim=2).cpu().numpy()
    want = x.do.float().reshape(1, 2, 2, 1280, 128).sum(dim=(2, 3)).numpy()
    assert np.abs(sv - want).max() <= 1e-2 * max(1.0, np.abs(want).max())


def test_grouped_heads_without_split():
    """Enough CTAs that each KV head's whole group stays in one CTA (no fp32 dK/dV pass)."""
    _check(Workload("t", 4, 32, 16, 1280, 1280, 128, "bf16", causal=True, backward=True), seed=17)


@pytest.mark.parametrize("h_kv", [1, 2])
def test_split_groups_small_batch(h_kv):
    """Few KV heads: the query heads of a group are split over several CTAs."""
    _check(Workload("t", 1, 16, h_kv, 700, 700, 64, "f16", causal=False, backward=True), seed=h_kv)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("s_q,s_kv", [(100, 300), (300, 130), (1, 1), (65, 200)])
def test_d256_unequal_lengths(causal, s_q, s_kv):
    _check(Workload("t", 1, 2, 2, s_q, s_kv, 256, "bf16", causal=causal, backward=True),
           seed=s_q + 5 * s_kv)


@pytest.mark.parametrize("h_q,h_kv", [(4, 2), (8, 1)])
def test_d256_grouped_heads_and_bshd(h_q, h_kv):
    _check(Workload("t", 2, h_q, h_kv, 200, 200, 256, "f16", layout="bshd", causal=True,
                    backward=True), seed=h_q)
