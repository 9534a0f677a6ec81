"""GPU parity of the additive bias tensor against the fp64 oracle.

Full and broadcast bias shapes ([b, h], [1, h], [b, 1], [1, 1] leading dims), rows padded to
a multiple of 8 elements with ragged s_kv (the kernels' partial-chunk path), every head dim,
both masks, with dropout and with variable lengths; forward and backward.  The oracle reads
the same 16-bit bias values."""
import numpy as np
import pytest
import torch

import oracle
from sdpa_workloads import Workload, make_inputs
from sdpa_testlib import assert_fwd_close, assert_grad_close, assert_lse_close, f64, run_bwd, run_fwd

pytestmark = pytest.mark.gpu


def _bias(w, nb, nh, seed, dtype, neg_blocks=False):
    """A [nb, nh, s_q, s_kv] bias of the workload's dtype on the GPU, in a buffer whose rows
    are padded to a multiple of 8 elements; returns (view, CPU copy)."""
    g = torch.Generator().manual_seed(seed)
    cpu = (2.0 * torch.randn(nb, nh, w.s_q, w.s_kv, generator=g)).to(dtype)
    if neg_blocks:   # -inf on a sparse pattern of off-diagonal 16 x 16 blocks
        i = torch.arange(w.s_q)[:, None] // 16
        j = torch.arange(w.s_kv)[None, :] // 16
        cpu[..., ((i * 7 + j * 3) % 5 == 0) & (i != j)] = float("-inf")
    pitch = (w.s_kv + 7) // 8 * 8
    buf = torch.zeros(nb, nh, w.s_q, pitch, dtype=dtype, device="cuda")
    buf[..., :w.s_kv] = cpu.cuda()
    return buf[..., :w.s_kv], cpu


def _case(w, nb, nh, seed, backward=True, neg_blocks=False, lq=None, lkv=None, dropout=None,
          bottom_right=False):
    x = make_inputs(w, seed=seed, with_do=backward)
    dt = x.q.dtype
    bdev, bcpu = _bias(w, nb, nh, seed + 1, dt, neg_blocks)
    causal = "bottom_right" if bottom_right else w.causal
    o, lse, dev = run_fwd(w, x, causal=causal, seq_lens_q=lq, seq_lens_kv=lkv, dropout=dropout, bias=bdev)
    bias64 = f64(bcpu)
    keep = None
    if dropout is not None:
        keep = oracle.dropout_keep(w.b, w.h_q, w.s_q, w.s_kv, float(np.float32(dropout[0])), dropout[1], dropout[2])
    pd = float(np.float32(dropout[0])) if dropout else 0.0
    q64, k64, v64 = f64(x.q), f64(x.k), f64(x.v)
    O, L = oracle.forward(q64, k64, v64, w.scale, w.causal or bottom_right, lq, lkv, bottom_right,
                          bias=bias64, dropout_p=pd, keep=keep)
    assert_fwd_close(f64(o) * (1 - pd), O * (1 - pd))
    got_l = lse.cpu().double().numpy()
    inf = np.isneginf(L)
    assert (np.isneginf(got_l) == inf).all()
    assert_lse_close(got_l[~inf], L[~inf])
    if backward:
        dq, dk, dv = run_bwd(w, dev, o, lse, x.do, causal=causal, seq_lens_q=lq, seq_lens_kv=lkv,
                             dropout=dropout, bias=bdev)
        dQ, dK, dV = oracle.backward(q64, k64, v64, f64(x.do), w.scale, w.causal or bottom_right, lq, lkv,
                                     bottom_right, bias=bias64, dropout_p=pd, keep=keep)
        assert_grad_close(f64(dq), dQ, "dQ")
        assert_grad_close(f64(dk), dK, "dK")
        assert_grad_close(f64(dv), dV, "dV")


@pytest.mark.parametrize("nb,nh", [(2, 4), (1, 4), (2, 1), (1, 1)])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_broadcast_shapes_and_head_dims(nb, nh, d):
    w = Workload("t", 2, 4, 2, 200, 333, d, "bf16", causal=False, backward=True)
    _case(w, nb, nh, seed=d + nb * 10 + nh)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_causal_with_masked_blocks(dtype):
    w = Workload("t", 1, 2, 2, 384, 384, 128, dtype, causal=True, backward=True)
    _case(w, 1, 2, seed=3, neg_blocks=True)


def test_with_dropout():
    w = Workload("t", 2, 2, 2, 256, 260, 128, "bf16", causal=True, backward=True)
    _case(w, 2, 2, seed=7, dropout=(0.2, 11, 5))


def test_with_lengths_and_bottom_right():
    w = Workload("t", 3, 2, 2, 150, 270, 128, "bf16", backward=True)
    _case(w, 3, 1, seed=8, lq=[150, 40, 1], lkv=[270, 100, 63], bottom_right=True)


@pytest.mark.parametrize("d", [64, 128])
def test_single_query_row(d):
    # One query row: the bias tile's rows beyond s_q come back zero and are never used.
    w = Workload("t", 2, 2, 2, 1, 300, d, "bf16", backward=False)
    _case(w, 2, 2, seed=12 + d, backward=False)


def test_split_groups():
    w = Workload("t", 1, 16, 1, 512, 512, 64, "f16", causal=True, backward=True)
    _case(w, 1, 16, seed=9)


def test_forward_only_inference_shape():
    w = Workload("t", 4, 12, 12, 1024, 1024, 64, "f16", causal=True)
    _case(w, 1, 12, seed=10, backward=False)


def _dbias_case(w, nb, nh, seed, dropout=None, lq=None, lkv=None, bottom_right=False):
    x = make_inputs(w, seed=seed, with_do=True)
    bdev, bcpu = _bias(w, nb, nh, seed + 1, x.q.dtype)
    causal = "bottom_right" if bottom_right else w.causal
    o, lse, dev = run_fwd(w, x, causal=causal, seq_lens_q=lq, seq_lens_kv=lkv, dropout=dropout, bias=bdev)
    gbuf, _ = _bias(w, nb, nh, seed + 2, x.q.dtype)       # garbage that must be overwritten
    run_bwd(w, dev, o, lse, x.do, causal=causal, seq_lens_q=lq, seq_lens_kv=lkv, dropout=dropout, bias=bdev,
            dbias=gbuf)
    pd = float(np.float32(dropout[0])) if dropout else 0.0
    keep = None
    if dropout is not None:
        keep = oracle.dropout_keep(w.b, w.h_q, w.s_q, w.s_kv, pd, dropout[1], dropout[2])
    want = oracle.bias_gradient(f64(x.q), f64(x.k), f64(x.v), f64(x.do), w.scale, w.causal or bottom_right,
                                f64(bcpu), lq, lkv, bottom_right, dropout_p=pd, keep=keep)
    assert_grad_close(f64(gbuf), want, "dBias")


@pytest.mark.parametrize("nb,nh", [(2, 4), (1, 4), (1, 1)])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_bias_gradient(nb, nh, d):
    w = Workload("t", 2, 4, 2, 200, 333, d, "bf16", causal=True, backward=True)
    _dbias_case(w, nb, nh, seed=40 + d + nh)


def test_bias_gradient_with_dropout_and_lengths():
    w = Workload("t", 3, 2, 2, 150, 270, 128, "f16", backward=True)
    _dbias_case(w, 3, 2, seed=50, dropout=(0.3, 1, 2), lq=[150, 40, 1], lkv=[270, 100, 63], bottom_right=True)
