"""GPU parity for variable sequence lengths (padding mask) and bottom-right causal alignment.

Padded batches (including one with no valid rows), KV-cache decoding shapes (few queries
against a long key sequence, bottom-right aligned), every head dim, forward, backward and
the FP8 forward.  Where a row sees no key the result must be exactly O = 0, LSE = -inf."""
import numpy as np
import pytest
import torch

import oracle
from sdpa_workloads import Workload, make_inputs
from sdpa_testlib import (FP8_REL_L2, assert_fwd_close, assert_grad_close, f64, rel_l2, run_bwd,
                          run_fwd)

pytestmark = pytest.mark.gpu

MODES = {"none": (False, False), "top_left": (True, False), "bottom_right": (True, True)}


def _lse_check(got: np.ndarray, want: np.ndarray):
    inf = np.isneginf(want)
    assert (np.isneginf(got) == inf).all(), "rows without a visible key must have LSE = -inf"
    if (~inf).any():
        assert np.abs(got[~inf] - want[~inf]).max() <= 1e-3


def _fwd_case(w, mode, lq, lkv, seed, out_dtype=torch.bfloat16, fp8=False):
    causal, br = MODES[mode]
    x = make_inputs(w, seed=seed, with_do=w.backward)
    o, lse, dev = run_fwd(w, x, causal=("bottom_right" if br else causal), seq_lens_q=lq,
                          seq_lens_kv=lkv, out_dtype=out_dtype)
    ds = (x.descale_q, x.descale_k, x.descale_v) if fp8 else (1.0, 1.0, 1.0)
    q64, k64, v64 = f64(x.q, ds[0]), f64(x.k, ds[1]), f64(x.v, ds[2])
    O, L = oracle.forward(q64, k64, v64, w.scale, causal, lq, lkv, br)
    got = f64(o)
    if fp8:
        assert rel_l2(got, O) <= FP8_REL_L2
    else:
        assert_fwd_close(got, O)
    _lse_check(lse.cpu().double().numpy(), L)
    return x, o, lse, dev


@pytest.mark.parametrize("mode", ["none", "top_left", "bottom_right"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_padded_batches_forward(mode, d):
    w = Workload("t", 3, 4, 2, 300, 333, d, "bf16")
    _fwd_case(w, mode, [300, 129, 0], [333, 200, 17], seed=d)


@pytest.mark.parametrize("mode", ["none", "top_left", "bottom_right"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_padded_batches_backward(mode, d):
    causal, br = MODES[mode]
    w = Workload("t", 3, 4, 2, 260, 300, d, "f16", backward=True)
    lq, lkv = [260, 100, 3], [300, 150, 257]
    x, o, lse, dev = _fwd_case(w, mode, lq, lkv, seed=d + 1)
    dq, dk, dv = run_bwd(w, dev, o, lse, x.do, causal=("bottom_right" if br else causal),
                         seq_lens_q=lq, seq_lens_kv=lkv)
    dQ, dK, dV = oracle.backward(f64(x.q), f64(x.k), f64(x.v), f64(x.do), w.scale, causal, lq, lkv, br)
    assert_grad_close(f64(dq), dQ, "dQ")
    assert_grad_close(f64(dk), dK, "dK")
    assert_grad_close(f64(dv), dV, "dV")


@pytest.mark.parametrize("s_q", [1, 7, 130])
def test_kv_cache_decode_bottom_right(s_q):
    """Few new queries against a long cache: bottom-right alignment, no explicit lengths."""
    w = Workload("t", 2, 8, 2, s_q, 1000, 128, "bf16", backward=True)
    x, o, lse, dev = _fwd_case(w, "bottom_right", None, None, seed=s_q)
    dq, dk, dv = run_bwd(w, dev, o, lse, x.do, causal="bottom_right")
    dQ, dK, dV = oracle.backward(f64(x.q), f64(x.k), f64(x.v), f64(x.do), w.scale, True, None,
                                 None, True)
    assert_grad_close(f64(dq), dQ, "dQ")
    assert_grad_close(f64(dk), dK, "dK")
    assert_grad_close(f64(dv), dV, "dV")


def test_bottom_right_more_queries_than_keys():
    """len_q > len_kv: the first len_q - len_kv rows see no key at all."""
    w = Workload("t", 1, 2, 2, 400, 150, 64, "bf16", backward=True)
    x, o, lse, dev = _fwd_case(w, "bottom_right", None, None, seed=3)
    assert (o[:, :, :250].float() == 0).all()
    dq, dk, dv = run_bwd(w, dev, o, lse, x.do, causal="bottom_right")
    dQ, dK, dV = oracle.backward(f64(x.q), f64(x.k), f64(x.v), f64(x.do), w.scale, True, None,
                                 None, True)
    assert_grad_close(f64(dq), dQ, "dQ")
    assert_grad_close(f64(dk), dK, "dK")
    assert_grad_close(f64(dv), dV, "dV")


@pytest.mark.parametrize("mode", ["top_left", "bottom_right"])
def test_padded_batches_fp8(mode):
    w = Workload("t", 2, 2, 2, 300, 320, 256, "e4m3")
    _fwd_case(w, mode, [300, 77], [320, 200], seed=9, fp8=True)
