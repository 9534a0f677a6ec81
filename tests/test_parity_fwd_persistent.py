"""Persistent forward CTAs: each CTA walks several work units (query tiles of one head) in a
fixed back-and-forth order, loading the next unit's tiles while it finishes the current one.

The schedule is chosen per call for plain 16-bit problems at d <= 128 whose units fill one to
four waves of the GPU; SDPA_FWD_PERSIST=N forces N CTAs, so that one CTA walking every unit,
a few CTAs walking many, and the default one-unit-per-CTA launch all meet the same ragged,
grouped, strided, padded and bottom-right shapes, with one and with two Q tiles per unit."""
import numpy as np
import pytest

import oracle
from sdpa_workloads import Workload, make_inputs
from sdpa_testlib import assert_fwd_close, assert_grad_close, assert_lse_close, f64, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

CASES = [
    (Workload("t", 2, 3, 3, 700, 700, 64, "f16", causal=True, backward=True), None, None, True),
    (Workload("t", 1, 4, 2, 1000, 600, 128, "bf16", causal=False, backward=True), None, None, True),
    (Workload("t", 2, 6, 3, 300, 300, 128, "f16", layout="bshd", causal=True, backward=False), None, None, False),
    (Workload("t", 3, 2, 2, 520, 520, 128, "bf16", causal=True, backward=True), [520, 131, 0], [520, 131, 0], True),
    (Workload("t", 2, 4, 2, 300, 900, 64, "bf16", causal=True, backward=False), [300, 77], [900, 400], "bottom_right"),
]


@pytest.mark.parametrize("ctas", ["1", "3", "0"])
@pytest.mark.parametrize("tiles", ["1", "2"])
@pytest.mark.parametrize("i", range(len(CASES)))
def test_persistent_schedule(ctas, tiles, i, monkeypatch):
    monkeypatch.setenv("SDPA_FWD_PERSIST", ctas)
    monkeypatch.setenv("SDPA_FWD_Q_TILES", tiles)
    w, lq, lkv, mode = CASES[i]
    causal = "bottom_right" if mode == "bottom_right" else w.causal
    br = mode == "bottom_right"
    x = make_inputs(w, seed=300 + i, with_do=w.backward)
    o, lse, dev = run_fwd(w, x, causal=causal, seq_lens_q=lq, seq_lens_kv=lkv)
    q64, k64, v64 = f64(x.q), f64(x.k), f64(x.v)
    O, L = oracle.forward(q64, k64, v64, w.scale, w.causal, lq, lkv, br)
    assert_fwd_close(f64(o), O)
    got_l = lse.cpu().double().numpy()
    inf = np.isneginf(L)
    assert (np.isneginf(got_l) == inf).all()
    assert_lse_close(got_l[~inf], L[~inf])
    if w.backward:
        dq, dk, dv = run_bwd(w, dev, o, lse, x.do, causal=causal, seq_lens_q=lq, seq_lens_kv=lkv)
        dQ, dK, dV = oracle.backward(q64, k64, v64, f64(x.do), w.scale, w.causal, lq, lkv, br)
        assert_grad_close(f64(dq), dQ, "dQ")
        assert_grad_close(f64(dk), dK, "dK")
        assert_grad_close(f64(dv), dV, "dV")
