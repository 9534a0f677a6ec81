"""Both forward schedules on the same shapes.

Plain 16-bit forward passes at d <= 128 run two Q tiles per CTA, or one Q tile per CTA when
the grid is small (the two softmax warpgroups then split the score columns).  The choice is
made per call; SDPA_FWD_Q_TILES forces either, so that each schedule meets every ragged,
grouped and strided shape here, forward and backward."""
import pytest

import oracle
from sdpa_workloads import Workload, make_inputs
from sdpa_testlib import assert_fwd_close, assert_grad_close, assert_lse_close, f64, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

SHAPES = [
    Workload("t", 2, 2, 2, 333, 333, 64, "f16", causal=True, backward=True),
    Workload("t", 1, 4, 2, 257, 130, 128, "bf16", causal=False, backward=True),
    Workload("t", 2, 6, 3, 200, 300, 128, "f16", layout="bshd", causal=True, backward=True),
    Workload("t", 1, 2, 2, 1, 129, 64, "bf16", causal=False, backward=True),
    Workload("t", 1, 8, 1, 640, 640, 128, "bf16", causal=True, backward=True),
]


@pytest.mark.parametrize("tiles", ["1", "2"])
@pytest.mark.parametrize("i", range(len(SHAPES)))
def test_schedule(tiles, i, monkeypatch):
    monkeypatch.setenv("SDPA_FWD_Q_TILES", tiles)
    w = SHAPES[i]
    x = make_inputs(w, seed=100 + i, with_do=True)
    o, lse, dev = run_fwd(w, x)
    q64, k64, v64 = f64(x.q), f64(x.k), f64(x.v)
    O, L = oracle.forward(q64, k64, v64, w.scale, w.causal)
    assert_fwd_close(f64(o), O)
    assert_lse_close(lse.cpu().double().numpy(), L)
    dq, dk, dv = run_bwd(w, dev, o, lse, x.do)
    dQ, dK, dV = oracle.backward(q64, k64, v64, f64(x.do), w.scale, w.causal)
    assert_grad_close(f64(dq), dQ, "dQ")
    assert_grad_close(f64(dk), dK, "dK")
    assert_grad_close(f64(dv), dV, "dV")
