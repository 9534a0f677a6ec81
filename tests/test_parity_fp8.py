"""GPU parity of the FP8 (E4M3) forward pass against the fp64 oracle.

The oracle decodes the same E4M3 bytes exactly and multiplies by the per-tensor descales;
the GPU output must be within relative L2 <= 6e-2 (the kernel also rounds P to E4M3)."""
import pytest
import torch

import oracle
from sdpa_workloads import Workload, make_inputs
from sdpa_testlib import FP8_REL_L2, f64, rel_l2, run_fwd, assert_lse_close

pytestmark = pytest.mark.gpu


def _check(w: Workload, seed=0, out_dtype=torch.bfloat16):
    x = make_inputs(w, seed=seed, with_do=False)
    o, lse, _ = run_fwd(w, x, out_dtype=out_dtype)
    q64, k64, v64 = f64(x.q, x.descale_q), f64(x.k, x.descale_k), f64(x.v, x.descale_v)
    O, L = oracle.forward(q64, k64, v64, w.scale, w.causal)
    got = f64(o)
    assert torch.isfinite(o.float()).all()
    e = rel_l2(got, O)
    assert e <= FP8_REL_L2, f"rel-L2 {e:.3e}"
    # LSE uses only the E4M3 scores (no P rounding), so it is as tight as the 16-bit path.
    assert_lse_close(lse.cpu().double().numpy(), L)


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("s", [256, 300])
def test_fp8_forward(d, causal, s):
    _check(Workload("t", 2, 2, 2, s, s, d, "e4m3", causal=causal), seed=d + s)


def test_fp8_forward_f16_output_grouped_bshd():
    _check(Workload("t", 1, 4, 2, 384, 384, 256, "e4m3", layout="bshd", causal=False), seed=1,
           out_dtype=torch.float16)
