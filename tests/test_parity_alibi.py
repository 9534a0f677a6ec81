"""GPU parity of the ALiBi position bias against the fp64 oracle.

Caller slopes (one per query head, mixing gentle and steep ones) and the library's default
geometric slopes; top-left and bottom-right causal (no mask is refused); every head dim; grouped heads
(including the split-group backward, where one CTA visits several query heads with
different slopes); variable lengths.  The bias joins the scaled scores before the softmax,
so O, LSE and all three gradients change; tolerances are those of the unbiased tests."""
import numpy as np
import pytest

import oracle
from sdpa_workloads import Workload, make_inputs
from sdpa_testlib import (assert_fwd_close, assert_grad_close, assert_lse_close, f64, run_bwd,
                          run_fwd)

pytestmark = pytest.mark.gpu

MODES = {"none": (False, False), "top_left": (True, False), "bottom_right": (True, True)}


def _slopes(h_q, seed):
    rng = np.random.default_rng(seed)
    s = rng.uniform(0.002, 0.6, size=h_q)
    s[0] = 1.5   # steep: a row sees little beyond its diagonal
    return [float(np.float32(v)) for v in s]


def _case(w, mode, alibi, seed, lq=None, lkv=None, backward=False):
    causal, br = MODES[mode]
    cflag = "bottom_right" if br else causal
    x = make_inputs(w, seed=seed, with_do=backward)
    o, lse, dev = run_fwd(w, x, causal=cflag, seq_lens_q=lq, seq_lens_kv=lkv, alibi=alibi)
    slopes = oracle.alibi_default_slopes(w.h_q) if alibi == "default" else alibi
    q64, k64, v64 = f64(x.q), f64(x.k), f64(x.v)
    O, L = oracle.forward(q64, k64, v64, w.scale, causal, lq, lkv, br, alibi_slopes=slopes)
    assert_fwd_close(f64(o), O)
    got_l = lse.cpu().double().numpy()
    inf = np.isneginf(L)
    assert (np.isneginf(got_l) == inf).all()
    assert_lse_close(got_l[~inf], L[~inf])
    if backward:
        dq, dk, dv = run_bwd(w, dev, o, lse, x.do, causal=cflag, seq_lens_q=lq, seq_lens_kv=lkv,
                             alibi=alibi)
        dQ, dK, dV = oracle.backward(q64, k64, v64, f64(x.do), w.scale, causal, lq, lkv, br,
                                     alibi_slopes=slopes)
        assert_grad_close(f64(dq), dQ, "dQ")
        assert_grad_close(f64(dk), dK, "dK")
        assert_grad_close(f64(dv), dV, "dV")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_no_mask_is_refused(d):
    """ALiBi is a penalty on the distance to earlier keys: without a causal mask both entry
    points refuse it (SDPA_ERR_UNSUPPORTED) before anything runs."""
    import torch
    from sdpa_testlib import lib, to_dev
    m = lib()
    w = Workload("t", 1, 2, 2, 130, 130, d, "bf16", backward=True)
    x = make_inputs(w, seed=d, with_do=True)
    q, k, v, do = to_dev(x.q), to_dev(x.k), to_dev(x.v), to_dev(x.do)
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 2, 130, device="cuda")
    with pytest.raises(m.SdpaError) as e:
        m.sdpa_fwd(q, k, v, o, lse, causal=False, alibi=True)
    assert e.value.status == 2 and "causal" in m.sdpa_last_error_string()
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.SdpaError) as e:
        m.sdpa_bwd(q, k, v, o, do, lse, torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), ws,
                   causal=False, alibi=True)
    assert e.value.status == 2
    assert not o.any(), "nothing may run before the refusal"


@pytest.mark.parametrize("mode", ["top_left", "bottom_right"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_forward_caller_slopes(mode, d):
    w = Workload("t", 2, 4, 2, 300, 333, d, "bf16")
    _case(w, mode, _slopes(4, d), seed=d)


@pytest.mark.parametrize("mode", ["top_left", "bottom_right"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_backward_caller_slopes(mode, d):
    w = Workload("t", 2, 4, 2, 260, 300, d, "f16", backward=True)
    _case(w, mode, _slopes(4, d + 1), seed=d + 1, backward=True)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_default_slopes_causal(d):
    w = Workload("t", 1, 8, 8, 384, 384, d, "bf16", backward=True)
    _case(w, "top_left", "default", seed=3 * d, backward=True)


def test_split_groups_per_head_slopes():
    """h_kv = 1 with 16 query heads: the backward pass shares each KV block between CTAs that
    each visit several query heads, each with its own slope."""
    w = Workload("t", 1, 16, 1, 700, 700, 64, "bf16", backward=True)
    _case(w, "top_left", _slopes(16, 5), seed=5, backward=True)


@pytest.mark.parametrize("d", [128, 256])
def test_variable_lengths_bottom_right(d):
    w = Workload("t", 3, 4, 2, 200, 450, d, "bf16", backward=True)
    _case(w, "bottom_right", _slopes(4, 9), seed=d + 9, lq=[200, 37, 1], lkv=[450, 300, 129],
          backward=True)


def test_decode_shape_with_kv_cache():
    """A few new queries against a long cache, bottom-right aligned: the bias is measured
    from each query's own position at the end of the sequence."""
    w = Workload("t", 2, 8, 2, 5, 1500, 128, "bf16")
    _case(w, "bottom_right", "default", seed=21)


def test_zero_slopes_equal_plain_attention():
    """Zero slopes give plain attention up to rounding (the ALiBi kernels visit the key blocks
    in the opposite order, so the sums are not formed in the same order)."""
    w = Workload("t", 1, 2, 2, 256, 256, 128, "bf16", causal=True)
    x = make_inputs(w, seed=4)
    o0, l0, _ = run_fwd(w, x)
    o1, l1, _ = run_fwd(w, x, alibi=[0.0, 0.0])
    assert_fwd_close(f64(o1), f64(o0))
    np.testing.assert_allclose(l1.cpu().numpy(), l0.cpu().numpy(), atol=1e-5)
