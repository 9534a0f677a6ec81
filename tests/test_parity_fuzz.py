"""Seeded random combinations of every option, forward and backward, against the oracle.

Each case draws a head dim, dtype, layout, head grouping, sizes (ragged), mask mode, optional
variable lengths (empty batches included), optional ALiBi or an additive bias tensor (with
its gradient), and optional dropout, then compares O, LSE, dQ, dK, dV (and dbias) with the
fp64 oracle.  The per-feature tests cover each option on its own; these cover how they
combine."""
import numpy as np
import pytest
import torch

import oracle
from sdpa_workloads import Workload, make_inputs
from sdpa_testlib import assert_fwd_close, assert_grad_close, assert_lse_close, f64, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

N_CASES = 64


def _draw(i):
    rng = np.random.default_rng(1000 + i)
    d = int(rng.choice([64, 128, 256]))
    dtype = str(rng.choice(["f16", "bf16"]))
    layout = str(rng.choice(["bhsd", "bshd"]))
    h_kv = int(rng.choice([1, 2, 3]))
    h_q = h_kv * int(rng.choice([1, 2, 4]))
    b = int(rng.integers(1, 4))
    s_q = int(rng.integers(1, 300))
    s_kv = int(rng.integers(1, 300))
    mode = str(rng.choice(["none", "top_left", "bottom_right"]))
    lens = None
    if rng.random() < 0.4:
        lens = ([int(x) for x in rng.integers(0, s_q + 1, size=b)],
                [int(x) for x in rng.integers(0, s_kv + 1, size=b)])
    if mode == "top_left" and lens is None:
        s_kv = max(s_kv, s_q)   # every row keeps at least one key
    extra = str(rng.choice(["plain", "alibi", "bias", "dbias"]))
    if extra == "alibi" and mode == "none":
        extra = "plain"   # ALiBi needs a causal mask
    dropout = (float(rng.choice([0.1, 0.4])), int(rng.integers(0, 2 ** 63)), int(rng.integers(0, 1000))) \
        if rng.random() < 0.35 else None
    return dict(d=d, dtype=dtype, layout=layout, h_kv=h_kv, h_q=h_q, b=b, s_q=s_q, s_kv=s_kv,
                mode=mode, lens=lens, extra=extra, dropout=dropout, seed=int(rng.integers(0, 10 ** 6)))


def _padded_bias(w, nb, nh, dt, seed):
    g = torch.Generator().manual_seed(seed)
    cpu = (1.5 * torch.randn(nb, nh, w.s_q, w.s_kv, generator=g)).to(dt)
    pitch = (w.s_kv + 7) // 8 * 8
    buf = torch.zeros(nb, nh, w.s_q, pitch, dtype=dt, device="cuda")
    buf[..., :w.s_kv] = cpu.cuda()
    return buf[..., :w.s_kv], cpu


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_combination(i):
    c = _draw(i)
    causal = c["mode"] != "none"
    br = c["mode"] == "bottom_right"
    w = Workload("fuzz", c["b"], c["h_q"], c["h_kv"], c["s_q"], c["s_kv"], c["d"], c["dtype"],
                 layout=c["layout"], causal=causal, backward=True)
    x = make_inputs(w, seed=c["seed"], with_do=True)
    lq, lkv = c["lens"] if c["lens"] is not None else (None, None)
    cflag = "bottom_right" if br else causal
    kw = dict(causal=cflag, seq_lens_q=lq, seq_lens_kv=lkv, dropout=c["dropout"])
    slopes = bias_dev = bias64 = dbias = None
    if c["extra"] == "alibi":
        slopes = [float(np.float32(s)) for s in np.random.default_rng(i).uniform(0.01, 0.5, size=w.h_q)]
        kw["alibi"] = slopes
    elif c["extra"] in ("bias", "dbias"):
        nb = 1 if i % 2 else w.b
        bias_dev, bcpu = _padded_bias(w, nb, w.h_q, x.q.dtype, c["seed"] + 1)
        bias64 = f64(bcpu)
        kw["bias"] = bias_dev
    o, lse, dev = run_fwd(w, x, **kw)
    pd = float(np.float32(c["dropout"][0])) if c["dropout"] else 0.0
    keep = None
    if c["dropout"]:
        keep = oracle.dropout_keep(w.b, w.h_q, w.s_q, w.s_kv, pd, c["dropout"][1], c["dropout"][2])
    q64, k64, v64, do64 = f64(x.q), f64(x.k), f64(x.v), f64(x.do)
    O, L = oracle.forward(q64, k64, v64, w.scale, causal, lq, lkv, br, alibi_slopes=slopes,
                          dropout_p=pd, keep=keep, bias=bias64)
    assert_fwd_close(f64(o) * (1 - pd), O * (1 - pd))
    got_l = lse.cpu().double().numpy()
    inf = np.isneginf(L)
    assert (np.isneginf(got_l) == inf).all(), "rows without a visible key must have LSE = -inf"
    if (~inf).any():
        assert_lse_close(got_l[~inf], L[~inf])
    if c["extra"] == "dbias":
        dbias, _ = _padded_bias(w, bias_dev.shape[0], w.h_q, x.q.dtype, c["seed"] + 2)
    bkw = dict(kw)
    if dbias is not None:
        bkw["dbias"] = dbias
    dq, dk, dv = run_bwd(w, dev, o, lse, x.do, **bkw)
    dQ, dK, dV = oracle.backward(q64, k64, v64, do64, w.scale, causal, lq, lkv, br, alibi_slopes=slopes,
                                 dropout_p=pd, keep=keep, bias=bias64)
    # Where dQ and dK vanish exactly (every valid row sees a single key, so dS = 0), what is
    # left on the GPU comes from Delta = rowsum(dO * O) with O rounded to the output dtype:
    # |dS_ij| <= P_ij |dDelta_i|, |dDelta_i| <= d max|dO| eps max|O|, max|O| <= max|V| / (1 - p).
    eps = 2.0 ** -8 if c["dtype"] == "bf16" else 2.0 ** -11
    d_delta = w.d * np.abs(do64).max() * eps * np.abs(v64).max() / (1.0 - pd)
    zero_tol = {"dQ": abs(w.scale) * d_delta * np.abs(k64).max(),
                "dK": abs(w.scale) * d_delta * np.abs(q64).max() * w.h_q // w.h_kv, "dV": 1e-4}
    for got, want, name in ((dq, dQ, "dQ"), (dk, dK, "dK"), (dv, dV, "dV")):
        assert_grad_close(f64(got), want, f"{name} (case {c})", zero_tol=max(zero_tol[name], 1e-4))
    if dbias is not None:
        want = oracle.bias_gradient(q64, k64, v64, do64, w.scale, causal, bias64, lq, lkv, br,
                                    dropout_p=pd, keep=keep)
        # dbias is dS itself (summed over a broadcast batch): the same residue, without K or Q.
        n_sum = w.b if bias_dev.shape[0] == 1 else 1
        assert_grad_close(f64(dbias), want, f"dbias (case {c})", zero_tol=max(d_delta * n_sum, 1e-4))
