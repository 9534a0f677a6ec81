"""GPU parity at the full workload sizes, on sampled outputs.

Each configuration runs exactly as bench.py launches it (same shapes, dtypes, layouts).
The oracle then checks what it can compute cheaply and exactly:
  * O and LSE of seeded (batch, head, row) triples (each row needs only its KV head);
  * dQ of the same rows;
  * full dK and dV of seeded (batch, KV head) pairs where the group is small enough;
  * for MQA, whose single KV head gathers 64 query heads, the exact sums that hold at any
    size (Σ_j dK_j = 0, Σ_j dV_j = Σ dO over the group) instead of a full dK/dV.
"""
import numpy as np
import pytest
import torch

import oracle
from sdpa_workloads import (backward_d256, fp8_large_head, gpt2_inference, grouped, make_bias,
                            make_inputs, prefill_bottom_right, sample_kv_heads, sample_rows, training,
                            training_alibi, training_bias, training_dropout, training_fp8, training_varlen)
from sdpa_testlib import (FP8_REL_L2, FWD_MAX_ABS, GRAD_REL_L2, LSE_ABS, assert_fwd_close,
                          assert_grad_close, f64, guarded_empty_like, check_guard, rel_l2, run_bwd,
                          run_bwd_fp8, run_fwd)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N_ROWS = 64


def _rows_f64(t, bi, h, rows, descale=1.0):
    # CPU float8 tensors cannot be indexed with a list: go through their bytes
    if t.dtype == torch.float8_e4m3fn:
        return oracle.decode_e4m3(t.view(torch.uint8)[bi, h, rows].numpy(), descale)
    if t.dtype == torch.float8_e5m2:
        return oracle.decode_e5m2(t.view(torch.uint8)[bi, h, rows].numpy(), descale)
    return oracle.to_f64(t[bi, h, rows].cpu(), descale)


def _check_rows(w, x, o, lse, dq=None, descales=(1.0, 1.0, 1.0, 1.0), rel=None, bias_rows=None,
                grad_rel=None, zdrop_rows=None):
    """O, LSE (and dQ) of the sampled rows against the row forms.  bias_rows: optional
    function (bi, hq, rows) -> [len(rows), s_kv] fp64 additive term (ALiBi or a bias tensor);
    zdrop_rows: the same for the dropout factor keep / (1 - p).  rel / grad_rel: relative-L2
    bounds replacing the 16-bit ones (FP8)."""
    dsq, dsk, dsv, dsdo = descales
    by_head = {}
    for bi, h, r in sample_rows(w, N_ROWS):
        by_head.setdefault((bi, h), []).append(r)
    got_o, want_o, got_l, want_l, got_q, want_q = [], [], [], [], [], []
    for (bi, h), rows in by_head.items():
        rows = sorted(set(rows))
        hk = oracle.kv_head_of(h, w.h_q, w.h_kv)
        kh = _rows_f64(x.k, bi, hk, slice(None), dsk)
        vh = _rows_f64(x.v, bi, hk, slice(None), dsv)
        qr = _rows_f64(x.q, bi, h, rows, dsq)
        br = None if bias_rows is None else bias_rows(bi, h, rows)
        zr = None if zdrop_rows is None else zdrop_rows(bi, h, rows)
        O, L = oracle.forward_rows(qr, rows, kh, vh, w.scale, w.causal, br, zr)
        got_o.append(f64(o[bi, h, rows]))
        want_o.append(O)
        if lse is not None:
            got_l.append(lse[bi, h, rows].cpu().double().numpy())
            want_l.append(L)
        if dq is not None:
            dor = _rows_f64(x.do, bi, h, rows, dsdo)
            want_q.append(oracle.backward_dq_rows(qr, dor, rows, kh, vh, w.scale, w.causal, br, zr))
            got_q.append(f64(dq[bi, h, rows]))
    go, wo = np.concatenate(got_o), np.concatenate(want_o)
    if rel is None:
        assert_fwd_close(go, wo)
    else:
        assert rel_l2(go, wo) <= rel, f"O rel-L2 {rel_l2(go, wo):.3e}"
    if got_l:
        err = np.abs(np.concatenate(got_l) - np.concatenate(want_l)).max()
        assert err <= LSE_ABS, f"LSE max abs err {err:.3e}"
    if got_q:
        gq, wq = np.concatenate(got_q), np.concatenate(want_q)
        if grad_rel is None:
            assert_grad_close(gq, wq, "dQ rows")
        else:
            assert rel_l2(gq, wq) <= grad_rel, f"dQ rows rel-L2 {rel_l2(gq, wq):.3e}"


def _check_kv_heads(w, x, dk, dv, n_pairs, descales=(1.0, 1.0, 1.0, 1.0), kv_bias_rows=None, grad_rel=None,
                    kv_zdrop_rows=None):
    """Whole dK, dV of seeded (batch, KV head) pairs.  kv_bias_rows: optional function
    (bi, hq, r0, r1) -> fp64 additive term of query rows r0..r1-1; kv_zdrop_rows: the same for
    the dropout factor."""
    q64, k64, v64, do64 = (oracle.to_f64(t, ds) for t, ds in zip((x.q, x.k, x.v, x.do), descales))
    for bi, hk in sample_kv_heads(w, n_pairs)[:n_pairs]:
        fn = None if kv_bias_rows is None else (lambda hq, r0, r1, bi=bi: kv_bias_rows(bi, hq, r0, r1))
        zf = None if kv_zdrop_rows is None else (lambda hq, r0, r1, bi=bi: kv_zdrop_rows(bi, hq, r0, r1))
        gk, gv = oracle.backward_kv_head(q64, k64, v64, do64, w.scale, w.causal, bi, hk, bias_rows=fn,
                                         zdrop_rows=zf)
        for got, want, n in ((dk, gk, "dK"), (dv, gv, "dV")):
            if grad_rel is None:
                assert_grad_close(f64(got[bi, hk]), want, f"{n}[{bi},{hk}]")
            else:
                e = rel_l2(f64(got[bi, hk]), want)
                assert e <= grad_rel, f"{n}[{bi},{hk}] rel-L2 {e:.3e}"


def _full_case(w, dkv_pairs: int):
    x = make_inputs(w, seed=0, with_do=True)
    o, lse, dev = run_fwd(w, x)
    dq, dk, dv = run_bwd(w, dev, o, lse, x.do)
    _check_rows(w, x, o, lse, dq)
    if dkv_pairs:
        _check_kv_heads(w, x, dk, dv, dkv_pairs)
    return x, dq, dk, dv


@pytest.mark.parametrize("s", [512, 1024, 2048, 4096])
def test_training_sweep_lengths(s):
    """The rest of the training sweep (b2 h16 d128 bf16 causal), as the sweep launches it."""
    _full_case(training(s), dkv_pairs=2)


def test_training_s8192_as_benchmarked():
    _full_case(training(8192), dkv_pairs=2)


def test_training_s16384_rows():
    w = training(16384)
    x = make_inputs(w, seed=0, with_do=True)
    o, lse, dev = run_fwd(w, x)
    dq, _, _ = run_bwd(w, dev, o, lse, x.do)
    _check_rows(w, x, o, lse, dq)


def test_gqa_70b():
    _full_case(grouped(8), dkv_pairs=1)


def test_mha_70b():
    _full_case(grouped(64), dkv_pairs=1)


def test_mqa_70b_rows_and_exact_sums():
    w = grouped(1)
    x, dq, dk, dv = _full_case(w, dkv_pairs=0)
    sk = dk.double().sum(dim=2).cpu().numpy()
    scale_k = np.abs(dk.double().cpu().numpy()).sum(axis=2).max()
    assert np.abs(sk).max() <= 1e-2 * scale_k
    sv = dv.double().sum(dim=2).cpu().numpy()[0, 0]
    want = x.do.double().sum(dim=(1, 2)).numpy()[0]
    assert rel_l2(sv, want) <= GRAD_REL_L2


def test_gpt2_inference_full():
    w = gpt2_inference()
    x = make_inputs(w, seed=0, with_do=False)
    o, lse, _ = run_fwd(w, x, with_lse=False)
    O, _ = oracle.forward(f64(x.q), f64(x.k), f64(x.v), w.scale, w.causal)
    assert_fwd_close(f64(o), O)


def test_fp8_large_head_rows():
    w = fp8_large_head()
    x = make_inputs(w, seed=0, with_do=False)
    o, lse, _ = run_fwd(w, x)
    _check_rows(w, x, o, lse, None, (x.descale_q, x.descale_k, x.descale_v, 1.0), rel=FP8_REL_L2)


def test_training_varlen_as_benchmarked():
    """Eight padded sequences of 1K..8K tokens, causal, forward and backward as the sweep runs
    them.  Valid rows: O, LSE and dQ of sampled rows against the oracle on the batch's own
    length; dK/dV of one KV head of the two shortest batches in full.  Padded rows: O = 0 and
    LSE = -inf exactly, gradients vanish."""
    w = training_varlen()
    lens = list(w.lens_q)
    x = make_inputs(w, seed=0, with_do=True)
    o, lse, dev = run_fwd(w, x, seq_lens_q=lens, seq_lens_kv=lens)
    dq, dk, dv = run_bwd(w, dev, o, lse, x.do, seq_lens_q=lens, seq_lens_kv=lens)
    g = torch.Generator().manual_seed(7)
    by_head = {}
    for n in range(N_ROWS):
        bi = int(torch.randint(0, w.b, (1,), generator=g))
        h = int(torch.randint(0, w.h_q, (1,), generator=g))
        r = lens[bi] - 1 if n % 8 == 0 else int(torch.randint(0, lens[bi], (1,), generator=g))
        by_head.setdefault((bi, h), set()).add(r)
    got_o, want_o, got_l, want_l, got_q, want_q = [], [], [], [], [], []
    for (bi, h), rows in by_head.items():
        rows, L = sorted(rows), lens[bi]
        hk = oracle.kv_head_of(h, w.h_q, w.h_kv)
        kh, vh = _rows_f64(x.k, bi, hk, slice(0, L)), _rows_f64(x.v, bi, hk, slice(0, L))
        qr, dor = _rows_f64(x.q, bi, h, rows), _rows_f64(x.do, bi, h, rows)
        O, Lse = oracle.forward_rows(qr, rows, kh, vh, w.scale, True)
        got_o.append(f64(o[bi, h, rows])); want_o.append(O)
        got_l.append(lse[bi, h, rows].cpu().double().numpy()); want_l.append(Lse)
        want_q.append(oracle.backward_dq_rows(qr, dor, rows, kh, vh, w.scale, True))
        got_q.append(f64(dq[bi, h, rows]))
    assert_fwd_close(np.concatenate(got_o), np.concatenate(want_o))
    err = np.abs(np.concatenate(got_l) - np.concatenate(want_l)).max()
    assert err <= LSE_ABS, f"LSE max abs err {err:.3e}"
    assert_grad_close(np.concatenate(got_q), np.concatenate(want_q), "dQ rows")
    for bi in (w.b - 2, w.b - 1):
        L = lens[bi]
        sl = lambda t: oracle.to_f64(t[bi:bi + 1, :, :L])
        gk, gv = oracle.backward_kv_head(sl(x.q), sl(x.k), sl(x.v), sl(x.do), w.scale, True, 0, 3)
        assert_grad_close(f64(dk[bi, 3, :L]), gk, f"dK[{bi},3]")
        assert_grad_close(f64(dv[bi, 3, :L]), gv, f"dV[{bi},3]")
    for bi, L in enumerate(lens):
        if L == w.s_q:
            continue
        assert (o[bi, :, L:] == 0).all(), "padded rows of O must be zero"
        assert torch.isneginf(lse[bi, :, L:]).all(), "padded rows of LSE must be -inf"
        for t, name in ((dq, "dQ"), (dk, "dK"), (dv, "dV")):
            pad = t[bi, :, L:].abs().max().item()
            ref = t[bi, :, :L].abs().max().item()
            assert pad <= 1e-3 * ref, f"padded rows of {name}: {pad} (valid max {ref})"


def test_prefill_bottom_right_rows():
    """A 2K-token chunk against an 8K context, bottom-right causal (GQA 32/8), as the sweep
    runs it: query row r sees keys j <= r + (s_kv - s_q), i.e. top-left rows shifted by 6144."""
    w = prefill_bottom_right()
    x = make_inputs(w, seed=0, with_do=False)
    o, lse, _ = run_fwd(w, x, causal="bottom_right")
    off = w.s_kv - w.s_q
    by_head = {}
    for bi, h, r in sample_rows(w, N_ROWS):
        by_head.setdefault((bi, h), set()).add(r)
    got_o, want_o, got_l, want_l = [], [], [], []
    for (bi, h), rows in by_head.items():
        rows = sorted(rows)
        hk = oracle.kv_head_of(h, w.h_q, w.h_kv)
        kh, vh = _rows_f64(x.k, bi, hk, slice(None)), _rows_f64(x.v, bi, hk, slice(None))
        O, Lse = oracle.forward_rows(_rows_f64(x.q, bi, h, rows), [r + off for r in rows], kh, vh,
                                     w.scale, True)
        got_o.append(f64(o[bi, h, rows])); want_o.append(O)
        got_l.append(lse[bi, h, rows].cpu().double().numpy()); want_l.append(Lse)
    assert_fwd_close(np.concatenate(got_o), np.concatenate(want_o))
    err = np.abs(np.concatenate(got_l) - np.concatenate(want_l)).max()
    assert err <= LSE_ABS, f"LSE max abs err {err:.3e}"


def test_training_alibi_s8192_as_benchmarked():
    """The training step with ALiBi (default slopes), as the sweep runs it: its key blocks are
    visited from the diagonal outward, a schedule only long rows exercise."""
    w = training_alibi(8192)
    x = make_inputs(w, seed=0, with_do=True)
    o, lse, dev = run_fwd(w, x, alibi="default")
    dq, dk, dv = run_bwd(w, dev, o, lse, x.do, alibi="default")
    slopes = oracle.alibi_default_slopes(w.h_q)
    rows_fn = lambda bi, hq, rows: oracle.alibi_bias(w.s_q, w.s_kv, slopes[hq], 0, rows=rows)
    _check_rows(w, x, o, lse, dq, bias_rows=rows_fn)
    _check_kv_heads(w, x, dk, dv, 2,
                    kv_bias_rows=lambda bi, hq, r0, r1: rows_fn(bi, hq, np.arange(r0, r1)))


def test_training_bias_s8192_as_benchmarked():
    """The training step with a [1, 16, 8192, 8192] bf16 bias and its gradient, as the sweep runs
    it: sampled rows of O, LSE, dQ and of dbias (dS summed over the batch), and two whole KV
    heads of dK, dV."""
    w = training_bias(8192)
    x = make_inputs(w, seed=0, with_do=True)
    bias_cpu = make_bias(w)
    bias = bias_cpu.cuda()
    dbias, dbuf = guarded_empty_like(bias)
    o, lse, dev = run_fwd(w, x, bias=bias)
    dq, dk, dv = run_bwd(w, dev, o, lse, x.do, bias=bias, dbias=dbias)
    check_guard(dbuf, "dbias")
    rows_fn = lambda bi, hq, rows: oracle.to_f64(bias_cpu[0, hq, rows])
    _check_rows(w, x, o, lse, dq, bias_rows=rows_fn)
    # dbias rows: the sum over the batch of each sampled row's dS
    by_head = {}
    for _, h, r in sample_rows(w, 16, seed=5):
        by_head.setdefault(h, set()).add(r)
    got, want = [], []
    for h, rows in by_head.items():
        rows = sorted(rows)
        acc = np.zeros((len(rows), w.s_kv))
        for bi in range(w.b):
            hk = oracle.kv_head_of(h, w.h_q, w.h_kv)
            acc += oracle.backward_ds_rows(_rows_f64(x.q, bi, h, rows), _rows_f64(x.do, bi, h, rows), rows,
                                           _rows_f64(x.k, bi, hk, slice(None)), _rows_f64(x.v, bi, hk, slice(None)),
                                           w.scale, True, rows_fn(bi, h, rows))
        want.append(acc)
        got.append(f64(dbias[0, h, rows]))
    assert_grad_close(np.concatenate(got), np.concatenate(want), "dbias rows")
    _check_kv_heads(w, x, dk, dv, 2, kv_bias_rows=lambda bi, hq, r0, r1: oracle.to_f64(bias_cpu[0, hq, r0:r1]))


def test_training_dropout_s8192_as_benchmarked():
    """The training step with dropout p = 0.1, as the sweep runs it: the library draws the keep
    mask (seed 1234, offset 0; both layouts, tiles above the diagonal skipped), the kernels read
    it, and the oracle draws its own keep bits for the rows it checks (O, LSE, dQ of sampled rows;
    two whole KV heads of dK, dV)."""
    w = training_dropout(8192)
    drop = (w.dropout, 1234, 0)
    x = make_inputs(w, seed=0, with_do=True)
    o, lse, dev = run_fwd(w, x, dropout=drop)
    dq, dk, dv = run_bwd(w, dev, o, lse, x.do, dropout=drop)
    zf = lambda bi, hq, r0, r1: oracle.dropout_keep_range(w.b, w.h_q, w.s_q, w.s_kv, drop[0], drop[1], drop[2],
                                                           bi * w.h_q + hq, r0, r1) / (1.0 - drop[0])
    rows_fn = lambda bi, hq, rows: np.concatenate([zf(bi, hq, r, r + 1) for r in rows])
    _check_rows(w, x, o, lse, dq, zdrop_rows=rows_fn)
    _check_kv_heads(w, x, dk, dv, 2, kv_zdrop_rows=zf)


def test_training_fp8_s8192_as_benchmarked():
    """The FP8 training step (E4M3 Q, K, V with a bf16 O; E5M2 dO; bf16 gradients) as the sweep
    runs it, against the oracle on the decoded inputs.  The forward's E4M3 rounding of P enters
    O and, through Delta = rowsum(dO∘O), the gradients: FP8 tolerances throughout, except the
    LSE, which the kernel sums from unrounded P."""
    w = training_fp8(8192)
    x = make_inputs(w, seed=0, with_do=True)
    o, lse, _ = run_fwd(w, x)
    dq, dk, dv = run_bwd_fp8(w, x, o, lse)
    ds = (x.descale_q, x.descale_k, x.descale_v, x.descale_do)
    _check_rows(w, x, o, lse, dq, descales=ds, rel=FP8_REL_L2, grad_rel=FP8_REL_L2)
    _check_kv_heads(w, x, dk, dv, 2, descales=ds, grad_rel=FP8_REL_L2)


@pytest.mark.parametrize("causal", [True, False])
def test_backward_d256_as_benchmarked(causal):
    """The d = 256 backward pass at b4 h16 s4096 (bf16, causal and without a mask): sampled rows
    and two whole KV heads."""
    _full_case(backward_d256(causal), dkv_pairs=2)
