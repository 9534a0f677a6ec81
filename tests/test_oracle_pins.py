"""Pins for the fp64 oracle: checks it against things other than itself.

Brute force written as explicit Python loops, hand-worked values (tests/golden),
closed forms, invariants the definition implies, and central finite differences
for the backward pass.  Each test is chosen so that a plausible slip in the oracle
(a dropped scale, a transposed operand, a wrong head index, a mask off by one, a
missing Delta term) fails at least one of them.
"""
import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from sdpa_workloads import Workload, make_inputs, gpt2_inference, quantize_e4m3, quantize_e5m2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(12345)


def _rand(*shape):
    return RNG.standard_normal(shape)


# ---------------------------------------------------------------------------
# brute force: explicit loops straight from the definition
# ---------------------------------------------------------------------------

def _brute_forward(q, k, v, scale, causal):
    b, h_q, s_q, d = q.shape
    h_kv, s_kv, dv = k.shape[1], k.shape[2], v.shape[3]
    g = h_q // h_kv
    O = np.zeros((b, h_q, s_q, dv))
    L = np.zeros((b, h_q, s_q))
    for bi in range(b):
        for h in range(h_q):
            hk = h // g
            for i in range(s_q):
                w = []
                for j in range(s_kv):
                    if causal and j > i:
                        w.append(0.0)
                        continue
                    dot = 0.0
                    for t in range(d):
                        dot += q[bi, h, i, t] * k[bi, hk, j, t]
                    w.append(math.exp(scale * dot))
                tot = sum(w)
                L[bi, h, i] = math.log(tot)
                for c in range(dv):
                    O[bi, h, i, c] = sum(w[j] / tot * v[bi, hk, j, c] for j in range(s_kv))
    return O, L


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("h_q,h_kv", [(2, 2), (4, 2), (3, 1)])
def test_forward_matches_brute_force(causal, h_q, h_kv):
    q, k, v = _rand(2, h_q, 5, 3), _rand(2, h_kv, 7, 3), _rand(2, h_kv, 7, 3)
    O, L = oracle.forward(q, k, v, 0.7, causal)
    Ob, Lb = _brute_forward(q, k, v, 0.7, causal)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_rows_matches_brute_force(causal):
    q, k, v = _rand(1, 2, 9, 4), _rand(1, 1, 9, 4), _rand(1, 1, 9, 4)
    Ob, Lb = _brute_forward(q, k, v, 0.5, causal)
    rows = [0, 3, 8]
    O, L = oracle.forward_rows(q[0, 1, rows], rows, k[0, 0], v[0, 0], 0.5, causal)
    np.testing.assert_allclose(O, Ob[0, 1, rows], atol=1e-12)
    np.testing.assert_allclose(L, Lb[0, 1, rows], atol=1e-12)


# ---------------------------------------------------------------------------
# hand-worked example (tests/golden/hand_worked_2x2.json)
# ---------------------------------------------------------------------------

def _num(x):
    env = {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4)}
    return float(eval(str(x), {"__builtins__": {}}, env))


def test_hand_worked_example():
    gold = json.load(open(os.path.join(GOLDEN, "hand_worked_2x2.json")))
    q = np.array([[_num(x) for x in r] for r in gold["q"]])[None, None]
    k = np.array(gold["k"], dtype=float)[None, None]
    v = np.array(gold["v"], dtype=float)[None, None]
    for case, causal in (("full", False), ("causal", True)):
        O, L = oracle.forward(q, k, v, 1.0, causal)
        np.testing.assert_allclose(O[0, 0], np.array(gold[case]["o"]), atol=1e-14)
        np.testing.assert_allclose(L[0, 0], [_num(x) for x in gold[case]["lse"]], atol=1e-14)
    do = np.array(gold["backward_dO"], dtype=float)[None, None]
    dQ, dK, dV = oracle.backward(q, k, v, do, 1.0, False)
    fb = gold["full_backward"]
    for name, got in (("dq", dQ), ("dk", dK), ("dv", dV)):
        want = np.array([[_num(x) for x in r] for r in fb[name]])
        np.testing.assert_allclose(got[0, 0], want, atol=1e-14, err_msg=name)


# ---------------------------------------------------------------------------
# softmax and forward invariants / closed forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_sum_to_one_and_mask_is_exact(causal):
    q, k, v = _rand(6, 8), _rand(10, 8), _rand(10, 8)
    mask = oracle.visible_mask(6, 10, causal)
    _, _, P = oracle.head_forward(q, k, v, 0.35, mask)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)
    assert (P >= 0).all()
    assert (P[~mask] == 0).all()
    if causal:
        assert mask.sum() == sum(min(i + 1, 10) for i in range(6))


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_returns_v(causal):
    q, k = _rand(1, 2, 7, 5), _rand(1, 2, 7, 5)
    c = _rand(5)
    v = np.broadcast_to(c, (1, 2, 7, 5)).copy()
    O, _ = oracle.forward(q, k, v, 1.3, causal)
    np.testing.assert_allclose(O, np.broadcast_to(c, O.shape), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_gives_mean_of_visible_values(causal):
    q, k, v = _rand(1, 1, 6, 3), _rand(1, 1, 6, 3), _rand(1, 1, 6, 3)
    O, L = oracle.forward(q, k, v, 0.0, causal)
    for i in range(6):
        n = i + 1 if causal else 6
        np.testing.assert_allclose(O[0, 0, i], v[0, 0, :n].mean(axis=0), atol=1e-12)
        np.testing.assert_allclose(L[0, 0, i], math.log(n), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_lse_is_log_count(causal):
    q = np.zeros((1, 1, 5, 4))
    k, v = _rand(1, 1, 8, 4), _rand(1, 1, 8, 4)
    _, L = oracle.forward(q, k, v, 0.9, causal)
    want = [math.log(min(i + 1, 8) if causal else 8) for i in range(5)]
    np.testing.assert_allclose(L[0, 0], want, atol=1e-12)


def test_causal_first_and_last_rows():
    """Row 0 attends only to key 0; the last row sees every key (codelab §7)."""
    q, k, v = _rand(1, 2, 9, 4), _rand(1, 2, 9, 4), _rand(1, 2, 9, 4)
    Oc, Lc = oracle.forward(q, k, v, 0.6, True)
    Of, Lf = oracle.forward(q, k, v, 0.6, False)
    np.testing.assert_allclose(Oc[:, :, 0], v[:, :, 0], atol=1e-12)
    np.testing.assert_allclose(Lc[:, :, 0], 0.6 * (q[:, :, 0] * k[:, :, 0]).sum(-1), atol=1e-12)
    np.testing.assert_allclose(Oc[:, :, -1], Of[:, :, -1], atol=1e-12)
    assert np.abs(Oc[:, :, 0] - Of[:, :, 0]).max() > 1e-3
    gold = json.load(open(os.path.join(GOLDEN, "page_shapes.json")))["codelab_causal_effect"]
    assert np.abs(Oc[:, :, -1] - Of[:, :, -1]).max() < gold["last_position_max_abs_diff_below"]


def test_causal_row_ignores_future_keys():
    q, k, v = _rand(1, 1, 8, 4), _rand(1, 1, 8, 4), _rand(1, 1, 8, 4)
    O1, L1 = oracle.forward(q, k, v, 0.8, True)
    k2, v2 = k.copy(), v.copy()
    i = 3
    k2[:, :, i + 1:] += 5 * _rand(1, 1, 8 - i - 1, 4)
    v2[:, :, i + 1:] -= 7.0
    O2, L2 = oracle.forward(q, k2, v2, 0.8, True)
    np.testing.assert_array_equal(O1[:, :, : i + 1], O2[:, :, : i + 1])
    np.testing.assert_array_equal(L1[:, :, : i + 1], L2[:, :, : i + 1])
    assert np.abs(O1[:, :, i + 1:] - O2[:, :, i + 1:]).max() > 1e-3


def test_two_key_closed_form():
    """With two keys, softmax is a logistic function of the score difference."""
    q, k, v = _rand(1, 1, 4, 6), _rand(1, 1, 2, 6), _rand(1, 1, 2, 6)
    O, L = oracle.forward(q, k, v, 0.4, False)
    s = 0.4 * q[0, 0] @ k[0, 0].T
    p0 = 1.0 / (1.0 + np.exp(s[:, 1] - s[:, 0]))
    np.testing.assert_allclose(O[0, 0], p0[:, None] * v[0, 0, 0] + (1 - p0)[:, None] * v[0, 0, 1],
                               atol=1e-12)
    np.testing.assert_allclose(L[0, 0], np.logaddexp(s[:, 0], s[:, 1]), atol=1e-12)


@pytest.mark.parametrize("h_kv", [1, 2, 4])
def test_grouped_heads_equal_repeated_mha(h_kv):
    """GQA/MQA equal MHA with each KV head repeated over its group (codelab §9)."""
    h_q = 4
    q, k, v = _rand(2, h_q, 6, 3), _rand(2, h_kv, 6, 3), _rand(2, h_kv, 6, 3)
    do = _rand(2, h_q, 6, 3)
    g = h_q // h_kv
    kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    for causal in (False, True):
        O, L = oracle.forward(q, k, v, 0.5, causal)
        Or, Lr = oracle.forward(q, kr, vr, 0.5, causal)
        np.testing.assert_allclose(O, Or, atol=1e-13)
        np.testing.assert_allclose(L, Lr, atol=1e-13)
        dQ, dK, dV = oracle.backward(q, k, v, do, 0.5, causal)
        dQr, dKr, dVr = oracle.backward(q, kr, vr, do, 0.5, causal)
        np.testing.assert_allclose(dQ, dQr, atol=1e-13)
        np.testing.assert_allclose(dK, dKr.reshape(2, h_kv, g, 6, 3).sum(2), atol=1e-13)
        np.testing.assert_allclose(dV, dVr.reshape(2, h_kv, g, 6, 3).sum(2), atol=1e-13)


def test_head_grouping_shapes_from_codelab():
    gold = json.load(open(os.path.join(GOLDEN, "page_shapes.json")))["codelab_head_grouping"]
    B, T, N, H = gold["q_btnh"]
    q = _rand(B, T, N, H).transpose(0, 2, 1, 3)
    for _, nk in gold["kv_heads"].items():
        k = _rand(B, T, nk, H).transpose(0, 2, 1, 3)
        O, _ = oracle.forward(q, k, k, 1 / 8, False)
        assert list(O.transpose(0, 2, 1, 3).shape) == gold["out_btnh"]
    with pytest.raises(ValueError):
        oracle.kv_head_of(0, 8, 3)


def test_bshd_view_equals_bhsd_in_the_oracle():
    """The layout is a view: BSHD-strided logical tensors give the same result."""
    w = Workload("t", 1, 2, 2, 16, 16, 8, "f16", layout="bshd", causal=True)
    x = make_inputs(w, seed=3, with_do=False)
    wc = Workload("t", 1, 2, 2, 16, 16, 8, "f16", layout="bhsd", causal=True)
    q = oracle.to_f64(x.q.contiguous())
    qs = oracle.to_f64(x.q)
    np.testing.assert_array_equal(q, qs)
    assert x.q.stride() == (16 * 2 * 8, 8, 2 * 8, 1)
    O1, _ = oracle.forward(qs, oracle.to_f64(x.k), oracle.to_f64(x.v), w.scale, True)
    O2, _ = oracle.forward(q, oracle.to_f64(x.k.contiguous()), oracle.to_f64(x.v.contiguous()),
                           wc.scale, True)
    np.testing.assert_array_equal(O1, O2)


def test_gpt2_workload_matches_page():
    gold = json.load(open(os.path.join(GOLDEN, "page_shapes.json")))["gpt2_like"]
    w = gpt2_inference()
    assert (w.b, w.h_q, w.s_q, w.d) == (gold["b"], gold["h"], gold["s"], gold["d"])
    assert w.causal == gold["causal"] and w.stats == gold["stats"] and w.dtype == gold["dtype"]
    x = make_inputs(Workload("g", 4, 12, 12, 1024, 1024, 64, "f16", layout="bshd"), with_do=False)
    assert list(x.q.stride()) == gold["strides"]
    assert abs(w.scale - 1 / math.sqrt(64)) < 1e-15


# ---------------------------------------------------------------------------
# backward: central finite differences and invariants
# ---------------------------------------------------------------------------

def _fd_grads(q, k, v, do, scale, causal, h=1e-6):
    def loss(q_, k_, v_):
        O, _ = oracle.forward(q_, k_, v_, scale, causal)
        return float((O * do).sum())
    grads = []
    for which in range(3):
        args = [q.copy(), k.copy(), v.copy()]
        x = args[which]
        gx = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = loss(*args)
            x[idx] = old - h
            lm = loss(*args)
            x[idx] = old
            gx[idx] = (lp - lm) / (2 * h)
        grads.append(gx)
    return grads


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("h_q,h_kv,s_q,s_kv", [(2, 2, 4, 4), (4, 2, 5, 3), (2, 1, 3, 6)])
def test_backward_matches_finite_differences(causal, h_q, h_kv, s_q, s_kv):
    if causal and s_kv < 1:
        pytest.skip()
    q, k, v, do = _rand(1, h_q, s_q, 3), _rand(1, h_kv, s_kv, 3), _rand(1, h_kv, s_kv, 3), \
        _rand(1, h_q, s_q, 3)
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.45, causal)
    fQ, fK, fV = _fd_grads(q, k, v, do, 0.45, causal)
    for got, want, name in ((dQ, fQ, "dQ"), (dK, fK, "dK"), (dV, fV, "dV")):
        err = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
        assert err < 1e-6, (name, err)
    # the sampled forms agree with the same finite differences
    rows = list(range(s_q))
    for hq in range(h_q):
        hk = oracle.kv_head_of(hq, h_q, h_kv)
        g = oracle.backward_dq_rows(q[0, hq], do[0, hq], rows, k[0, hk], v[0, hk], 0.45, causal)
        assert np.linalg.norm(g - fQ[0, hq]) / np.linalg.norm(fQ[0, hq]) < 1e-6
    for hk in range(h_kv):
        gk, gv = oracle.backward_kv_head(q, k, v, do, 0.45, causal, 0, hk, row_chunk=2)
        assert np.linalg.norm(gk - fK[0, hk]) / max(np.linalg.norm(fK[0, hk]), 1e-30) < 1e-6
        assert np.linalg.norm(gv - fV[0, hk]) / max(np.linalg.norm(fV[0, hk]), 1e-30) < 1e-6


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(causal):
    h_q, h_kv = 4, 2
    q, k, v, do = _rand(2, h_q, 7, 5), _rand(2, h_kv, 7, 5), _rand(2, h_kv, 7, 5), \
        _rand(2, h_q, 7, 5)
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.3, causal)
    # each row of dS sums to zero, so the keys' gradients sum to zero per KV head
    np.testing.assert_allclose(dK.sum(axis=2), 0.0, atol=1e-12)
    # each row of P sums to one, so Σ_j dV_j = Σ over the group's rows of dO
    np.testing.assert_allclose(dV.sum(axis=2),
                               do.reshape(2, h_kv, 2, 7, 5).sum(axis=(2, 3)), atol=1e-12)
    # identical keys make P independent of Q, so dQ vanishes
    kc = np.broadcast_to(k[:, :, :1], k.shape).copy()
    dQc, _, _ = oracle.backward(q, kc, v, do, 0.3, causal)
    np.testing.assert_allclose(dQc, 0.0, atol=1e-12)


# ---------------------------------------------------------------------------
# E4M3
# ---------------------------------------------------------------------------

def test_e4m3_table_matches_torch_cast_for_all_codes():
    tab = oracle.e4m3_decode_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    np.testing.assert_array_equal(np.isnan(tab), nan)
    np.testing.assert_array_equal(tab[~nan], ref[~nan])


def test_e4m3_special_values():
    tab = oracle.e4m3_decode_table()
    assert tab[0x7E] == 448.0 and tab[0xFE] == -448.0
    assert tab[0x01] == 2.0 ** -9 and tab[0x08] == 2.0 ** -6 and tab[0x38] == 1.0
    assert tab[0x80] == 0.0 and math.copysign(1, tab[0x80]) == -1.0


def test_e4m3_quantisation_round_trip_within_half_ulp():
    x = torch.randn(4096, generator=torch.Generator().manual_seed(0))
    q8, descale = quantize_e4m3(x)
    y = oracle.to_f64(q8, descale)
    scale = 1.0 / descale
    xs = x.double().numpy() * scale
    ys = y * scale
    # spacing of E4M3 near |x|: 2**(floor(log2|x|) - 3) for normals, 2**-9 below 2**-6
    e = np.floor(np.log2(np.maximum(np.abs(xs), 2.0 ** -6)))
    ulp = 2.0 ** (e - 3)
    assert (np.abs(ys - xs) <= ulp / 2 + 1e-12).all()
    assert np.abs(oracle.to_f64(q8)).max() <= 448.0


# ---------------------------------------------------------------------------
# E5M2 (gradient format)
# ---------------------------------------------------------------------------

def test_e5m2_table_matches_torch_cast_for_all_codes():
    tab = oracle.e5m2_decode_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]
    np.testing.assert_array_equal(np.isnan(tab), nan)
    np.testing.assert_array_equal(tab[~nan], ref[~nan])


def test_e5m2_special_values():
    tab = oracle.e5m2_decode_table()
    assert tab[0x7B] == 57344.0 and tab[0x7C] == math.inf and tab[0xFC] == -math.inf
    assert tab[0x01] == 2.0 ** -16 and tab[0x04] == 2.0 ** -14 and tab[0x3C] == 1.0


def test_e5m2_quantisation_round_trip_within_half_ulp():
    x = torch.randn(4096, generator=torch.Generator().manual_seed(1))
    q8, descale = quantize_e5m2(x)
    y = oracle.to_f64(q8, descale)
    scale = 1.0 / descale
    xs = x.double().numpy() * scale
    ys = y * scale
    # spacing of E5M2 near |x|: 2**(floor(log2|x|) - 2) for normals, 2**-16 below 2**-14
    e = np.floor(np.log2(np.maximum(np.abs(xs), 2.0 ** -14)))
    ulp = 2.0 ** (e - 2)
    assert (np.abs(ys - xs) <= ulp / 2 + 1e-12).all()
    assert np.abs(oracle.to_f64(q8)).max() <= 57344.0


# ---------------------------------------------------------------------------
# variable lengths and bottom-right causal alignment
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal,bottom_right", [(False, False), (True, False), (True, True)])
def test_varlen_equals_unpadded_problem(causal, bottom_right):
    """Padding changes nothing: each batch equals the problem cut to its own lengths, and
    padded rows are zero (O, dQ, dK, dV) with LSE = -inf."""
    b, h_q, h_kv, s_q, s_kv, d = 3, 4, 2, 9, 11, 3
    q, k, v, do = _rand(b, h_q, s_q, d), _rand(b, h_kv, s_kv, d), _rand(b, h_kv, s_kv, d), \
        _rand(b, h_q, s_q, d)
    lq, lkv = [9, 5, 7], [11, 6, 3]
    O, L = oracle.forward(q, k, v, 0.6, causal, lq, lkv, bottom_right)
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.6, causal, lq, lkv, bottom_right)
    for bi in range(b):
        a, c = lq[bi], lkv[bi]
        sl = lambda t, n: t[bi:bi + 1, :, :n]
        if bottom_right and causal and c < a:
            # rows with no visible key: exactly the first a - c rows
            n0 = a - c
            assert (L[bi, :, :n0] == -np.inf).all() and (O[bi, :, :n0] == 0).all()
            Ou, Lu = oracle.forward(q[bi:bi + 1, :, n0:a], sl(k, c), sl(v, c), 0.6, True)
            np.testing.assert_allclose(O[bi:bi + 1, :, n0:a], Ou, atol=1e-13)
            np.testing.assert_allclose(L[bi:bi + 1, :, n0:a], Lu, atol=1e-13)
        else:
            shifted = bottom_right and causal and c > a
            if shifted:
                # bottom-right with more keys than queries: row i sees keys j <= i + (c - a)
                Ou, Lu = oracle.forward(sl(q, a), sl(k, c), sl(v, c), 0.6, True, [a], [c], True)
            else:
                Ou, Lu = oracle.forward(sl(q, a), sl(k, c), sl(v, c), 0.6, causal)
            np.testing.assert_allclose(O[bi:bi + 1, :, :a], Ou, atol=1e-13)
            np.testing.assert_allclose(L[bi:bi + 1, :, :a], Lu, atol=1e-13)
        assert (O[bi, :, a:] == 0).all() and (L[bi, :, a:] == -np.inf).all()
        assert (dQ[bi, :, a:] == 0).all() and (dK[bi, :, c:] == 0).all() and (dV[bi, :, c:] == 0).all()
        if not (bottom_right and causal):
            gq, gk, gv = oracle.backward(sl(q, a), sl(k, c), sl(v, c), sl(do, a), 0.6, causal)
            np.testing.assert_allclose(dQ[bi:bi + 1, :, :a], gq, atol=1e-12)
            np.testing.assert_allclose(dK[bi:bi + 1, :, :c], gk, atol=1e-12)
            np.testing.assert_allclose(dV[bi:bi + 1, :, :c], gv, atol=1e-12)


def test_bottom_right_closed_forms():
    """Equal lengths: bottom-right = top-left.  One query row (a decoding step): it sees
    every key, so it equals the unmasked row.  Brute force on a ragged case."""
    q, k, v = _rand(1, 2, 6, 4), _rand(1, 2, 6, 4), _rand(1, 2, 6, 4)
    O1, L1 = oracle.forward(q, k, v, 0.5, True, [6], [6], True)
    O2, L2 = oracle.forward(q, k, v, 0.5, True)
    np.testing.assert_allclose(O1, O2, atol=1e-14)
    q1, k9, v9 = _rand(1, 1, 1, 4), _rand(1, 1, 9, 4), _rand(1, 1, 9, 4)
    Od, Ld = oracle.forward(q1, k9, v9, 0.5, True, [1], [9], True)
    Of, Lf = oracle.forward(q1, k9, v9, 0.5, False)
    np.testing.assert_allclose(Od, Of, atol=1e-14)
    np.testing.assert_allclose(Ld, Lf, atol=1e-14)
    # brute force: 4 queries, 7 keys, bottom-right: row i sees keys j <= i + 3
    q4, k7, v7 = _rand(1, 1, 4, 3), _rand(1, 1, 7, 3), _rand(1, 1, 7, 3)
    O, L = oracle.forward(q4, k7, v7, 0.9, True, [4], [7], True)
    for i in range(4):
        w = [math.exp(0.9 * float(q4[0, 0, i] @ k7[0, 0, jj])) for jj in range(i + 4)]
        tot = sum(w)
        np.testing.assert_allclose(O[0, 0, i], sum(w[jj] / tot * v7[0, 0, jj] for jj in range(i + 4)),
                                   atol=1e-12)
        np.testing.assert_allclose(L[0, 0, i], math.log(tot), atol=1e-12)


def test_varlen_backward_matches_finite_differences():
    q, k, v, do = _rand(2, 2, 5, 3), _rand(2, 2, 6, 3), _rand(2, 2, 6, 3), _rand(2, 2, 5, 3)
    lq, lkv = [5, 3], [4, 6]
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.7, True, lq, lkv, True)

    def loss(q_, k_, v_):
        O, _ = oracle.forward(q_, k_, v_, 0.7, True, lq, lkv, True)
        return float((O * do).sum())
    for which, got in ((0, dQ), (1, dK), (2, dV)):
        args = [q.copy(), k.copy(), v.copy()]
        x = args[which]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + 1e-6
            lp = loss(*args)
            x[idx] = old - 1e-6
            lm = loss(*args)
            x[idx] = old
            fd[idx] = (lp - lm) / 2e-6
        assert np.linalg.norm(got - fd) / np.linalg.norm(fd) < 1e-6


# ---------------------------------------------------------------------------
# ALiBi
# ---------------------------------------------------------------------------

def test_alibi_brute_force_and_limits():
    """Brute force with explicit loops; zero slopes change nothing; a huge slope makes a
    causal row attend only to its own key (every earlier key is penalised away)."""
    q, k, v = _rand(1, 2, 5, 3), _rand(1, 2, 7, 3), _rand(1, 2, 7, 3)
    slopes = [0.25, 1.5]
    for causal in (True,):
        O, L = oracle.forward(q, k, v, 0.8, causal, alibi_slopes=slopes)
        for h in range(2):
            for i in range(5):
                w = [0.0 if (causal and j > i) else
                     math.exp(0.8 * float(q[0, h, i] @ k[0, h, j]) - slopes[h] * (i - j)) for j in range(7)]
                tot = sum(w)
                np.testing.assert_allclose(O[0, h, i], sum(w[j] / tot * v[0, h, j] for j in range(7)), atol=1e-12)
                np.testing.assert_allclose(L[0, h, i], math.log(tot), atol=1e-12)
    O0, _ = oracle.forward(q, k, v, 0.8, True, alibi_slopes=[0.0, 0.0])
    Oc, _ = oracle.forward(q, k, v, 0.8, True)
    np.testing.assert_allclose(O0, Oc, atol=1e-14)
    Oh, _ = oracle.forward(q, k, v, 0.8, True, alibi_slopes=[200.0, 200.0])
    np.testing.assert_allclose(Oh[0, :, :5], v[0, :, :5], atol=1e-12)


def test_alibi_needs_a_causal_mask():
    """ALiBi penalises the distance to earlier keys (the ALiBi paper, §3); with no causal mask
    there would be later keys, which the linear term rewards: the oracle refuses that case."""
    q, k, v, do = _rand(1, 1, 4, 2), _rand(1, 1, 4, 2), _rand(1, 1, 4, 2), _rand(1, 1, 4, 2)
    with pytest.raises(ValueError):
        oracle.forward(q, k, v, 0.5, False, alibi_slopes=[0.3])
    with pytest.raises(ValueError):
        oracle.backward(q, k, v, do, 0.5, False, alibi_slopes=[0.3])


@pytest.mark.parametrize("bottom_right,s_q,s_kv", [(False, 9, 9), (False, 5, 12), (True, 5, 12), (True, 12, 5)])
def test_alibi_weights_fall_geometrically_with_distance(bottom_right, s_q, s_kv):
    """With Q = 0 every score is 0, so the weights are the softmax of the ALiBi term alone: a
    penalty m per key of distance from the aligned diagonal.  Row i's visible keys j = i + off,
    i + off - 1, ..., 0 then get the truncated geometric weights r^t (1 - r) / (1 - r^n) with
    r = e^-m, t the distance and n the number of visible keys, largest on the diagonal and never
    rising with distance; V = I reads the weights out of O."""
    m = 0.4
    q = np.zeros((1, 1, s_q, 2))
    k = _rand(1, 1, s_kv, 2)
    v = np.eye(s_kv)[None, None]
    O, L = oracle.forward(q, k, v, 0.7, True, None, None, bottom_right, alibi_slopes=[m])
    off = (s_kv - s_q) if bottom_right else 0
    r = math.exp(-m)
    for i in range(s_q):
        last = min(i + off, s_kv - 1)
        if last < 0:
            assert np.isneginf(L[0, 0, i]) and not O[0, 0, i].any()
            continue
        n = last + 1
        want = np.zeros(s_kv)
        for j in range(n):
            t = i + off - j
            want[j] = r ** (t - (i + off - last)) * (1 - r) / (1 - r ** n)
        np.testing.assert_allclose(O[0, 0, i], want, atol=1e-13)
        w = O[0, 0, i, :n]
        assert np.all(np.diff(w) >= 0), "weights must not rise with distance from the diagonal"


def test_alibi_bottom_right_offset_and_gradients():
    """Bottom-right: the bias is zero on the aligned diagonal (j = i + off).  Backward with
    ALiBi against finite differences (the bias has no gradient)."""
    q, k, v, do = _rand(1, 1, 3, 2), _rand(1, 1, 6, 2), _rand(1, 1, 6, 2), _rand(1, 1, 3, 2)
    O, L = oracle.forward(q, k, v, 0.5, True, None, None, True, alibi_slopes=[0.7])
    for i in range(3):
        w = [math.exp(0.5 * float(q[0, 0, i] @ k[0, 0, j]) + 0.7 * (j - i - 3)) for j in range(i + 4)]
        np.testing.assert_allclose(L[0, 0, i], math.log(sum(w)), atol=1e-12)
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.5, True, None, None, True, alibi_slopes=[0.7])

    def loss(q_, k_, v_):
        Ox, _ = oracle.forward(q_, k_, v_, 0.5, True, None, None, True, alibi_slopes=[0.7])
        return float((Ox * do).sum())
    for which, got in ((0, dQ), (1, dK), (2, dV)):
        args = [q.copy(), k.copy(), v.copy()]
        x = args[which]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + 1e-6
            lp = loss(*args)
            x[idx] = old - 1e-6
            lm = loss(*args)
            x[idx] = old
            fd[idx] = (lp - lm) / 2e-6
        assert np.linalg.norm(got - fd) / np.linalg.norm(fd) < 1e-6


def test_alibi_default_slopes_match_the_alibi_paper():
    """Press, Smith and Lewis, "Train Short, Test Long", §3: with 8 heads the slopes are
    1/2, 1/4, ..., 1/256; with 16 heads they start at 2^-0.5 and halve every two heads."""
    np.testing.assert_array_equal(oracle.alibi_default_slopes(8), [1 / 2 ** k for k in range(1, 9)])
    s16 = oracle.alibi_default_slopes(16)
    np.testing.assert_allclose(s16[0], 2 ** -0.5, rtol=1e-15)
    np.testing.assert_allclose(s16[1::2], [1 / 2 ** k for k in range(1, 9)], rtol=1e-15)
    np.testing.assert_allclose(s16[1:] / s16[:-1], 2 ** -0.5, rtol=1e-14)


# ---------------------------------------------------------------------------
# Dropout: Philox4x32-10 and the keep mask
# ---------------------------------------------------------------------------

def test_philox4x32_known_answers():
    """The generator's published known-answer vectors (tests/golden/philox4x32_10_kat.json)."""
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.json")) as f:
        kat = json.load(f)
    for v in kat["vectors"]:
        c = [int(x, 16) for x in v["counter"]]
        k = [int(x, 16) for x in v["key"]]
        assert list(oracle.philox4x32(c, k)) == [int(x, 16) for x in v["out"]]


_TRITON_PHILOX = r"""
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import torch, triton, triton.language as tl
from triton.language.random import philox_impl

@triton.jit
def kern(c_ptr, k_ptr, o_ptr, N: tl.constexpr):
    i = tl.arange(0, N)
    r = philox_impl(tl.load(c_ptr + 4 * i), tl.load(c_ptr + 4 * i + 1), tl.load(c_ptr + 4 * i + 2),
                    tl.load(c_ptr + 4 * i + 3), tl.load(k_ptr + 2 * i), tl.load(k_ptr + 2 * i + 1), 10)
    for w in tl.static_range(4):
        tl.store(o_ptr + 4 * i + w, r[w])

cs, ks = json.loads(sys.argv[1])
n = len(ks)
c = torch.tensor(sum(cs, []), dtype=torch.int64).to(torch.uint32)
k = torch.tensor(sum(ks, []), dtype=torch.int64).to(torch.uint32)
o = torch.zeros(4 * n, dtype=torch.uint32)
kern[(1,)](c, k, o, N=n)
print(json.dumps([int(x) & 0xffffffff for x in o.to(torch.int64)]))
"""


def test_philox4x32_matches_triton_interpreter():
    """Triton's own Philox4x32 (its language library, run by its CPU interpreter in a child
    process) on seeded counters and keys, including all-ones words."""
    pytest.importorskip("triton")
    rng = np.random.default_rng(11)
    cs = [[int(x) for x in rng.integers(0, 2 ** 32, size=4)] for _ in range(14)] + [[2 ** 32 - 1] * 4, [0, 1, 2, 3]]
    ks = [[int(x) for x in rng.integers(0, 2 ** 32, size=2)] for _ in range(14)] + [[2 ** 32 - 1, 0], [5, 2 ** 31]]
    r = subprocess.run([sys.executable, "-c", _TRITON_PHILOX, json.dumps([cs, ks])], capture_output=True, text=True,
                       timeout=600)
    if r.returncode != 0:
        pytest.skip("Triton's interpreter is unavailable here: " + r.stderr[-300:])
    got = json.loads(r.stdout.strip().splitlines()[-1])
    for n, (c, k) in enumerate(zip(cs, ks)):
        assert list(oracle.philox4x32(c, k)) == got[4 * n:4 * n + 4]


def test_keep_mask_layout_of_one_block():
    """Element n of a row takes the 16-bit half n % 2 of word (n % 8) // 2 of block n // 8:
    the 8 elements of one block, drawn through dropout_keep, against the block's words."""
    seed, offset = 0x1234_5678_9ABC_DEF0, 0x0000_0003_0000_0007
    b, h, s_q, s_kv = 1, 1, 2, 128
    keep_lo = oracle.dropout_keep(b, h, s_q, s_kv, 0.5, seed, offset)[0, 0]
    for i in range(s_q):
        for g in (0, 5, 15):
            blk = (i * 128) // 8 + g
            words = oracle.philox4x32((blk, 0, offset & 0xFFFFFFFF, offset >> 32), (seed & 0xFFFFFFFF, seed >> 32))
            halves = [(words[e // 2] >> (16 * (e % 2))) & 0xFFFF for e in range(8)]
            assert [bool(x >= 32768) for x in halves] == list(keep_lo[i, 8 * g:8 * g + 8])


def test_dropout_threshold():
    assert oracle.dropout_threshold(0.0) == 0
    assert oracle.dropout_threshold(0.5) == 32768
    assert oracle.dropout_threshold(0.1) == 6554
    assert oracle.dropout_threshold(1 - 2 ** -20) == 65536
    with pytest.raises(ValueError):
        oracle.dropout_threshold(1.0)


def test_dropout_keep_mask_properties():
    """p = 0 keeps everything; the kept fraction is 1 - p within 5 sigma; a larger p drops a
    superset (same draws, higher threshold); drawing selected rows equals the full draw;
    seeds and offsets change the draw."""
    b, h, s_q, s_kv = 1, 2, 40, 300
    assert oracle.dropout_keep(b, h, s_q, s_kv, 0.0, 1, 0).all()
    k3 = oracle.dropout_keep(b, h, s_q, s_kv, 0.3, 1234, 7)
    k6 = oracle.dropout_keep(b, h, s_q, s_kv, 0.6, 1234, 7)
    n = k3.size
    for kk, p in ((k3, 0.3), (k6, 0.6)):
        assert abs(kk.sum() - n * (1 - p)) < 5 * math.sqrt(n * p * (1 - p))
    assert not (k6 & ~k3).any()
    rows = [(1, 0), (0, 39), (1, 17)]
    sub = oracle.dropout_keep(b, h, s_q, s_kv, 0.3, 1234, 7, rows=rows)
    for r, (bh, i) in enumerate(rows):
        assert (sub[r] == k3[0, bh, i]).all()
    assert (oracle.dropout_keep(b, h, s_q, s_kv, 0.3, 1235, 7) != k3).mean() > 0.2
    assert (oracle.dropout_keep(b, h, s_q, s_kv, 0.3, 1234, 8) != k3).mean() > 0.2


def test_dropout_forward_is_unbiased_exactly():
    """Averaging O over every keep pattern of one row, weighted by its probability, gives the
    undropped O exactly (E[keep / (1 - p)] = 1); LSE never depends on the mask."""
    q, k, v = _rand(1, 1, 1, 4), _rand(1, 1, 3, 4), _rand(1, 1, 3, 4)
    p = 0.35
    O0, L0 = oracle.forward(q, k, v, 0.7, False)
    acc = np.zeros_like(O0)
    for bits in range(8):
        keep = np.array([[[[bool(bits >> j & 1) for j in range(3)]]]])
        w = (1 - p) ** keep.sum() * p ** (3 - keep.sum())
        O, L = oracle.forward(q, k, v, 0.7, False, dropout_p=p, keep=keep)
        np.testing.assert_allclose(L, L0, atol=1e-15)
        acc += w * O
    np.testing.assert_allclose(acc, O0, atol=1e-12)


def test_dropout_backward_matches_finite_differences():
    rng = np.random.default_rng(3)
    q, k, v, do = _rand(1, 2, 5, 3), _rand(1, 1, 6, 3), _rand(1, 1, 6, 3), _rand(1, 2, 5, 3)
    keep = rng.random((1, 2, 5, 6)) > 0.4
    p = 0.4
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.6, True, dropout_p=p, keep=keep)

    def loss(q_, k_, v_):
        O, _ = oracle.forward(q_, k_, v_, 0.6, True, dropout_p=p, keep=keep)
        return float((O * do).sum())
    for which, got in ((0, dQ), (1, dK), (2, dV)):
        args = [q.copy(), k.copy(), v.copy()]
        x = args[which]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + 1e-6
            lp = loss(*args)
            x[idx] = old - 1e-6
            lm = loss(*args)
            x[idx] = old
            fd[idx] = (lp - lm) / 2e-6
        assert np.linalg.norm(got - fd) / np.linalg.norm(fd) < 1e-6


# ---------------------------------------------------------------------------
# Additive bias tensor
# ---------------------------------------------------------------------------

def test_bias_brute_force_and_broadcast():
    q, k, v = _rand(2, 3, 4, 3), _rand(2, 3, 5, 3), _rand(2, 3, 5, 3)
    rng = np.random.default_rng(11)
    for shape in ((2, 3, 4, 5), (1, 3, 4, 5), (2, 1, 4, 5), (1, 1, 4, 5)):
        bias = rng.standard_normal(shape)
        O, L = oracle.forward(q, k, v, 0.9, False, bias=bias)
        for b in range(2):
            for h in range(3):
                bb = bias[b if shape[0] > 1 else 0, h if shape[1] > 1 else 0]
                for i in range(4):
                    w = [math.exp(0.9 * float(q[b, h, i] @ k[b, h, j]) + bb[i, j]) for j in range(5)]
                    np.testing.assert_allclose(O[b, h, i], sum(w[j] / sum(w) * v[b, h, j] for j in range(5)),
                                               atol=1e-12)
                    np.testing.assert_allclose(L[b, h, i], math.log(sum(w)), atol=1e-12)


def test_bias_invariances():
    """A bias constant along each row changes O but not P (shift invariance of softmax), and
    only shifts LSE; a -inf bias above the diagonal is the causal mask; the ALiBi matrix
    passed as a bias equals the ALiBi option."""
    q, k, v = _rand(1, 2, 6, 4), _rand(1, 2, 6, 4), _rand(1, 2, 6, 4)
    O0, L0 = oracle.forward(q, k, v, 0.5, False)
    rows = np.arange(6, dtype=np.float64)[None, None, :, None] * np.ones((1, 2, 6, 6))
    O1, L1 = oracle.forward(q, k, v, 0.5, False, bias=rows)
    np.testing.assert_allclose(O1, O0, atol=1e-13)
    np.testing.assert_allclose(L1 - L0, np.arange(6.0)[None, None, :] * np.ones((1, 2, 6)), atol=1e-13)
    neg = np.where(np.arange(6)[None, :] > np.arange(6)[:, None], -np.inf, 0.0)[None, None]
    Oc, Lc = oracle.forward(q, k, v, 0.5, True)
    Ob, Lb = oracle.forward(q, k, v, 0.5, False, bias=neg)
    np.testing.assert_allclose(Ob, Oc, atol=1e-13)
    np.testing.assert_allclose(Lb, Lc, atol=1e-13)
    slopes = [0.3, 0.05]
    al = np.stack([oracle.alibi_bias(6, 6, s) for s in slopes])[None]
    Oa, La = oracle.forward(q, k, v, 0.5, True, alibi_slopes=slopes)
    Ot, Lt = oracle.forward(q, k, v, 0.5, True, bias=al)
    np.testing.assert_allclose(Ot, Oa, atol=1e-13)
    np.testing.assert_allclose(Lt, La, atol=1e-13)


def test_bias_backward_matches_finite_differences():
    rng = np.random.default_rng(5)
    q, k, v, do = _rand(1, 2, 4, 3), _rand(1, 1, 5, 3), _rand(1, 1, 5, 3), _rand(1, 2, 4, 3)
    bias = rng.standard_normal((1, 2, 4, 5))
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.7, True, bias=bias)

    def loss(q_, k_, v_):
        O, _ = oracle.forward(q_, k_, v_, 0.7, True, bias=bias)
        return float((O * do).sum())
    for which, got in ((0, dQ), (1, dK), (2, dV)):
        args = [q.copy(), k.copy(), v.copy()]
        x = args[which]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + 1e-6
            lp = loss(*args)
            x[idx] = old - 1e-6
            lm = loss(*args)
            x[idx] = old
            fd[idx] = (lp - lm) / 2e-6
        assert np.linalg.norm(got - fd) / np.linalg.norm(fd) < 1e-6


@pytest.mark.parametrize("shape", [(1, 2, 4, 5), (1, 1, 4, 5)])
def test_bias_gradient_finite_differences_and_row_sums(shape):
    """dL/dbias against central differences of L = sum(O * dO), for a per-head and a fully
    broadcast bias; each row of dS sums to zero (sum_j P_ij (dP_ij - Delta_i) = 0)."""
    rng = np.random.default_rng(21)
    q, k, v, do = _rand(1, 2, 4, 3), _rand(1, 2, 5, 3), _rand(1, 2, 5, 3), _rand(1, 2, 4, 3)
    bias = rng.standard_normal(shape)
    g = oracle.bias_gradient(q, k, v, do, 0.8, False, bias)
    assert g.shape == bias.shape
    fd = np.zeros_like(bias)
    for idx in np.ndindex(bias.shape):
        bp, bm = bias.copy(), bias.copy()
        bp[idx] += 1e-6
        bm[idx] -= 1e-6
        lp = float((oracle.forward(q, k, v, 0.8, False, bias=bp)[0] * do).sum())
        lm = float((oracle.forward(q, k, v, 0.8, False, bias=bm)[0] * do).sum())
        fd[idx] = (lp - lm) / 2e-6
    assert np.linalg.norm(g - fd) / np.linalg.norm(fd) < 1e-6
    np.testing.assert_allclose(g.sum(axis=-1), 0.0, atol=1e-12)


def test_row_forms_reproduce_lengths_and_bottom_right():
    """The reductions the full-size sampled tests rely on: a bottom-right row r of a
    [s_q, s_kv] problem is the top-left row r + (s_kv - s_q) of the row form, and a valid row
    of a padded batch is the row form over that batch's own keys.  Checked against the full
    forward (with its own explicit mask) and dQ against the full backward."""
    q, k, v, do = _rand(2, 2, 5, 4), _rand(2, 2, 9, 4), _rand(2, 2, 9, 4), _rand(2, 2, 5, 4)
    O, L = oracle.forward(q, k, v, 0.6, True, bottom_right=True)
    dQ, _, _ = oracle.backward(q, k, v, do, 0.6, True, bottom_right=True)
    rows = [0, 2, 4]
    for bi in range(2):
        for h in range(2):
            Or, Lr = oracle.forward_rows(q[bi, h, rows], [r + 4 for r in rows], k[bi, h], v[bi, h], 0.6, True)
            np.testing.assert_allclose(Or, O[bi, h, rows], atol=1e-13)
            np.testing.assert_allclose(Lr, L[bi, h, rows], atol=1e-13)
            dqr = oracle.backward_dq_rows(q[bi, h, rows], do[bi, h, rows], [r + 4 for r in rows], k[bi, h],
                                          v[bi, h], 0.6, True)
            np.testing.assert_allclose(dqr, dQ[bi, h, rows], atol=1e-12)
    q, k, v, do = _rand(2, 2, 9, 4), _rand(2, 2, 9, 4), _rand(2, 2, 9, 4), _rand(2, 2, 9, 4)
    lens = [9, 6]
    O, L = oracle.forward(q, k, v, 0.6, True, lens, lens)
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.6, True, lens, lens)
    bi, n = 1, lens[1]
    rows = list(range(n))
    Or, Lr = oracle.forward_rows(q[bi, 1, rows], rows, k[bi, 1, :n], v[bi, 1, :n], 0.6, True)
    np.testing.assert_allclose(Or, O[bi, 1, :n], atol=1e-13)
    np.testing.assert_allclose(Lr, L[bi, 1, :n], atol=1e-13)
    gk, gv = oracle.backward_kv_head(q[bi:bi + 1, :, :n], k[bi:bi + 1, :, :n], v[bi:bi + 1, :, :n],
                                     do[bi:bi + 1, :, :n], 0.6, True, 0, 1)
    np.testing.assert_allclose(gk, dK[bi, 1, :n], atol=1e-12)
    np.testing.assert_allclose(gv, dV[bi, 1, :n], atol=1e-12)
    assert (O[bi, :, n:] == 0).all() and np.isneginf(L[bi, :, n:]).all()
    assert (dK[bi, :, n:] == 0).all() and (dV[bi, :, n:] == 0).all() and (dQ[bi, :, n:] == 0).all()


def test_row_forms_with_a_bias_or_alibi():
    """The row forms with an additive term, as the full-size ALiBi and bias tests use them:
    rows of the full forward (O, LSE), of the full backward (dQ), of the bias gradient (dS
    summed over the batch of a broadcast bias) and whole KV heads of dK, dV, for ALiBi rows
    (top-left and bottom-right) and for slices of a bias tensor."""
    rng = np.random.default_rng(17)
    b, h, s = 2, 2, 7
    q, k, v, do = _rand(b, h, s, 3), _rand(b, h, s, 3), _rand(b, h, s, 3), _rand(b, h, s, 3)
    slopes = [0.35, 1.2]
    rows = [0, 3, 6]
    for br in (False, True):
        s_q = 4 if br else s
        qq, dd = q[:, :, :s_q], do[:, :, :s_q]
        off = s - s_q if br else 0
        O, L = oracle.forward(qq, k, v, 0.6, True, None, None, br, alibi_slopes=slopes)
        dQ, dK, dV = oracle.backward(qq, k, v, dd, 0.6, True, None, None, br, alibi_slopes=slopes)
        rr = [r for r in rows if r < s_q]
        for bi in range(b):
            for hq in range(h):
                al = oracle.alibi_bias(s_q, s, slopes[hq], off, rows=rr)
                np.testing.assert_allclose(al, oracle.alibi_bias(s_q, s, slopes[hq], off)[rr], atol=0)
                shifted = [r + off for r in rr]
                Or, Lr = oracle.forward_rows(qq[bi, hq, rr], shifted, k[bi, hq], v[bi, hq], 0.6, True, al)
                np.testing.assert_allclose(Or, O[bi, hq, rr], atol=1e-13)
                np.testing.assert_allclose(Lr, L[bi, hq, rr], atol=1e-13)
                g = oracle.backward_dq_rows(qq[bi, hq, rr], dd[bi, hq, rr], shifted, k[bi, hq], v[bi, hq], 0.6,
                                            True, al)
                np.testing.assert_allclose(g, dQ[bi, hq, rr], atol=1e-12)
        if not br:
            fn = lambda hq, r0, r1: oracle.alibi_bias(s, s, slopes[hq], 0, rows=np.arange(r0, r1))
            gk, gv = oracle.backward_kv_head(q, k, v, do, 0.6, True, 1, 1, row_chunk=3, bias_rows=fn)
            np.testing.assert_allclose(gk, dK[1, 1], atol=1e-12)
            np.testing.assert_allclose(gv, dV[1, 1], atol=1e-12)
    # a bias tensor broadcast over the batch, GQA (2 query heads on 1 KV head)
    k1, v1 = k[:, :1], v[:, :1]
    bias = rng.standard_normal((1, h, s, s))
    O, L = oracle.forward(q, k1, v1, 0.6, True, bias=bias)
    dQ, dK, dV = oracle.backward(q, k1, v1, do, 0.6, True, bias=bias)
    dB = oracle.bias_gradient(q, k1, v1, do, 0.6, True, bias)
    for hq in range(h):
        acc = np.zeros((len(rows), s))
        for bi in range(b):
            Or, Lr = oracle.forward_rows(q[bi, hq, rows], rows, k1[bi, 0], v1[bi, 0], 0.6, True, bias[0, hq, rows])
            np.testing.assert_allclose(Or, O[bi, hq, rows], atol=1e-13)
            np.testing.assert_allclose(Lr, L[bi, hq, rows], atol=1e-13)
            g = oracle.backward_dq_rows(q[bi, hq, rows], do[bi, hq, rows], rows, k1[bi, 0], v1[bi, 0], 0.6, True,
                                        bias[0, hq, rows])
            np.testing.assert_allclose(g, dQ[bi, hq, rows], atol=1e-12)
            acc += oracle.backward_ds_rows(q[bi, hq, rows], do[bi, hq, rows], rows, k1[bi, 0], v1[bi, 0], 0.6,
                                           True, bias[0, hq, rows])
        np.testing.assert_allclose(acc, dB[0, hq, rows], atol=1e-12)
    fn = lambda hq, r0, r1: bias[0, hq, r0:r1]
    gk, gv = oracle.backward_kv_head(q, k1, v1, do, 0.6, True, 0, 0, row_chunk=2, bias_rows=fn)
    np.testing.assert_allclose(gk, dK[0, 0], atol=1e-12)
    np.testing.assert_allclose(gv, dV[0, 0], atol=1e-12)


def test_philox4x32_arrays_known_answers_and_scalar_form():
    """The array form of the generator: the published known-answer vectors, and the scalar
    form on random counters and keys (including words with the top bit set)."""
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.json")) as f:
        kat = json.load(f)
    for v in kat["vectors"]:
        c = [int(x, 16) for x in v["counter"]]
        k = [int(x, 16) for x in v["key"]]
        got = oracle.philox4x32_arrays(*(np.array([w]) for w in c), k)
        assert [int(w[0]) for w in got] == [int(x, 16) for x in v["out"]]
    rng = np.random.default_rng(11)
    ctr = rng.integers(0, 2 ** 32, size=(4, 64), dtype=np.uint64)
    for key in [(0, 0), (0xFFFFFFFF, 0x80000001), (int(rng.integers(0, 2 ** 32)), int(rng.integers(0, 2 ** 32)))]:
        got = oracle.philox4x32_arrays(ctr[0], ctr[1], ctr[2], ctr[3], key)
        for n in range(64):
            want = oracle.philox4x32([int(ctr[i, n]) for i in range(4)], key)
            assert tuple(int(w[n]) for w in got) == want


@pytest.mark.parametrize("s_q,s_kv,p", [(5, 200, 0.1), (3, 128, 0.5), (4, 9, 0.25)])
def test_dropout_keep_range_is_the_row_draw(s_q, s_kv, p):
    """The range draw equals dropout_keep's element-by-element draw, row for row (ragged key
    lengths, so that rows start in a new 128-element stretch; a large offset and seed)."""
    seed, offset = (1 << 40) + 77, (3 << 33) + 5
    b, h = 2, 3
    full = oracle.dropout_keep(b, h, s_q, s_kv, p, seed, offset)
    for bh in (0, 4, 5):
        got = oracle.dropout_keep_range(b, h, s_q, s_kv, p, seed, offset, bh, 1, s_q)
        np.testing.assert_array_equal(got, full[bh // h, bh % h, 1:s_q])


def test_row_forms_with_dropout():
    """The row forms with a dropout factor, as the full-size dropout test uses them: rows of
    the full forward (O, LSE) and backward (dQ), and whole KV heads of dK, dV, causal and not,
    with GQA (2 query heads on 1 KV head)."""
    b, h_q, h_kv, s, d, p = 2, 4, 2, 9, 3, 0.3
    q, do = _rand(b, h_q, s, d), _rand(b, h_q, s, d)
    k, v = _rand(b, h_kv, s, d), _rand(b, h_kv, s, d)
    keep = oracle.dropout_keep(b, h_q, s, s, p, 99, 1)
    z = keep.astype(np.float64) / (1.0 - p)
    rows = [0, 4, 8]
    for causal in (False, True):
        O, L = oracle.forward(q, k, v, 0.6, causal, dropout_p=p, keep=keep)
        dQ, dK, dV = oracle.backward(q, k, v, do, 0.6, causal, dropout_p=p, keep=keep)
        for bi in range(b):
            for hq in range(h_q):
                hk = oracle.kv_head_of(hq, h_q, h_kv)
                Or, Lr = oracle.forward_rows(q[bi, hq, rows], rows, k[bi, hk], v[bi, hk], 0.6, causal,
                                             zdrop=z[bi, hq, rows])
                np.testing.assert_allclose(Or, O[bi, hq, rows], atol=1e-13)
                np.testing.assert_allclose(Lr, L[bi, hq, rows], atol=1e-13)
                g = oracle.backward_dq_rows(q[bi, hq, rows], do[bi, hq, rows], rows, k[bi, hk], v[bi, hk], 0.6,
                                            causal, zdrop=z[bi, hq, rows])
                np.testing.assert_allclose(g, dQ[bi, hq, rows], atol=1e-12)
        for bi, hk in ((0, 1), (1, 0)):
            fn = lambda hq, r0, r1, bi=bi: z[bi, hq, r0:r1]
            gk, gv = oracle.backward_kv_head(q, k, v, do, 0.6, causal, bi, hk, row_chunk=4, zdrop_rows=fn)
            np.testing.assert_allclose(gk, dK[bi, hk], atol=1e-12)
            np.testing.assert_allclose(gv, dV[bi, hk], atol=1e-12)
