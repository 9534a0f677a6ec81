"""GPU parity of dropout: the Philox4x32-10 keep bits bit for bit, then forward and backward
against the fp64 oracle driven by the oracle's own keep mask.

The mask kernel must reproduce the oracle's draw exactly (row-major and transposed, ragged
sizes, 64-bit seeds and offsets, several probabilities).  The attention kernels read those
bits; the oracle draws its own and applies O = (P * keep) V / (1 - p)."""
import numpy as np
import pytest
import torch

import oracle
from sdpa_workloads import Workload, make_inputs
from sdpa_testlib import (assert_fwd_close, assert_grad_close, assert_lse_close, dropout_masks, f64,
                          lib, run_bwd, run_fwd)

pytestmark = pytest.mark.gpu

MODES = {"none": (False, False), "top_left": (True, False), "bottom_right": (True, True)}


def _tbit(i):
    """Bit of element i within its word of either mask (an even/odd pair sits 16 bits apart):
    16 * (i % 2) + (i % 32) / 2."""
    i = np.asarray(i)
    return (16 * (i % 2) + (i % 32) // 2).astype(np.uint32)


def _unpack(words: torch.Tensor, n_rows: int, n_words: int, n_valid: int) -> np.ndarray:
    """Row-major keep bits: key j of a row at bit _tbit(j) of word j / 32."""
    w = words.cpu().numpy().view(np.uint32).reshape(n_rows, n_words)
    j = np.arange(n_valid)
    return ((w[:, j // 32] >> _tbit(j)) & 1).astype(bool)


def _unpack_t(words: torch.Tensor, n_rows: int, n_words: int, n_valid: int) -> np.ndarray:
    """Transposed keep bits: query row i of a key at bit _tbit(i) of word i / 32."""
    w = words.cpu().numpy().view(np.uint32).reshape(n_rows, n_words)
    i = np.arange(n_valid)
    return ((w[:, i // 32] >> _tbit(i)) & 1).astype(bool)


def _p32(p):
    return float(np.float32(p))   # the library takes the probability as fp32


@pytest.mark.parametrize("b,h,s_q,s_kv", [(1, 1, 1, 1), (2, 3, 100, 129), (1, 2, 300, 77),
                                          (1, 1, 128, 256), (2, 1, 257, 300)])
@pytest.mark.parametrize("p,seed,offset", [(0.1, 0, 0), (0.5, 2 ** 64 - 1, 12345),
                                           (0.9, 987654321, 2 ** 63 + 5)])
def test_mask_bits_equal_the_oracle_draw(b, h, s_q, s_kv, p, seed, offset):
    mask, mask_t = dropout_masks(b, h, s_q, s_kv, (p, seed, offset))
    torch.cuda.synchronize()
    keep = oracle.dropout_keep(b, h, s_q, s_kv, _p32(p), seed, offset).reshape(b * h, s_q, s_kv)
    kvw, qw = (s_kv + 127) // 128 * 4, (s_q + 127) // 128 * 4
    rows = _unpack(mask, b * h * s_q, kvw, s_kv).reshape(b * h, s_q, s_kv)
    assert (rows == keep).all()
    cols = _unpack_t(mask_t, b * h * s_kv, qw, s_q).reshape(b * h, s_kv, s_q)
    assert (cols == keep.transpose(0, 2, 1)).all()


def test_mask_p_zero_keeps_everything_and_sizes():
    m = lib()
    n, n_t = m.sdpa_dropout_mask_size(2, 3, 200, 300)
    assert n == 2 * 3 * 200 * 12 * 4 and n_t == 2 * 3 * 300 * 8 * 4
    mask, mask_t = dropout_masks(2, 3, 200, 300, (0.0, 5, 6))
    assert _unpack(mask, 6 * 200, 12, 300).all() and _unpack_t(mask_t, 6 * 300, 8, 200).all()


def _case(w, mode, p, seed, offset, lq=None, lkv=None, alibi=None, backward=False):
    causal, br = MODES[mode]
    cflag = "bottom_right" if br else causal
    drop = (p, seed, offset)
    x = make_inputs(w, seed=seed % 1000, with_do=backward)
    o, lse, dev = run_fwd(w, x, causal=cflag, seq_lens_q=lq, seq_lens_kv=lkv, alibi=alibi, dropout=drop)
    keep = oracle.dropout_keep(w.b, w.h_q, w.s_q, w.s_kv, _p32(p), seed, offset)
    slopes = oracle.alibi_default_slopes(w.h_q) if alibi == "default" else alibi
    q64, k64, v64 = f64(x.q), f64(x.k), f64(x.v)
    O, L = oracle.forward(q64, k64, v64, w.scale, causal, lq, lkv, br, alibi_slopes=slopes,
                          dropout_p=_p32(p), keep=keep)
    # Kept P are scaled by 1/(1 - p), so O's magnitude (and its bf16 rounding) grows by that
    # factor: compare (1 - p) O with the usual absolute tolerances.
    assert_fwd_close(f64(o) * (1 - p), O * (1 - p))
    got_l = lse.cpu().double().numpy()
    inf = np.isneginf(L)
    assert (np.isneginf(got_l) == inf).all()
    assert_lse_close(got_l[~inf], L[~inf])
    if backward:
        dq, dk, dv = run_bwd(w, dev, o, lse, x.do, causal=cflag, seq_lens_q=lq, seq_lens_kv=lkv,
                             alibi=alibi, dropout=drop)
        dQ, dK, dV = oracle.backward(q64, k64, v64, f64(x.do), w.scale, causal, lq, lkv, br,
                                     alibi_slopes=slopes, dropout_p=_p32(p), keep=keep)
        assert_grad_close(f64(dq), dQ, "dQ")
        assert_grad_close(f64(dk), dK, "dK")
        assert_grad_close(f64(dv), dV, "dV")


@pytest.mark.parametrize("mode", ["none", "top_left"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_forward_backward(mode, d, dtype):
    w = Workload("t", 2, 4, 2, 260, 300, d, dtype, backward=True)
    _case(w, mode, 0.2, 1000 + d, 3, backward=True)


@pytest.mark.parametrize("p", [0.05, 0.5, 0.9])
def test_probabilities(p):
    w = Workload("t", 1, 2, 2, 384, 384, 128, "bf16", causal=True, backward=True)
    _case(w, "top_left", p, 77, 11, backward=True)


def test_with_alibi_lengths_and_bottom_right():
    w = Workload("t", 3, 4, 2, 200, 333, 128, "bf16", backward=True)
    _case(w, "bottom_right", 0.3, 5, 9, lq=[200, 57, 0], lkv=[333, 200, 100], alibi="default",
          backward=True)


def test_split_groups():
    """h_kv = 1: the backward pass splits a KV block's 16 query heads over several CTAs, each
    reading the keep bits of its own heads."""
    w = Workload("t", 1, 16, 1, 640, 640, 64, "f16", causal=True, backward=True)
    _case(w, "top_left", 0.25, 2024, 1, backward=True)


def test_d256_ragged():
    w = Workload("t", 1, 2, 2, 129, 70, 256, "bf16", backward=True)
    _case(w, "none", 0.4, 31, 4, backward=True)


def test_training_shape_sampled_rows():
    """At the full training shape (b2 h16 s8192) the mask kernel's bits match the oracle on
    sampled rows of both layouts."""
    b, h, s = 2, 16, 8192
    mask, mask_t = dropout_masks(b, h, s, s, (0.1, 42, 7))
    torch.cuda.synchronize()
    words = s // 32
    rows = [(0, 0), (5, 4097), (31, 8191), (17, 1234)]
    keep = oracle.dropout_keep(b, h, s, s, _p32(0.1), 42, 7, rows=rows)
    mw = mask.view(b * h, s, words)
    mtw = mask_t.view(b * h, s, words)
    for r, (bh, i) in enumerate(rows):
        got = _unpack(mw[bh, i].contiguous(), 1, words, s)[0]
        assert (got == keep[r]).all()
        # transposed: bit i of key j's words for j in a sample of columns
        js = np.array([0, 1, 31, 32, 4096, 8191])
        col = mtw[bh, js].cpu().numpy().view(np.uint32)
        bits = ((col[:, i // 32] >> _tbit(i)) & 1).astype(bool)
        assert (bits == keep[r][js]).all()


@pytest.mark.parametrize("causal", [True, "bottom_right"])
def test_causal_draw_writes_every_visible_tile(causal):
    """A causal draw skips only tiles wholly above the diagonal: every bit a row can see still
    equals the oracle's, and the skipped tiles keep their previous contents."""
    b, h, s_q, s_kv = 1, 2, 300, 400
    mask, mask_t = dropout_masks(b, h, s_q, s_kv, (0.3, 99, 1), causal=causal)
    torch.cuda.synchronize()
    keep = oracle.dropout_keep(b, h, s_q, s_kv, _p32(0.3), 99, 1).reshape(b * h, s_q, s_kv)
    off = s_kv - s_q if causal == "bottom_right" else 0
    vis = np.arange(s_kv)[None, :] <= np.arange(s_q)[:, None] + off
    rows = _unpack(mask, b * h * s_q, 16, s_kv).reshape(b * h, s_q, s_kv)
    cols = _unpack_t(mask_t, b * h * s_kv, 12, s_q).reshape(b * h, s_kv, s_q)
    assert (rows[:, vis] == keep[:, vis]).all()
    assert (cols.transpose(0, 2, 1)[:, vis] == keep[:, vis]).all()
    # a tile wholly above the diagonal (rows 0-127, keys 256-383 top-left) is untouched (-1)
    if causal is True:
        assert rows[:, :128, 256:384].all()
