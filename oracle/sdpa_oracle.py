"""fp64 CPU oracle for scaled dot-product attention (forward and backward).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and ``--impl reference`` arm) may import
this module.  The product path (the CUDA library and its Python binding) never
imports, calls or links it, and this module imports nothing from the product.

What it computes is the plain definition, written out step by step in float64 on
the exact input values (fp16 / bf16 upcast exactly; E4M3 bytes decoded by this
module's own table and multiplied by their descale):

* scores ``S = attn_scale * Q Kᵀ``, a naive matrix product
  [attention codelab, §1 "How attention works", step 1; §4 "Implementing
  attention from scratch"; cuDNN 9 blog, "SDPA as a cuDNN graph", Fig. 4: the
  scale is a pointwise multiply right after BMM1];
* an explicit mask: with ``causal`` key j is visible to query i iff ``j <= i``
  (top-left alignment) [codelab §7 "Adding a causal mask": position 0 sees only
  itself, the last position sees every position];
* a three-pass softmax over the visible keys: row max, sum of exponentials,
  normalise [codelab §1 step 2];
* ``O = P V`` [codelab §1 step 3], output with Q's shape [step 4];
* the per-row statistics ``LSE_i = m_i + ln l_i`` (natural log) — the reading of the
  "stats" output that the SDPA node returns for training [cuDNN 9 blog, SDPA
  walkthrough sample; cuDNN-in-Python post: the second return value is for
  training];
* variable lengths (the padding mask and per-batch sequence lengths of the SDPA node's
  options in the cuDNN 9 blog's walkthrough): for batch b only query rows i < len_q[b] and
  keys j < len_kv[b] take part; with bottom-right causal alignment key j is visible to query
  i iff j <= i + len_kv[b] - len_q[b] (the last query sees every key, as in decoding with a
  KV cache).  A row with no visible key (a padded row, or an early row of a bottom-right
  mask with len_kv < len_q) gives O = 0 and LSE = -inf, and passes no gradient;
* ALiBi (the SDPA node's ALiBi-mask option in the cuDNN 9 blog's walkthrough): with one
  slope m_h per query head, the scaled score of (i, j) gains m_h * (j - i - off), off being
  the bottom-right offset len_kv - len_q (0 otherwise), before the mask and the softmax — a
  linear penalty on the distance to the aligned diagonal.  The pages name the option but no
  slopes; without caller slopes the default is the geometric sequence m_h = 2^(-8 (h+1) / H)
  of the ALiBi paper (Press, Smith and Lewis, "Train Short, Test Long", §3: 1/2 ... 1/256 for
  8 heads), applied by the same formula to any head count.  That paper defines the bias for
  causal attention only, as a penalty growing with a query's distance to the earlier keys it
  sees; without a causal mask the linear term would reward later keys more the farther they
  are, so ALiBi without a causal mask is not defined here and is refused (ValueError);
* an additive bias (the SDPA node's bias input in the cuDNN 9 blog's walkthrough): a tensor
  [b or 1, h_q or 1, s_q, s_kv] added to the scaled scores before the mask and the softmax
  (broadcast over a batch or head dimension of size 1).  Its gradient is dS = ∂L/∂S, the
  gradient of the scores after the scale, summed over the broadcast dimensions;
* dropout (the SDPA node's dropout option in the cuDNN 9 blog's walkthrough, named and not
  defined): after the softmax each probability is kept with a keep mask Z and the kept ones
  are scaled by 1/(1 - p), so O = (P * Z) V / (1 - p); the LSE is that of the undropped
  softmax.  The mask is drawn by the counter-based Philox4x32-10 generator (Salmon, Moraes,
  Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11): element n of the
  row-major grid [b*h_q][s_q][s_kv rounded up to 128] takes 16-bit half n % 2 (0 = low) of
  32-bit word (n % 8) // 2 of the block drawn for the 128-bit counter (n // 8, offset) and the
  64-bit key seed (each split into 32-bit words, low word first), and is kept iff that value
  is >= round(p * 65536);
* head grouping: query head ``hq`` reads KV head ``hq // (h_q // h_kv)`` (contiguous
  groups; the codelab's §9 "Comparing MHA, GQA and MQA" broadcasts each KV head to
  its group of query heads);
* the backward pass is the analytic derivative of O with respect to Q, K and V
  (the pages show a backward graph exists but print no formula): with the incoming
  gradient dO, dV = Pᵀ dO, dP = dO Vᵀ, Delta_i = Σ_j P_ij dP_ij,
  dS = P ∘ (dP − Delta), dQ = scale·dS K, dK = scale·dSᵀ Q, with dK and dV summed
  over the query heads of each KV group.  With dropout, Z = keep / (1 - p) enters as
  dV = (P∘Z)ᵀ dO and dP = Z ∘ (dO Vᵀ); the rest is unchanged.

Every function here is pinned by ``tests/test_oracle_pins.py`` against brute force,
closed forms, invariants and finite differences; none is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Iterable, Sequence, Tuple

import numpy as np

__all__ = [
    "philox4x32", "philox4x32_arrays", "dropout_threshold", "dropout_keep", "dropout_keep_range",
    "bias_gradient",
    "visible_mask", "kv_head_of", "alibi_default_slopes", "alibi_bias", "head_forward", "forward", "forward_rows",
    "backward", "backward_dq_rows", "backward_ds_rows", "backward_kv_rows", "backward_kv_head",
    "e4m3_decode_table",
    "decode_e4m3", "e5m2_decode_table", "decode_e5m2", "to_f64",
]


# ---------------------------------------------------------------------------
# Format helpers
# ---------------------------------------------------------------------------

def e4m3_decode_table() -> np.ndarray:
    """The 256 values of OCP FP8 E4M3 ("FN": no infinities, one NaN pattern per sign).

    Bit layout: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits
    [codelab §10: E4M3 = 4 exponent bits, 3 mantissa bits, used in the forward pass].
    Exponent field 0 encodes subnormals m/8 * 2**(1-7); exponent field 15 with
    mantissa 7 is NaN; every other pattern is (1 + m/8) * 2**(e-7).
    """
    tab = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            tab[code] = math.nan
        elif e == 0:
            tab[code] = sign * (m / 8.0) * 2.0 ** (1 - 7)
        else:
            tab[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return tab


_E4M3 = e4m3_decode_table()


def decode_e4m3(codes: np.ndarray, descale: float = 1.0) -> np.ndarray:
    """Exact fp64 value of E4M3 bytes times a per-tensor descale."""
    return _E4M3[np.asarray(codes, dtype=np.uint8)] * float(descale)


def e5m2_decode_table() -> np.ndarray:
    """The 256 values of OCP FP8 E5M2 (IEEE-like: infinities and NaNs).

    Bit layout: 1 sign bit, 5 exponent bits (bias 15), 2 mantissa bits — the gradient
    format of the HYBRID recipe [codelab §10: E4M3 forward, E5M2 backward].  Exponent field
    0 encodes subnormals m/4 * 2**(1-15); field 31 is infinity (m = 0) or NaN; every other
    pattern is (1 + m/4) * 2**(e-15).
    """
    tab = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 2) & 0x1F
        m = code & 0x3
        if e == 0x1F:
            tab[code] = sign * math.inf if m == 0 else math.nan
        elif e == 0:
            tab[code] = sign * (m / 4.0) * 2.0 ** (1 - 15)
        else:
            tab[code] = sign * (1.0 + m / 4.0) * 2.0 ** (e - 15)
    return tab


_E5M2 = e5m2_decode_table()


def decode_e5m2(codes: np.ndarray, descale: float = 1.0) -> np.ndarray:
    """Exact fp64 value of E5M2 bytes times a per-tensor descale."""
    return _E5M2[np.asarray(codes, dtype=np.uint8)] * float(descale)


def to_f64(t, descale: float = 1.0) -> np.ndarray:
    """Exact fp64 copy of a CPU torch tensor (fp16 / bf16 / fp32 / float8_e4m3fn /
    float8_e5m2)."""
    import torch  # plumbing only: reads the bytes of a tensor

    t = t.detach().cpu()
    if t.dtype == torch.float8_e4m3fn:
        return decode_e4m3(t.contiguous().view(torch.uint8).numpy(), descale)
    if t.dtype == torch.float8_e5m2:
        return decode_e5m2(t.contiguous().view(torch.uint8).numpy(), descale)
    return t.to(torch.float64).numpy() * float(descale)


# ---------------------------------------------------------------------------
# Forward
# ---------------------------------------------------------------------------

# Philox4x32-10 constants: the round multipliers and the Weyl key increments of the paper.
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = (1 << 32) - 1


def philox4x32(counter: Sequence[int], key: Sequence[int], rounds: int = 10) -> Tuple[int, ...]:
    """One Philox4x32 block: four 32-bit words for a 128-bit counter and a 64-bit key.

    Each round multiplies words 0 and 2 by the two constants (full 64-bit products), and
    the new words are (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0); the key gains the Weyl
    increments between rounds.  Plain Python integers, one block at a time."""
    x0, x1, x2, x3 = (int(c) & _MASK32 for c in counter)
    k0, k1 = (int(k) & _MASK32 for k in key)
    for r in range(rounds):
        if r > 0:
            k0 = (k0 + PHILOX_W0) & _MASK32
            k1 = (k1 + PHILOX_W1) & _MASK32
        p0 = PHILOX_M0 * x0
        p1 = PHILOX_M1 * x2
        hi0, lo0 = p0 >> 32, p0 & _MASK32
        hi1, lo1 = p1 >> 32, p1 & _MASK32
        x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
    return x0, x1, x2, x3


def dropout_threshold(p: float) -> int:
    """16-bit drop threshold: an element is dropped iff its 16-bit draw is below it."""
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return min(65536, int(math.floor(p * 65536.0 + 0.5)))


def dropout_keep(b: int, h_q: int, s_q: int, s_kv: int, p: float, seed: int, offset: int,
                 rows: Iterable[Tuple[int, int]] | None = None) -> np.ndarray:
    """Keep mask [b, h_q, s_q, s_kv] (bool) of the Philox draw defined in the module header.

    rows: optional (b*h_q + h, i) pairs; then only those rows are drawn and the result is
    [len(rows), s_kv]."""
    t = dropout_threshold(p)
    row_pitch = (s_kv + 127) // 128 * 128
    want = list(rows) if rows is not None else [(bh, i) for bh in range(b * h_q) for i in range(s_q)]
    out = np.empty((len(want), s_kv), dtype=bool)
    key = (seed & _MASK32, (seed >> 32) & _MASK32)
    off = (offset & _MASK32, (offset >> 32) & _MASK32)
    for r, (bh, i) in enumerate(want):
        n0 = (bh * s_q + i) * row_pitch           # multiple of 8: rows start a new block
        for g in range(row_pitch // 8):
            blk = n0 // 8 + g
            words = philox4x32((blk & _MASK32, blk >> 32, off[0], off[1]), key)
            for e in range(8):
                j = g * 8 + e
                if j < s_kv:
                    u = (words[e // 2] >> (16 * (e % 2))) & 0xFFFF
                    out[r, j] = u >= t
    if rows is None:
        return out.reshape(b, h_q, s_q, s_kv)
    return out


def visible_mask(s_q: int, s_kv: int, causal: bool, len_q: int | None = None,
                 len_kv: int | None = None, bottom_right: bool = False) -> np.ndarray:
    """Boolean [s_q, s_kv]: True where key j is visible to query i.

    len_q / len_kv: valid rows of this batch (default: all).  causal: top-left (j <= i) or,
    with bottom_right, j <= i + len_kv - len_q."""
    lq = s_q if len_q is None else len_q
    lkv = s_kv if len_kv is None else len_kv
    i = np.arange(s_q)[:, None]
    j = np.arange(s_kv)[None, :]
    m = (i < lq) & (j < lkv)
    if causal:
        off = (lkv - lq) if bottom_right else 0
        m &= j <= i + off
    return m


def kv_head_of(hq: int, h_q: int, h_kv: int) -> int:
    """KV head read by query head ``hq`` (contiguous groups of h_q // h_kv)."""
    if h_kv <= 0 or h_q % h_kv:
        raise ValueError("h_q must be a positive multiple of h_kv")
    return hq // (h_q // h_kv)


def alibi_default_slopes(h_q: int) -> np.ndarray:
    """m_h = 2^(-8 (h + 1) / h_q) for h = 0 .. h_q - 1."""
    return np.array([2.0 ** (-8.0 * (h + 1) / h_q) for h in range(h_q)], dtype=np.float64)


def alibi_bias(s_q: int, s_kv: int, slope: float, off: int = 0, rows=None) -> np.ndarray:
    """[s_q, s_kv] additive bias slope * (j - i - off); with ``rows``, only those query rows
    ([len(rows), s_kv])."""
    i = (np.arange(s_q) if rows is None else np.asarray(rows))[:, None]
    j = np.arange(s_kv)[None, :]
    return slope * (j - i - off).astype(np.float64)


def _check_alibi(causal: bool, alibi_slopes) -> None:
    """ALiBi is a distance penalty on the keys before a query (the ALiBi paper, §3): it needs
    a causal mask, which keeps every visible key at or before the aligned diagonal."""
    if alibi_slopes is not None and not causal:
        raise ValueError("ALiBi is defined for causal attention only")


def head_forward(qh: np.ndarray, kh: np.ndarray, vh: np.ndarray, scale: float,
                 mask: np.ndarray, allow_empty: bool = False, bias: np.ndarray | None = None,
                 zdrop: np.ndarray | None = None):
    """One (batch, head) slice: returns (O [s_q,d], LSE [s_q], P [s_q,s_kv]).

    bias: optional additive term on the scaled scores.  zdrop: optional dropout factor
    keep / (1 - p) applied to P for O only (P and LSE are those of the softmax).  A row with
    no visible key has no softmax: it is rejected, or with allow_empty gives O = 0,
    LSE = -inf and P = 0."""
    S = scale * (qh @ kh.T)                                   # step 1 + scale
    if bias is not None:
        S = S + bias
    has = mask.any(axis=1)
    if not allow_empty and not has.all():
        raise ValueError("a query row has no visible key")
    m = np.where(mask, S, -np.inf).max(axis=1)                # pass 1: row max
    m_safe = np.where(has, m, 0.0)
    E = np.exp(np.where(mask, S - m_safe[:, None], -np.inf))  # masked: exp(-inf) = 0
    l = E.sum(axis=1)                                         # pass 2: row sum
    P = E / np.where(has, l, 1.0)[:, None]                    # pass 3: normalise
    O = (P if zdrop is None else P * zdrop) @ vh              # step 3 (dropout on P)
    with np.errstate(divide="ignore"):
        lse = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)
    return O, lse, P


def _batch_mask(s_q, s_kv, causal, bi, seq_lens_q, seq_lens_kv, bottom_right):
    lq = None if seq_lens_q is None else int(seq_lens_q[bi])
    lkv = None if seq_lens_kv is None else int(seq_lens_kv[bi])
    return visible_mask(s_q, s_kv, causal, lq, lkv, bottom_right)


def _batch_off(s_q, s_kv, bi, seq_lens_q, seq_lens_kv, bottom_right):
    if not bottom_right:
        return 0
    lq = s_q if seq_lens_q is None else int(seq_lens_q[bi])
    lkv = s_kv if seq_lens_kv is None else int(seq_lens_kv[bi])
    return lkv - lq


def _bias_of(bias, alibi_slopes, s_q, s_kv, bi, hq, off):
    """The additive term on the scaled scores of (bi, hq): ALiBi plus a bias tensor."""
    out = None
    if alibi_slopes is not None:
        out = alibi_bias(s_q, s_kv, float(alibi_slopes[hq]), off)
    if bias is not None:
        t = np.asarray(bias, dtype=np.float64)
        term = t[bi if t.shape[0] > 1 else 0, hq if t.shape[1] > 1 else 0]
        out = term if out is None else out + term
    return out


def _zdrop(keep, dropout_p, bi, hq):
    if keep is None:
        return None
    return keep[bi, hq].astype(np.float64) / (1.0 - dropout_p)


def forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, causal: bool,
            seq_lens_q=None, seq_lens_kv=None, bottom_right: bool = False, alibi_slopes=None,
            dropout_p: float = 0.0, keep=None, bias=None):
    """Full forward on logical BHSD fp64 arrays.

    q: [b, h_q, s_q, d]; k, v: [b, h_kv, s_kv, d]; optional per-batch valid lengths,
    per-query-head ALiBi slopes, a dropout keep mask [b, h_q, s_q, s_kv] with its
    probability, and an additive bias [b|1, h_q|1, s_q, s_kv].  Returns (O [b,h_q,s_q,d],
    LSE [b,h_q,s_q])."""
    _check_alibi(causal, alibi_slopes)
    b, h_q, s_q, d = q.shape
    h_kv, s_kv = k.shape[1], k.shape[2]
    varlen = seq_lens_q is not None or seq_lens_kv is not None or bottom_right
    O = np.empty((b, h_q, s_q, v.shape[3]), dtype=np.float64)
    L = np.empty((b, h_q, s_q), dtype=np.float64)
    for bi in range(b):
        mask = _batch_mask(s_q, s_kv, causal, bi, seq_lens_q, seq_lens_kv, bottom_right)
        off = _batch_off(s_q, s_kv, bi, seq_lens_q, seq_lens_kv, bottom_right)
        for hq in range(h_q):
            hk = kv_head_of(hq, h_q, h_kv)
            term = _bias_of(bias, alibi_slopes, s_q, s_kv, bi, hq, off)
            O[bi, hq], L[bi, hq], _ = head_forward(q[bi, hq], k[bi, hk], v[bi, hk], scale, mask,
                                                   allow_empty=varlen, bias=term,
                                                   zdrop=_zdrop(keep, dropout_p, bi, hq))
    return O, L


def philox4x32_arrays(c0, c1, c2, c3, key: Sequence[int], rounds: int = 10):
    """philox4x32 on arrays of counters: the same rounds, elementwise, in numpy uint64 (a 32 x
    32-bit product fits).  c0..c3: integer arrays of 32-bit counter words (broadcast
    together).  Returns the four output word arrays (uint64 holding 32-bit values)."""
    m32 = np.uint64(_MASK32)
    x0, x1, x2, x3 = (np.asarray(c, dtype=np.uint64) & m32 for c in (c0, c1, c2, c3))
    x0, x1, x2, x3 = np.broadcast_arrays(x0, x1, x2, x3)
    k0, k1 = (int(k) & _MASK32 for k in key)
    for r in range(rounds):
        if r > 0:
            k0 = (k0 + PHILOX_W0) & _MASK32
            k1 = (k1 + PHILOX_W1) & _MASK32
        p0 = np.uint64(PHILOX_M0) * x0
        p1 = np.uint64(PHILOX_M1) * x2
        hi0, lo0 = p0 >> np.uint64(32), p0 & m32
        hi1, lo1 = p1 >> np.uint64(32), p1 & m32
        x0, x1, x2, x3 = hi1 ^ x1 ^ np.uint64(k0), lo1, hi0 ^ x3 ^ np.uint64(k1), lo0
    return x0, x1, x2, x3


def dropout_keep_range(b: int, h_q: int, s_q: int, s_kv: int, p: float, seed: int, offset: int,
                       bh: int, r0: int, r1: int) -> np.ndarray:
    """Keep mask [r1 - r0, s_kv] (bool) of query rows r0..r1-1 of (batch·h_q + head) bh: the
    draw of dropout_keep, with the blocks of all those rows generated at once by
    philox4x32_arrays (whole heads at s = 8192 in seconds)."""
    t = dropout_threshold(p)
    row_pitch = (s_kv + 127) // 128 * 128
    n0 = (bh * s_q + np.arange(r0, r1, dtype=np.uint64)) * np.uint64(row_pitch)   # first element of each row
    blk = (n0 // np.uint64(8))[:, None] + np.arange(row_pitch // 8, dtype=np.uint64)[None, :]
    words = philox4x32_arrays(blk & np.uint64(_MASK32), blk >> np.uint64(32), offset & _MASK32,
                              (offset >> 32) & _MASK32, (seed & _MASK32, (seed >> 32) & _MASK32))
    # element 8g + e of a row: 16-bit half e % 2 of word e // 2 of block g
    u = np.stack([(words[e // 2] >> np.uint64(16 * (e % 2))) & np.uint64(0xFFFF) for e in range(8)], axis=-1)
    return (u.reshape(r1 - r0, row_pitch) >= np.uint64(t))[:, :s_kv]


def _rows_mask(rows, s_kv: int, causal: bool) -> np.ndarray:
    rows = np.asarray(rows)
    if causal:
        return np.arange(s_kv)[None, :] <= rows[:, None]
    return np.ones((len(rows), s_kv), dtype=bool)


def forward_rows(q_rows: np.ndarray, rows: Sequence[int], kh: np.ndarray, vh: np.ndarray,
                 scale: float, causal: bool, bias: np.ndarray | None = None,
                 zdrop: np.ndarray | None = None):
    """Forward for selected query rows of one (batch, head).

    q_rows: [n, d] fp64 rows of Q; rows: their sequence positions; kh, vh: the
    row's KV head [s_kv, d]; bias: optional [n, s_kv] additive term on these rows' scaled
    scores (a slice of a bias tensor, or ALiBi's rows); zdrop: optional [n, s_kv] dropout
    factor keep / (1 - p) of these rows (as in head_forward).  Returns (O rows [n, d], LSE [n]).
    Cost O(n·s_kv·d), which lets large shapes be checked row by row."""
    O, lse, _ = head_forward(q_rows, kh, vh, scale, _rows_mask(rows, kh.shape[0], causal), bias=bias,
                             zdrop=zdrop)
    return O, lse


# ---------------------------------------------------------------------------
# Backward
# ---------------------------------------------------------------------------

def _head_backward(qh, kh, vh, doh, scale, mask, allow_empty=False, bias=None, zdrop=None):
    _, _, P = head_forward(qh, kh, vh, scale, mask, allow_empty, bias)
    Z = 1.0 if zdrop is None else zdrop
    dV = (P * Z).T @ doh
    dP = Z * (doh @ vh.T)
    delta = (P * dP).sum(axis=1)
    dS = P * (dP - delta[:, None])
    dQ = scale * (dS @ kh)
    dK = scale * (dS.T @ qh)
    return dQ, dK, dV, dS


def backward(q, k, v, do, scale: float, causal: bool, seq_lens_q=None, seq_lens_kv=None,
             bottom_right: bool = False, alibi_slopes=None, dropout_p: float = 0.0, keep=None,
             bias=None):
    """Full backward on logical BHSD fp64 arrays: returns (dQ, dK, dV).

    dK, dV have K's and V's shapes and hold the sum over each KV head's group.  With
    variable lengths, padded rows of dQ, dK and dV are zero."""
    _check_alibi(causal, alibi_slopes)
    b, h_q, s_q, _ = q.shape
    h_kv, s_kv = k.shape[1], k.shape[2]
    varlen = seq_lens_q is not None or seq_lens_kv is not None or bottom_right
    dQ = np.empty_like(q, dtype=np.float64)
    dK = np.zeros(k.shape, dtype=np.float64)
    dV = np.zeros(v.shape, dtype=np.float64)
    for bi in range(b):
        mask = _batch_mask(s_q, s_kv, causal, bi, seq_lens_q, seq_lens_kv, bottom_right)
        off = _batch_off(s_q, s_kv, bi, seq_lens_q, seq_lens_kv, bottom_right)
        for hq in range(h_q):
            hk = kv_head_of(hq, h_q, h_kv)
            term = _bias_of(bias, alibi_slopes, s_q, s_kv, bi, hq, off)
            gq, gk, gv, _ = _head_backward(q[bi, hq], k[bi, hk], v[bi, hk], do[bi, hq], scale, mask,
                                           allow_empty=varlen, bias=term,
                                           zdrop=_zdrop(keep, dropout_p, bi, hq))
            dQ[bi, hq] = gq
            dK[bi, hk] += gk
            dV[bi, hk] += gv
    return dQ, dK, dV


def bias_gradient(q, k, v, do, scale: float, causal: bool, bias, seq_lens_q=None, seq_lens_kv=None,
                  bottom_right: bool = False, dropout_p: float = 0.0, keep=None):
    """dL/dbias with the bias's shape [b|1, h_q|1, s_q, s_kv]: dS of every (batch, head),
    summed over the broadcast dimensions."""
    b, h_q, s_q, _ = q.shape
    h_kv, s_kv = k.shape[1], k.shape[2]
    t = np.asarray(bias, dtype=np.float64)
    out = np.zeros(t.shape, dtype=np.float64)
    varlen = seq_lens_q is not None or seq_lens_kv is not None or bottom_right
    for bi in range(b):
        mask = _batch_mask(s_q, s_kv, causal, bi, seq_lens_q, seq_lens_kv, bottom_right)
        off = _batch_off(s_q, s_kv, bi, seq_lens_q, seq_lens_kv, bottom_right)
        for hq in range(h_q):
            hk = kv_head_of(hq, h_q, h_kv)
            term = _bias_of(t, None, s_q, s_kv, bi, hq, off)
            _, _, _, dS = _head_backward(q[bi, hq], k[bi, hk], v[bi, hk], do[bi, hq], scale, mask,
                                         allow_empty=varlen, bias=term,
                                         zdrop=_zdrop(keep, dropout_p, bi, hq))
            out[bi if t.shape[0] > 1 else 0, hq if t.shape[1] > 1 else 0] += dS
    return out


def backward_ds_rows(q_rows, do_rows, rows: Sequence[int], kh, vh, scale: float, causal: bool,
                     bias: np.ndarray | None = None, zdrop: np.ndarray | None = None):
    """dS = P ∘ (dP − Delta) for selected query rows of one (batch, head): [n, s_kv] — the
    gradient of the scaled scores, and so of an additive bias on them.

    Row i needs only its own P_i, dP_i = Z_i ∘ (dO_i Vᵀ) and Delta_i = Σ_j P_ij dP_ij (Z the
    dropout factor zdrop of these rows, 1 without dropout), so the cost is O(n·s_kv·d)."""
    _, _, P = head_forward(q_rows, kh, vh, scale, _rows_mask(rows, kh.shape[0], causal), bias=bias)
    dP = do_rows @ vh.T
    if zdrop is not None:
        dP = zdrop * dP
    delta = (P * dP).sum(axis=1)
    return P * (dP - delta[:, None])


def backward_dq_rows(q_rows, do_rows, rows: Sequence[int], kh, vh, scale: float, causal: bool,
                     bias: np.ndarray | None = None, zdrop: np.ndarray | None = None):
    """dQ = scale · dS K for selected query rows of one (batch, head): [n, d] (bias and zdrop
    as in forward_rows)."""
    return scale * (backward_ds_rows(q_rows, do_rows, rows, kh, vh, scale, causal, bias, zdrop) @ kh)


def backward_kv_rows(q_rows, do_rows, rows: Sequence[int], kh, vh, scale: float, causal: bool,
                     bias: np.ndarray | None = None, zdrop: np.ndarray | None = None):
    """The contribution of selected query rows of one head to dK and dV: ([s_kv, d], [s_kv, d]).

    dK and dV of a KV head are the sums of these contributions over every query row of
    every query head in its group (bias and zdrop as in forward_rows)."""
    _, _, P = head_forward(q_rows, kh, vh, scale, _rows_mask(rows, kh.shape[0], causal), bias=bias)
    Z = 1.0 if zdrop is None else zdrop
    dV = (P * Z).T @ do_rows
    dP = Z * (do_rows @ vh.T)
    delta = (P * dP).sum(axis=1)
    dS = P * (dP - delta[:, None])
    dK = scale * (dS.T @ q_rows)
    return dK, dV


def backward_kv_head(q, k, v, do, scale: float, causal: bool, bi: int, hk: int,
                     row_chunk: int = 1024, bias_rows=None, zdrop_rows=None):
    """dK, dV of one (batch, KV head) at any size: [s_kv, d] each.

    Sums over the KV head's group of query heads, visiting query rows in chunks
    so that at most row_chunk x s_kv scores are held at a time.  bias_rows: optional
    function (hq, r0, r1) -> [r1 - r0, s_kv] fp64, the additive term on the scaled scores of
    query rows r0..r1-1 of head hq (a bias tensor's slice, or ALiBi's rows); zdrop_rows: the
    same for the dropout factor keep / (1 - p)."""
    b, h_q, s_q, _ = q.shape
    h_kv, s_kv = k.shape[1], k.shape[2]
    g = h_q // h_kv
    kh, vh = k[bi, hk], v[bi, hk]
    dK = np.zeros_like(kh, dtype=np.float64)
    dV = np.zeros_like(vh, dtype=np.float64)
    for hq in range(hk * g, (hk + 1) * g):
        for r0 in range(0, s_q, row_chunk):
            r1 = min(s_q, r0 + row_chunk)
            bias = None if bias_rows is None else bias_rows(hq, r0, r1)
            z = None if zdrop_rows is None else zdrop_rows(hq, r0, r1)
            gk, gv = backward_kv_rows(q[bi, hq, r0:r1], do[bi, hq, r0:r1], np.arange(r0, r1),
                                      kh, vh, scale, causal, bias, z)
            dK += gk
            dV += gv
    return dK, dV
