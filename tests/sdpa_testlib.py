"""Shared helpers for the SDPA tests: run the CUDA path through the C ABI and compare it
with the fp64 oracle.  Test-only code (it imports the oracle)."""
from __future__ import annotations

import math
from typing import Optional

import numpy as np
import torch

import oracle
from sdpa_workloads import Inputs, Workload, make_inputs

# Tolerances of the method (forward fp16/bf16, LSE, gradients, FP8 forward).
FWD_MAX_ABS = 2e-2
FWD_MEAN_ABS = 2e-3
LSE_ABS = 1e-3
GRAD_REL_L2 = 1e-2
FP8_REL_L2 = 6e-2

SENTINEL = -12288.0  # exactly representable in fp16, bf16 and fp32
PAD = 4096  # guard-band elements before and after every output buffer


def lib():
    import attention_flashattention_sdpa_gb300 as m
    return m


def guarded_empty_like(t: torch.Tensor, dtype=None):
    """An uninitialised tensor with t's shape and strides, inside a buffer whose PAD
    elements on each side hold SENTINEL (checked by check_guard)."""
    dtype = dtype or t.dtype
    span = 1 + sum((n - 1) * s for n, s in zip(t.shape, t.stride()))
    buf = torch.full((span + 2 * PAD,), SENTINEL, dtype=dtype, device="cuda")
    out = buf.as_strided(t.shape, t.stride(), PAD)
    out.fill_(float("nan"))
    return out, buf


def check_guard(buf: torch.Tensor, name: str):
    head = buf[:PAD].float().cpu()
    tail = buf[-PAD:].float().cpu()
    assert (head == SENTINEL).all() and (tail == SENTINEL).all(), f"{name}: write outside the tensor"


def to_dev(t: torch.Tensor) -> torch.Tensor:
    """Copy to the GPU keeping the (possibly BSHD-permuted) strides."""
    out = torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, device="cuda")
    out.copy_(t)
    return out


def f64(t: torch.Tensor, descale: float = 1.0) -> np.ndarray:
    return oracle.to_f64(t.cpu(), descale)


def _alibi_kwargs(alibi) -> dict:
    """None: off; "default": the library's geometric slopes; a sequence: per-head slopes."""
    if alibi is None:
        return {}
    if isinstance(alibi, str):
        assert alibi == "default"
        return {"alibi": True}
    return {"alibi_slopes": torch.tensor(list(alibi), dtype=torch.float32, device="cuda")}


def dropout_masks(b, h_q, s_q, s_kv, dropout, causal=False):
    """(row-major, transposed) keep-bit tensors drawn by the library for dropout = (p, seed,
    offset), or (None, None); with `causal` the tiles above the diagonal stay unwritten (-1)."""
    if dropout is None:
        return None, None
    m = lib()
    n, n_t = m.sdpa_dropout_mask_size(b, h_q, s_q, s_kv)
    mask = torch.full((n // 4,), -1, dtype=torch.int32, device="cuda")
    mask_t = torch.full((n_t // 4,), -1, dtype=torch.int32, device="cuda")
    m.sdpa_dropout_mask(b, h_q, s_q, s_kv, dropout[0], dropout[1], dropout[2], mask, mask_t,
                        causal=causal)
    return mask, mask_t


def run_fwd(w: Workload, x: Inputs, with_lse: bool = True, out_dtype=torch.bfloat16,
            causal=None, seq_lens_q=None, seq_lens_kv=None, alibi=None, dropout=None, bias=None):
    m = lib()
    causal = w.causal if causal is None else causal
    lens = _alibi_kwargs(alibi)
    if bias is not None:
        lens["bias"] = bias
    if dropout is not None:
        lens["dropout_p"] = dropout[0]
        # a causal draw (tiles above the diagonal unwritten) when no lengths are given
        dc = causal if seq_lens_q is None and seq_lens_kv is None else False
        lens["dropout_mask"] = dropout_masks(w.b, w.h_q, w.s_q, w.s_kv, dropout, dc)[0]
    if seq_lens_q is not None:
        lens["seq_lens_q"] = torch.tensor(seq_lens_q, dtype=torch.int32, device="cuda")
    if seq_lens_kv is not None:
        lens["seq_lens_kv"] = torch.tensor(seq_lens_kv, dtype=torch.int32, device="cuda")
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    odt = out_dtype if w.dtype == "e4m3" else q.dtype
    o, obuf = guarded_empty_like(q, odt)
    lse = lbuf = None
    if with_lse:
        lse, lbuf = guarded_empty_like(torch.empty(w.b, w.h_q, w.s_q), torch.float32)
    kw = {}
    if w.dtype == "e4m3":
        kw = dict(descale_q=torch.tensor([x.descale_q], device="cuda"),
                  descale_k=torch.tensor([x.descale_k], device="cuda"),
                  descale_v=torch.tensor([x.descale_v], device="cuda"))
    m.sdpa_fwd(q, k, v, o, lse, attn_scale=w.scale, causal=causal, **kw, **lens)
    torch.cuda.synchronize()
    assert m.sdpa_device_error() == 0
    check_guard(obuf, "O")
    if lbuf is not None:
        check_guard(lbuf, "LSE")
    return o, lse, (q, k, v)


def run_bwd(w: Workload, dev_qkv, o, lse, do_cpu: torch.Tensor, causal=None, seq_lens_q=None,
            seq_lens_kv=None, alibi=None, dropout=None, bias=None, dbias=None):
    m = lib()
    causal = w.causal if causal is None else causal
    lens = _alibi_kwargs(alibi)
    if bias is not None:
        lens["bias"] = bias
    if dbias is not None:
        lens["dbias"] = dbias
    if dropout is not None:
        lens["dropout_p"] = dropout[0]
        dc = causal if seq_lens_q is None and seq_lens_kv is None else False
        lens["dropout_mask_t"] = dropout_masks(w.b, w.h_q, w.s_q, w.s_kv, dropout, dc)[1]
    if seq_lens_q is not None:
        lens["seq_lens_q"] = torch.tensor(seq_lens_q, dtype=torch.int32, device="cuda")
    if seq_lens_kv is not None:
        lens["seq_lens_kv"] = torch.tensor(seq_lens_kv, dtype=torch.int32, device="cuda")
    q, k, v = dev_qkv
    do = to_dev(do_cpu)
    dq, dqb = guarded_empty_like(q)
    dk, dkb = guarded_empty_like(k)
    dv, dvb = guarded_empty_like(v)
    p = m.make_problem(q, k, v, o, attn_scale=w.scale, causal=causal, dout=do, dq=dq, dk=dk, dv=dv,
                       bias=bias, dbias=dbias)
    ws = torch.empty(m.sdpa_workspace_size(p, True), dtype=torch.uint8, device="cuda")
    ws.fill_(0xAB)  # contents on entry must not matter
    m.sdpa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, attn_scale=w.scale, causal=causal, **lens)
    torch.cuda.synchronize()
    assert m.sdpa_device_error() == 0
    for b, n in ((dqb, "dQ"), (dkb, "dK"), (dvb, "dV")):
        check_guard(b, n)
    return dq, dk, dv


def rel_l2(got: np.ndarray, want: np.ndarray) -> float:
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))


def assert_fwd_close(o_gpu: np.ndarray, o_ref: np.ndarray, what: str = "O"):
    err = np.abs(o_gpu - o_ref)
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite values"
    assert err.max() <= FWD_MAX_ABS, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= FWD_MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"


def assert_lse_close(l_gpu: np.ndarray, l_ref: np.ndarray):
    err = np.abs(l_gpu - l_ref)
    assert np.isfinite(l_gpu).all(), "LSE: non-finite values"
    assert err.max() <= LSE_ABS, f"LSE: max abs err {err.max():.3e}"


# When the exact gradient is identically zero (e.g. dQ with a single key: P = 1 whatever
# Q is), a relative error is undefined; the result must then be zero up to fp32 residue.
ZERO_GRAD_ABS = 1e-4


def assert_grad_close(g_gpu: np.ndarray, g_ref: np.ndarray, what: str, zero_tol: float = ZERO_GRAD_ABS):
    """Relative L2 within GRAD_REL_L2; where the exact gradient is identically zero, every
    entry within zero_tol (the caller may pass a bound derived from its inputs)."""
    assert np.isfinite(g_gpu).all(), f"{what}: non-finite values"
    if np.abs(g_ref).max() == 0.0:
        assert np.abs(g_gpu).max() <= zero_tol, f"{what}: should vanish, max {np.abs(g_gpu).max():.3e}"
        return
    e = rel_l2(g_gpu, g_ref)
    assert e <= GRAD_REL_L2, f"{what}: rel-L2 {e:.3e}"


def run_bwd_fp8(w: Workload, x: Inputs, o, lse, out_dtype=torch.bfloat16):
    """FP8 backward pass (E4M3 Q, K, V with their descales; dO in x.do's FP8 format with
    x.descale_do) through the C ABI, gradients in out_dtype."""
    m = lib()
    q, k, v, do = to_dev(x.q), to_dev(x.k), to_dev(x.v), to_dev(x.do)
    ds = {n: torch.tensor([getattr(x, "descale_" + n)], dtype=torch.float32, device="cuda")
          for n in ("q", "k", "v", "do")}
    dq, dqb = guarded_empty_like(q, out_dtype)
    dk, dkb = guarded_empty_like(k, out_dtype)
    dv, dvb = guarded_empty_like(v, out_dtype)
    p = m.make_problem(q, k, v, o, attn_scale=w.scale, causal=w.causal, dout=do, dq=dq, dk=dk, dv=dv,
                       descale_q=ds["q"], descale_k=ds["k"], descale_v=ds["v"], descale_do=ds["do"])
    ws = torch.empty(m.sdpa_workspace_size(p, True), dtype=torch.uint8, device="cuda")
    ws.fill_(0xAB)
    m.sdpa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, attn_scale=w.scale, causal=w.causal,
               descale_q=ds["q"], descale_k=ds["k"], descale_v=ds["v"], descale_do=ds["do"])
    torch.cuda.synchronize()
    assert m.sdpa_device_error() == 0
    for b, n in ((dqb, "dQ"), (dkb, "dK"), (dvb, "dV")):
        check_guard(b, n)
    return dq, dk, dv
