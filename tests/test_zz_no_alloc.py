"""sdpa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Such a caller (a plugin inside a framework that owns all device memory, or a loop that
must not call cudaMalloc because it can synchronise the device) passes only its inputs
and outputs; the scratch is a fixed array inside the library.  These tests call it through
the C ABI and check it against sdpa_bwd with a caller-allocated workspace, twice in a row,
because every call reuses the same array and must clear whatever the last call left.

This file is named to be collected last, so a run that stops at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

from sdpa_workloads import Workload, make_inputs, tiny
from sdpa_testlib import assert_grad_close, f64, guarded_empty_like, check_guard, lib, run_bwd, run_fwd


def _noalloc(w, dev_qkv, o, lse, do_dev):
    m = lib()
    q, k, v = dev_qkv
    dq, dqb = guarded_empty_like(q)
    dk, dkb = guarded_empty_like(k)
    dv, dvb = guarded_empty_like(v)
    p = m.make_problem(q, k, v, o, attn_scale=w.scale, causal=w.causal, dout=do_dev, dq=dq, dk=dk,
                       dv=dv)
    st = m.lib.sdpa_bwd_noalloc(ctypes.byref(p), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                o.data_ptr(), do_dev.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                                dk.data_ptr(), dv.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
    assert st == 0, m.sdpa_last_error_string()
    torch.cuda.synchronize()
    assert m.sdpa_device_error() == 0
    for b, n in ((dqb, "dQ"), (dkb, "dK"), (dvb, "dV")):
        check_guard(b, n)
    return dq, dk, dv


CASES = [
    tiny(True),
    Workload("t", 2, 4, 4, 333, 333, 128, "bf16", causal=False, backward=True),
    # few KV heads: the split path, whose fp32 dK/dV partials live in the scratch too
    Workload("t", 1, 8, 2, 700, 700, 64, "f16", causal=True, backward=True),
]


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=["tiny_causal", "bf16_d128", "split_groups"])
def test_noalloc_matches_workspace_entry_point_twice(w):
    x = make_inputs(w, seed=7, with_do=True)
    o, lse, dev = run_fwd(w, x)
    ref = run_bwd(w, dev, o, lse, x.do)
    do_dev = torch.empty_strided(x.do.shape, x.do.stride(), dtype=x.do.dtype, device="cuda")
    do_dev.copy_(x.do)
    for call in range(2):
        got = _noalloc(w, dev, o, lse, do_dev)
        for g, r, name in zip(got, ref, ("dQ", "dK", "dV")):
            assert_grad_close(f64(g), f64(r), f"{name} (call {call + 1})")


def test_noalloc_rejects_problems_beyond_its_scratch():
    """A problem whose workspace exceeds the built-in scratch is refused before anything runs
    (so this check needs no GPU)."""
    m = lib()
    p = m.Problem()
    p.b, p.h_q, p.h_kv, p.s_q, p.s_kv, p.d = 2, 16, 16, 8192, 8192, 128
    p.in_dtype = p.out_dtype = 1
    p.attn_scale = 0.088
    p.causal = 1
    st_q = m.Strides(16 * 8192 * 128, 8192 * 128, 128, 1)
    p.q = p.k = p.v = p.o = p.dout = p.dq = p.dk = p.dv = st_q
    need = m.sdpa_workspace_size(p, True)
    assert need > m.NOALLOC_SCRATCH_BYTES
    fake = 0x7F0000000000  # never dereferenced: the size check fails first
    st = m.lib.sdpa_bwd_noalloc(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake, fake,
                                fake, None)
    assert st == 2
    msg = m.sdpa_last_error_string()
    assert str(need) in msg and str(m.NOALLOC_SCRATCH_BYTES) in msg


def _refusal(p):
    """Calls sdpa_bwd_noalloc on a problem expected to be refused by its size check (fake
    addresses, never dereferenced: nothing runs before the check)."""
    m = lib()
    need = m.sdpa_workspace_size(p, True)
    assert need > m.NOALLOC_SCRATCH_BYTES
    fake = 0x7F0000000000
    st = m.lib.sdpa_bwd_noalloc(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake, fake,
                                fake, None)
    assert st == 2, m.sdpa_last_error_string()
    msg = m.sdpa_last_error_string()
    assert str(need) in msg and str(m.NOALLOC_SCRATCH_BYTES) in msg


def _plain_problem(m, b, h, s, d, dtype):
    p = m.Problem()
    p.b, p.h_q, p.h_kv, p.s_q, p.s_kv, p.d = b, h, h, s, s, d
    p.in_dtype = p.out_dtype = dtype
    p.attn_scale = d ** -0.5
    p.causal = 1
    st = m.Strides(h * s * d, s * d, d, 1)
    p.q = p.k = p.v = p.o = p.dout = p.dq = p.dk = p.dv = st
    return p


def test_noalloc_counts_the_fp8_copies():
    """An FP8 problem whose base scratch (dQ accumulator, row vectors) fits in the built-in
    array but whose widened 16-bit copies of Q, K, V and dO do not: refused with
    SDPA_ERR_UNSUPPORTED and the full size, not passed on to fail as a workspace error."""
    m = lib()
    p = _plain_problem(m, 1, 8, 4096, 128, m.DTYPE_BF16)
    p.in_dtype = m.DTYPE_E4M3
    p.out_dtype = m.DTYPE_BF16
    p.dout_dtype = m.DTYPE_E5M2
    p.descale_q = p.descale_k = p.descale_v = p.descale_do = 0x7F0000001000
    base = 8 * 4096 * 128 * 4 + 2 * 8 * 4096 * 4
    assert base < m.NOALLOC_SCRATCH_BYTES
    _refusal(p)


def test_noalloc_counts_the_bias_copy():
    """A bias problem whose transposed bias copy takes the workspace over the array's size."""
    m = lib()
    p = _plain_problem(m, 1, 4, 2048, 128, m.DTYPE_BF16)
    p.bias = 0x7F0000002000
    p.bias_strides = m.Strides(0, 2048 * 2048, 2048, 1)
    assert 4 * 2048 * 128 * 4 < m.NOALLOC_SCRATCH_BYTES
    _refusal(p)
    p.dbias = 0x7F0000003000
    p.dbias_strides = m.Strides(0, 2048 * 2048, 2048, 1)
    _refusal(p)


@pytest.mark.gpu
def test_noalloc_fp8_small_problem_against_the_oracle():
    """An FP8 backward pass (E4M3 Q, K, V; E5M2 dO) small enough for the built-in scratch,
    widened copies included: twice in a row against the fp64 oracle on the decoded inputs,
    with O and LSE from the oracle (the 16-bit tolerance applies)."""
    import numpy as np
    import oracle
    from sdpa_testlib import to_dev
    m = lib()
    w = Workload("t", 1, 4, 2, 384, 384, 128, "e4m3", causal=True, backward=True)
    x = make_inputs(w, seed=11, with_do=True)
    q64, k64, v64, do64 = (f64(x.q, x.descale_q), f64(x.k, x.descale_k), f64(x.v, x.descale_v),
                           f64(x.do, x.descale_do))
    O, L = oracle.forward(q64, k64, v64, w.scale, w.causal)
    dQ, dK, dV = oracle.backward(q64, k64, v64, do64, w.scale, w.causal)
    q, k, v, do = to_dev(x.q), to_dev(x.k), to_dev(x.v), to_dev(x.do)
    o = torch.empty(x.q.shape, dtype=torch.bfloat16, device="cuda")
    o.copy_(torch.from_numpy(O).to(torch.bfloat16))
    lse = torch.from_numpy(np.ascontiguousarray(L)).float().cuda()
    ds = {n: torch.tensor([getattr(x, "descale_" + n)], dtype=torch.float32, device="cuda")
          for n in ("q", "k", "v", "do")}
    for call in range(2):
        dq, dqb = guarded_empty_like(q, torch.bfloat16)
        dk, dkb = guarded_empty_like(k, torch.bfloat16)
        dv, dvb = guarded_empty_like(v, torch.bfloat16)
        p = m.make_problem(q, k, v, o, attn_scale=w.scale, causal=True, dout=do, dq=dq, dk=dk, dv=dv,
                           descale_q=ds["q"], descale_k=ds["k"], descale_v=ds["v"], descale_do=ds["do"])
        assert m.sdpa_workspace_size(p, True) <= m.NOALLOC_SCRATCH_BYTES
        st = m.lib.sdpa_bwd_noalloc(ctypes.byref(p), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                    o.data_ptr(), do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                                    dk.data_ptr(), dv.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == 0, m.sdpa_last_error_string()
        torch.cuda.synchronize()
        assert m.sdpa_device_error() == 0
        for b, n in ((dqb, "dQ"), (dkb, "dK"), (dvb, "dV")):
            check_guard(b, n)
        for g, r, n in ((dq, dQ, "dQ"), (dk, dK, "dK"), (dv, dV, "dV")):
            assert_grad_close(f64(g), r, f"{n} (call {call + 1})")
