"""Failure detection without a GPU fault: every wait inside the kernels is bounded, and a
wait that runs out makes its kernel give up cleanly (the other roles drop out, copies and
MMAs already issued are drained, tensor memory is freed) and report SDPA_ERR_TIMEOUT.

A child process shortens the bound to one SM cycle (SDPA_WAIT_LIMIT_CYCLES), so that every
wait not already satisfied at its first test gives up (the waits for the first tiles of a
normal problem do), and checks the status of the forward pass and of both backward kernels
(d = 128 and d = 256), of the forward pass with a bias tensor and of a forward pass on
persistent CTAs, under SDPA_DEBUG_SYNC.  It
then restores the default bound in the same process and checks that the same calls give
correct results: the context is still usable."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import os, sys
sys.path.insert(0, os.path.join(ROOT, "tests")); sys.path.insert(0, ROOT)
import numpy as np, torch
import attention_flashattention_sdpa_gb300 as m
import oracle
from sdpa_workloads import Workload, make_inputs
from sdpa_testlib import assert_fwd_close, assert_grad_close, f64, to_dev

def step(w, x):
    q, k, v, do = to_dev(x.q), to_dev(x.k), to_dev(x.v), to_dev(x.do)
    o = torch.empty_like(q)
    lse = torch.empty(w.b, w.h_q, w.s_q, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    p = m.make_problem(q, k, v, o, attn_scale=w.scale, causal=True, dout=do, dq=dq, dk=dk, dv=dv)
    ws = torch.empty(m.sdpa_workspace_size(p, True), dtype=torch.uint8, device="cuda")
    st = []
    for f in (lambda: m.sdpa_fwd(q, k, v, o, lse, attn_scale=w.scale, causal=True),
              lambda: m.sdpa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, attn_scale=w.scale, causal=True)):
        try:
            f()
            st.append(0)
        except m.SdpaError as e:
            st.append(e.status)
    torch.cuda.synchronize()
    return st, (o, lse, dq, dk, dv)

for d in (128, 256):
    w = Workload("t", 1, 4, 4, 1024, 1024, d, "bf16", causal=True, backward=True)
    x = make_inputs(w, seed=d, with_do=True)
    os.environ["SDPA_WAIT_LIMIT_CYCLES"] = "1"
    st, _ = step(w, x)
    assert st == [6, 6], f"d={d}: statuses {st}, want SDPA_ERR_TIMEOUT for both passes"
    assert "bounded device wait" in m.sdpa_last_error_string()
    assert m.sdpa_device_error() == 0, "the flag is reported once and then cleared"
    del os.environ["SDPA_WAIT_LIMIT_CYCLES"]
    st, (o, lse, dq, dk, dv) = step(w, x)
    assert st == [0, 0], f"d={d}: statuses {st} after restoring the bound"
    q64, k64, v64, do64 = f64(x.q), f64(x.k), f64(x.v), f64(x.do)
    O, L = oracle.forward(q64, k64, v64, w.scale, True)
    assert_fwd_close(f64(o), O)
    dQ, dK, dV = oracle.backward(q64, k64, v64, do64, w.scale, True)
    for g, r, n in ((dq, dQ, "dQ"), (dk, dK, "dK"), (dv, dV, "dV")):
        assert_grad_close(f64(g), r, n)
# Forward-only instances with waits of their own: TMA bias tiles (one Q tile per CTA) and
# persistent CTAs walking several work units (b4 h12 s1024 d64: 192 units on the SMs).
def fwd_only(w, x, bias=None):
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    o = torch.empty_like(q)
    lse = torch.empty(w.b, w.h_q, w.s_q, device="cuda")
    try:
        m.sdpa_fwd(q, k, v, o, lse, attn_scale=w.scale, causal=True, bias=bias)
        st = 0
    except m.SdpaError as e:
        st = e.status
    torch.cuda.synchronize()
    return st, o

g = torch.Generator().manual_seed(7)
wb = Workload("t", 2, 4, 4, 512, 512, 128, "bf16", causal=True)
bias = (2.0 * torch.randn(1, 4, 512, 512, generator=g)).to(torch.bfloat16)
wp = Workload("t", 4, 12, 12, 1024, 1024, 64, "f16", causal=True)
for w, b in ((wb, bias), (wp, None)):
    x = make_inputs(w, seed=w.d, with_do=False)
    bd = None if b is None else b.cuda()
    os.environ["SDPA_WAIT_LIMIT_CYCLES"] = "1"
    st, _ = fwd_only(w, x, bd)
    assert st == 6, f"forward {w.b}x{w.h_q}x{w.s_q}x{w.d}: status {st}, want SDPA_ERR_TIMEOUT"
    assert m.sdpa_device_error() == 0
    del os.environ["SDPA_WAIT_LIMIT_CYCLES"]
    st, o = fwd_only(w, x, bd)
    assert st == 0
    O, _ = oracle.forward(f64(x.q), f64(x.k), f64(x.v), w.scale, True,
                          bias=None if b is None else f64(b))
    assert_fwd_close(f64(o), O)
print("WAIT_TIMEOUT_OK")
'''


@pytest.mark.gpu
def test_waits_that_run_out_report_a_timeout_and_leave_the_context_usable():
    env = dict(os.environ, SDPA_DEBUG_SYNC="1")
    env.pop("SDPA_WAIT_LIMIT_CYCLES", None)
    r = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + CHILD], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "WAIT_TIMEOUT_OK" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]

