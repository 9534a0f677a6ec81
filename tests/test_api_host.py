"""Host-side checks of the C ABI: the library loads, exports every declared symbol, and
rejects bad arguments with the right status and message before launching anything.
No GPU is needed: validation runs before any CUDA call."""
import ctypes
import os
import re
import threading

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    import attention_flashattention_sdpa_gb300 as mod
    return mod


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "sdpa.h")).read()
    return sorted(set(re.findall(r"SDPA_API\s+[\w\s\*]+?\b(sdpa_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    syms = _declared_symbols()
    for name in ("sdpa_fwd", "sdpa_bwd", "sdpa_workspace_size", "sdpa_last_error_string"):
        assert name in syms


def test_library_exports_every_declared_symbol(m):
    L = ctypes.CDLL(m.LIB_PATH)
    for name in _declared_symbols():
        assert hasattr(L, name), f"{name} declared in include/sdpa.h but not exported"


def test_struct_layout_and_version(m):
    assert m.lib.sdpa_problem_struct_size() == ctypes.sizeof(m.Problem)
    assert m.sdpa_version() >= 100


def _problem(m, **over):
    if "bias_strides" in over:   # a tuple, or None for a zero (invalid) stride set
        bst = over.pop("bias_strides")
        over["bias_strides"] = m.Strides(*(bst or (0, 0, 0, 0)))
    elif "bias" in over:
        over["bias_strides"] = m.Strides(0, 128 * 128, 128, 1)
    p = m.Problem()
    p.b, p.h_q, p.h_kv, p.s_q, p.s_kv, p.d = 1, 2, 2, 128, 128, 64
    p.in_dtype = p.out_dtype = m.DTYPE_F16
    p.attn_scale = 0.125
    p.causal = 0
    st = m.Strides(2 * 128 * 64, 128 * 64, 64, 1)
    stk = m.Strides(2 * 128 * 64, 128 * 64, 64, 1)
    p.q = p.o = p.dout = p.dq = st
    p.k = p.v = p.dk = p.dv = stk
    for k, v in over.items():
        setattr(p, k, v)
    return p


# 16-byte aligned but not a real allocation.  Every call below fails host validation, so
# no kernel is ever launched on it (these tests must stay safe on a machine with a GPU).
FAKE = 0x7F0000000000


def _fwd(m, p, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None):
    return m.lib.sdpa_fwd(ctypes.byref(p), q, k, v, o, lse, None, 0, None)


def _bwd(m, p, ws=FAKE, ws_bytes=1 << 40, lse=FAKE, q=FAKE):
    return m.lib.sdpa_bwd(ctypes.byref(p), q, FAKE, FAKE, FAKE, FAKE, lse, FAKE, FAKE, FAKE, ws,
                          ws_bytes, None)


@pytest.mark.parametrize("over,status,msg", [
    (dict(d=96), 2, "head dim"),
    (dict(d=0), 1, "sizes"),
    (dict(s_q=0), 1, "sizes"),
    (dict(s_kv=0), 1, "sizes"),
    (dict(h_kv=3, h_q=4), 1, "multiple"),
    (dict(causal=3), 1, "causal"),
    (dict(causal=-1), 1, "causal"),
    (dict(attn_scale=float("nan")), 1, "finite"),
    (dict(in_dtype=7), 1, "in_dtype"),
    (dict(out_dtype=1), 2, "same dtype"),
    (dict(in_dtype=2, out_dtype=1, d=128), 1, "descale"),
    (dict(in_dtype=2, out_dtype=1), 2, "d = 128 or 256"),
    (dict(in_dtype=2, out_dtype=2), 2, "output"),
    (dict(alibi=2), 1, "alibi"),
    (dict(bias=FAKE + 8), 3, "bias"),
    (dict(bias=FAKE, alibi=1, causal=1), 2, "alibi"),
    (dict(alibi=1), 2, "ALiBi needs a causal mask"),
    (dict(alibi=1, causal=0, alibi_slopes=FAKE), 2, "ALiBi needs a causal mask"),
    (dict(bias=FAKE, bias_strides=None), 3, "key stride"),
    (dict(bias=FAKE, bias_strides=(0, 0, 130, 1)), 3, "multiples of 8"),
    (dict(bias=FAKE, bias_strides=(0, 0, 120, 1)), 3, "row stride"),
    (dict(dropout_p=-0.1), 1, "dropout_p"),
    (dict(dropout_p=1.0), 1, "dropout_p"),
    (dict(dropout_p=float("nan")), 1, "dropout_p"),
    (dict(dropout_p=0.1), 1, "dropout_mask"),
    (dict(dropout_p=0.1, dropout_mask=FAKE + 8), 3, "dropout_mask"),
    (dict(dropout_p=0.1, in_dtype=2, out_dtype=1, d=128, descale_q=FAKE, descale_k=FAKE,
          descale_v=FAKE), 2, "dropout"),
    (dict(alibi=1, alibi_slopes=FAKE + 2), 3, "alibi_slopes"),
    (dict(alibi=1, in_dtype=2, out_dtype=1, d=128, descale_q=FAKE, descale_k=FAKE,
          descale_v=FAKE), 2, "ALiBi"),
])
def test_forward_rejects_bad_problem(m, over, status, msg):
    assert _fwd(m, _problem(m, **over)) == status
    assert msg in m.sdpa_last_error_string()


def test_forward_rejects_bad_views(m):
    p = _problem(m)
    assert _fwd(m, p, q=None) == 1 and "q: null" in m.sdpa_last_error_string()
    assert _fwd(m, p, o=FAKE + 8) == 3 and "16-byte" in m.sdpa_last_error_string()
    bad = _problem(m)
    bad.q = m.Strides(2 * 128 * 64, 128 * 64, 64, 2)
    assert _fwd(m, bad) == 3 and "innermost" in m.sdpa_last_error_string()
    bad = _problem(m)
    bad.k = m.Strides(2 * 128 * 64, 128 * 64, 60, 1)
    assert _fwd(m, bad) == 3 and "multiple of 16" in m.sdpa_last_error_string()
    bad = _problem(m)
    bad.v = m.Strides(2 * 128 * 64, -64, 64, 1)
    assert _fwd(m, bad) == 3 and "positive" in m.sdpa_last_error_string()


def test_unit_dimension_strides_are_ignored(m):
    # b = 1: the batch stride is never used, so an odd value must not be rejected.
    # The call is stopped by a later check (a misaligned O) so nothing is launched; the
    # message names O, which shows Q's odd batch stride passed validation.
    p = _problem(m)
    p.q = m.Strides(3, 128 * 64, 64, 1)
    assert _fwd(m, p, o=FAKE + 8) == 3
    assert m.sdpa_last_error_string().startswith("o:")


def test_backward_rejections(m):
    fp8 = dict(in_dtype=2, out_dtype=1, descale_q=FAKE, descale_k=FAKE, descale_v=FAKE)
    assert _bwd(m, _problem(m, in_dtype=2, out_dtype=1)) == 1
    assert "descale" in m.sdpa_last_error_string()
    assert _bwd(m, _problem(m, dout_dtype=1, descale_do=FAKE, **fp8)) == 2
    assert "dout_dtype" in m.sdpa_last_error_string()
    assert _bwd(m, _problem(m, dout_dtype=3, **fp8)) == 1 and "descale_do" in m.sdpa_last_error_string()
    assert _bwd(m, _problem(m, in_dtype=3, out_dtype=1)) == 2 and "E5M2" in m.sdpa_last_error_string()
    # a valid FP8 problem is stopped by its workspace size (it needs room for the widened copies)
    ok8 = _problem(m, dout_dtype=3, descale_do=FAKE, **fp8)
    need8 = m.sdpa_workspace_size(ok8, True)
    assert need8 == m.sdpa_workspace_size(_problem(m, in_dtype=1, out_dtype=1), True) + 4 * 2 * 128 * 64 * 2
    assert _bwd(m, ok8, ws_bytes=need8 - 1) == 4
    assert _bwd(m, _problem(m, d=200)) == 2
    assert _bwd(m, _problem(m), lse=None) == 1 and "lse" in m.sdpa_last_error_string()
    assert _bwd(m, _problem(m), ws=None) == 4 and "workspace" in m.sdpa_last_error_string()
    assert _bwd(m, _problem(m), ws_bytes=100) == 4
    assert _bwd(m, _problem(m), ws=FAKE + 16) == 4 and "256-byte" in m.sdpa_last_error_string()
    assert _bwd(m, _problem(m), q=None) == 1


def test_workspace_size(m):
    p = _problem(m)
    assert m.sdpa_workspace_size(p, False) == 0
    n = m.sdpa_workspace_size(p, True)
    # fp32 dQ accumulator + Delta + LSE*log2(e), rows padded to 128, each 256-aligned
    assert n >= 1 * 2 * 128 * 64 * 4 + 2 * 1 * 2 * 128 * 4
    p2 = _problem(m, s_q=129)
    assert m.sdpa_workspace_size(p2, True) >= 1 * 2 * 256 * 64 * 4
    with pytest.raises(m.SdpaError) as e:
        m.sdpa_workspace_size(_problem(m, d=100), True)
    assert e.value.status == 2


def test_last_error_is_thread_local(m):
    assert _fwd(m, _problem(m, d=96)) == 2
    seen = []
    t = threading.Thread(target=lambda: seen.append(m.sdpa_last_error_string()))
    t.start()
    t.join()
    assert seen == [""]
    assert "head dim" in m.sdpa_last_error_string()


def test_null_problem(m):
    assert m.lib.sdpa_fwd(None, FAKE, FAKE, FAKE, FAKE, None, None, 0, None) == 1
    n = ctypes.c_size_t()
    assert m.lib.sdpa_workspace_size(None, 0, ctypes.byref(n)) == 1


def test_dropout_mask_sizes_and_validation(m):
    assert m.sdpa_dropout_mask_size(2, 3, 200, 300) == (2 * 3 * 200 * 12 * 4, 2 * 3 * 300 * 8 * 4)
    assert m.sdpa_dropout_mask_size(1, 1, 1, 1) == (16, 16)
    p = _problem(m, dropout_p=1.5)
    assert m.lib.sdpa_dropout_mask(ctypes.byref(p), 1, 2, FAKE, FAKE, None) == 1
    assert "dropout_p" in m.sdpa_last_error_string()
    p = _problem(m, dropout_p=0.5)
    assert m.lib.sdpa_dropout_mask(ctypes.byref(p), 1, 2, FAKE + 4, None, None) == 3
    p = _problem(m, b=300, h_q=300, h_kv=300, dropout_p=0.5)
    assert m.lib.sdpa_dropout_mask(ctypes.byref(p), 1, 2, FAKE, FAKE, None) == 2


def test_backward_dropout_needs_the_transposed_mask(m):
    p = _problem(m, dropout_p=0.2, dropout_mask=FAKE)
    assert _bwd(m, p) == 1 and "dropout_mask_t" in m.sdpa_last_error_string()


def test_bias_workspace_holds_a_transposed_copy(m):
    base = m.sdpa_workspace_size(_problem(m), True)
    with_bias = m.sdpa_workspace_size(_problem(m, bias=FAKE), True)   # [1, h_q, 128, 128] bf16
    assert with_bias - base == 2 * 128 * 128 * 2
    assert m.sdpa_workspace_size(_problem(m, bias=FAKE), False) == 0


def test_bias_gradient_validation_and_workspace(m):
    st = m.Strides(0, 128 * 128, 128, 1)
    p = _problem(m, dbias=FAKE, dbias_strides=(0, 128 * 128, 128, 1))
    assert _bwd(m, p) == 1 and "needs a bias" in m.sdpa_last_error_string()
    p = _problem(m, bias=FAKE, dbias=FAKE + 8, dbias_strides=(0, 128 * 128, 128, 1))
    p.bias_strides = st
    assert _bwd(m, p) == 3 and "dbias must be 16-byte" in m.sdpa_last_error_string()
    p = _problem(m, bias=FAKE, dbias=FAKE, dbias_strides=(2 * 128 * 128, 128 * 128, 128, 1))
    p.bias_strides = st
    assert _bwd(m, p) == 3 and "same dimensions" in m.sdpa_last_error_string()
    base = m.sdpa_workspace_size(_problem(m, bias=FAKE), True)
    p = _problem(m, bias=FAKE, dbias=FAKE, dbias_strides=(0, 128 * 128, 128, 1))
    p.bias_strides = st
    assert m.sdpa_workspace_size(p, True) - base == 2 * 128 * 128 * 4


def _problem_by_fields(m, q, k, v, o, causal, scale, dout=None, dq=None, dk=None, dv=None, descale=None,
                       lens=None, alibi=None, drop=None, bias=None, dbias=None):
    """Field-by-field construction of the sdpa_problem_t that make_problem must produce."""
    P = m.Problem()
    P.b, P.h_q, P.s_q, P.d = q.shape
    P.h_kv, P.s_kv = k.shape[1], k.shape[2]
    P.in_dtype = m.dtype_code(q)
    P.out_dtype = m.dtype_code(o) if o is not None else (
        m.DTYPE_BF16 if P.in_dtype == m.DTYPE_E4M3 else P.in_dtype)
    P.attn_scale = scale
    P.causal = m.causal_code(causal)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv)):
        setattr(P, name, m.Strides(*(t.stride() if t is not None else (0, 0, 0, 1))))
    if descale is not None:
        P.descale_q, P.descale_k, P.descale_v = (descale.data_ptr() + 4 * i for i in range(3))
        P.descale_do = descale.data_ptr() + 12
    if lens is not None:
        P.seq_lens_q, P.seq_lens_kv = lens[0].data_ptr(), lens[1].data_ptr()
    if alibi is not None:
        P.alibi, P.alibi_slopes = 1, alibi.data_ptr()
    if drop is not None:
        P.dropout_p, P.dropout_mask, P.dropout_mask_t = drop[0], drop[1].data_ptr(), drop[2].data_ptr()
    P.dout_dtype = m.dtype_code(dout) if dout is not None else P.in_dtype
    for t, pf, sf in ((bias, "bias", "bias_strides"), (dbias, "dbias", "dbias_strides")):
        if t is not None:
            st = list(t.stride())
            st[0] = 0 if t.shape[0] == 1 else st[0]
            st[1] = 0 if t.shape[1] == 1 else st[1]
            setattr(P, pf, t.data_ptr())
            setattr(P, sf, m.Strides(*st))
    return P


@pytest.mark.parametrize("seed", range(24))
def test_make_problem_matches_field_by_field_struct(m, seed):
    """make_problem packs the whole struct at once; every byte must equal the struct that
    assigning each field through ctypes gives (CPU tensors: only shapes, strides, dtypes and
    addresses are read)."""
    import random
    import torch
    rnd = random.Random(seed)
    dts = [torch.float16, torch.bfloat16, torch.float8_e4m3fn]
    dt = rnd.choice(dts)
    b, h_kv = rnd.randint(1, 3), rnd.randint(1, 3)
    h_q, s_q, s_kv, d = h_kv * rnd.choice([1, 2, 4]), rnd.randint(1, 300), rnd.randint(1, 300), rnd.choice([64, 128, 256])

    def t4(h, s):
        if rnd.random() < 0.5:
            return torch.empty(b, h, s, d, dtype=dt)
        return torch.empty(b, s, h, d, dtype=dt).permute(0, 2, 1, 3)   # BSHD view
    q, k, v = t4(h_q, s_q), t4(h_kv, s_kv), t4(h_kv, s_kv)
    o = None if (dt == torch.float8_e4m3fn and rnd.random() < 0.5) else \
        torch.empty(b, h_q, s_q, d, dtype=torch.bfloat16 if dt == torch.float8_e4m3fn else dt)
    causal = rnd.choice([False, True, "bottom_right"])
    scale = rnd.choice([None, 0.3])
    kw, ref = {}, {}
    if rnd.random() < 0.5:
        kw.update(dout=torch.empty_like(q), dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v))
        ref.update(kw)
    if dt == torch.float8_e4m3fn:
        ds = torch.ones(4)
        kw.update(descale_q=ds[0:1], descale_k=ds[1:2], descale_v=ds[2:3], descale_do=ds[3:4])
        ref["descale"] = ds
    if rnd.random() < 0.4:
        lq, lkv = torch.zeros(b, dtype=torch.int32), torch.zeros(b, dtype=torch.int32)
        kw.update(seq_lens_q=lq, seq_lens_kv=lkv)
        ref["lens"] = (lq, lkv)
    if rnd.random() < 0.3:
        sl = torch.ones(h_q)
        kw["alibi_slopes"] = sl
        ref["alibi"] = sl
    if rnd.random() < 0.3:
        mk, mt = torch.zeros(8, dtype=torch.int32), torch.zeros(8, dtype=torch.int32)
        kw.update(dropout_p=0.25, dropout_mask=mk, dropout_mask_t=mt)
        ref["drop"] = (0.25, mk, mt)
    if rnd.random() < 0.4:
        bias = torch.empty(rnd.choice([1, b]), rnd.choice([1, h_q]), s_q, s_kv, dtype=torch.float16)
        kw["bias"] = ref["bias"] = bias
        if rnd.random() < 0.5:
            kw["dbias"] = ref["dbias"] = torch.empty_like(bias)
    got = m.make_problem(q, k, v, o, attn_scale=scale, causal=causal, **kw)
    want = _problem_by_fields(m, q, k, v, o, causal, (1.0 / d ** 0.5) if scale is None else scale, **ref)
    assert bytes(got) == bytes(want)


def test_make_problem_rejects_non_4d(m):
    import torch
    k = torch.empty(2, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        m.make_problem(torch.empty(1, 2, 8, 64, dtype=torch.float16), k, k, None)
