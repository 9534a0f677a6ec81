"""Python binding of the GB300 fused SDPA library (``include/sdpa.h``).

Argument marshalling only: every step of the attention computation runs in the CUDA
kernels of ``libsdpa_gb300.so``.  PyTorch supplies device memory and the current stream.
The binding keeps the C names: :func:`sdpa_fwd`, :func:`sdpa_bwd`,
:func:`sdpa_workspace_size`, :func:`sdpa_last_error_string`, :func:`sdpa_device_error`.

Importing this package loads the library and raises ``ImportError`` if it has not been
built (``python -m attention_flashattention_sdpa_gb300._build``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import struct
from typing import Optional

__all__ = [
    "SdpaError", "Strides", "Problem", "lib", "LIB_PATH", "dtype_code", "make_problem",
    "sdpa_workspace_size", "sdpa_fwd", "sdpa_bwd", "sdpa_last_error_string", "causal_code",
    "sdpa_device_error", "sdpa_version", "sdpa_bwd_noalloc", "NOALLOC_SCRATCH_BYTES", "STATUS",
    "sdpa_dropout_mask_size", "sdpa_dropout_mask",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsdpa_gb300.so")

STATUS = {0: "SDPA_OK", 1: "SDPA_ERR_INVALID_ARG", 2: "SDPA_ERR_UNSUPPORTED",
          3: "SDPA_ERR_LAYOUT", 4: "SDPA_ERR_WORKSPACE", 5: "SDPA_ERR_CUDA",
          6: "SDPA_ERR_TIMEOUT"}

DTYPE_F16, DTYPE_BF16, DTYPE_E4M3, DTYPE_E5M2 = 0, 1, 2, 3


class SdpaError(RuntimeError):
    """A non-OK status from the library; ``status`` holds the code."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class Strides(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("h", ctypes.c_int64), ("s", ctypes.c_int64),
                ("d", ctypes.c_int64)]


class Problem(ctypes.Structure):
    _fields_ = [
        ("b", ctypes.c_int32), ("h_q", ctypes.c_int32), ("h_kv", ctypes.c_int32),
        ("s_q", ctypes.c_int32), ("s_kv", ctypes.c_int32), ("d", ctypes.c_int32),
        ("in_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
        ("attn_scale", ctypes.c_float), ("causal", ctypes.c_int32),
        ("q", Strides), ("k", Strides), ("v", Strides), ("o", Strides),
        ("dout", Strides), ("dq", Strides), ("dk", Strides), ("dv", Strides),
        ("descale_q", ctypes.c_void_p), ("descale_k", ctypes.c_void_p),
        ("descale_v", ctypes.c_void_p),
        ("seq_lens_q", ctypes.c_void_p), ("seq_lens_kv", ctypes.c_void_p),
        ("alibi", ctypes.c_int32), ("alibi_slopes", ctypes.c_void_p),
        ("dropout_p", ctypes.c_float), ("dropout_mask", ctypes.c_void_p),
        ("dropout_mask_t", ctypes.c_void_p),
        ("dout_dtype", ctypes.c_int32), ("descale_do", ctypes.c_void_p),
        ("bias", ctypes.c_void_p), ("bias_strides", Strides),
        ("dbias", ctypes.c_void_p), ("dbias_strides", Strides),
    ]


def _packer():
    """One struct.Struct that lays out a whole Problem at the offsets ctypes gives it, so
    that a problem is marshalled by a single pack instead of one ctypes assignment per field."""
    fmt, pos = ["="], 0
    codes = {ctypes.c_int32: "i", ctypes.c_float: "f", ctypes.c_void_p: "Q"}
    for name, typ in Problem._fields_:
        off = getattr(Problem, name).offset
        fmt.append("x" * (off - pos))
        if typ is Strides:
            fmt.append("qqqq")
        else:
            fmt.append(codes[typ])
        pos = off + ctypes.sizeof(typ)
    fmt.append("x" * (ctypes.sizeof(Problem) - pos))
    st = struct.Struct("".join(fmt))
    assert st.size == ctypes.sizeof(Problem)
    return st


_PACK = _packer()
_NO_STRIDES = (0, 0, 0, 1)


def causal_code(causal) -> int:
    """False/0: no mask; True/1/"top_left": top-left causal; 2/"bottom_right": bottom-right."""
    if causal in (False, None, 0):
        return 0
    if causal in (True, 1, "top_left"):
        return 1
    if causal in (2, "bottom_right"):
        return 2
    raise ValueError(f"unknown causal mode {causal!r}")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m attention_flashattention_sdpa_gb300._build` (nvcc, sm_103a)")
    L = ctypes.CDLL(LIB_PATH)
    P, VP, SZ = ctypes.POINTER(Problem), ctypes.c_void_p, ctypes.c_size_t
    L.sdpa_workspace_size.argtypes = [P, ctypes.c_int, ctypes.POINTER(SZ)]
    L.sdpa_workspace_size.restype = ctypes.c_int
    L.sdpa_fwd.argtypes = [P, VP, VP, VP, VP, VP, VP, SZ, VP]
    L.sdpa_fwd.restype = ctypes.c_int
    L.sdpa_bwd.argtypes = [P, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, SZ, VP]
    L.sdpa_bwd.restype = ctypes.c_int
    L.sdpa_bwd_noalloc.argtypes = [P, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP]
    L.sdpa_bwd_noalloc.restype = ctypes.c_int
    L.sdpa_dropout_mask_size.argtypes = [P, ctypes.POINTER(SZ), ctypes.POINTER(SZ)]
    L.sdpa_dropout_mask_size.restype = ctypes.c_int
    L.sdpa_dropout_mask.argtypes = [P, ctypes.c_uint64, ctypes.c_uint64, VP, VP, VP]
    L.sdpa_dropout_mask.restype = ctypes.c_int
    L.sdpa_last_error_string.argtypes = []
    L.sdpa_last_error_string.restype = ctypes.c_char_p
    L.sdpa_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.sdpa_device_error.restype = ctypes.c_int
    L.sdpa_version.argtypes = []
    L.sdpa_version.restype = ctypes.c_int
    L.sdpa_problem_struct_size.argtypes = []
    L.sdpa_problem_struct_size.restype = SZ
    if L.sdpa_problem_struct_size() != ctypes.sizeof(Problem):
        raise ImportError("sdpa_problem_t layout mismatch between the library and the binding")
    return L


lib = _load()


def sdpa_last_error_string() -> str:
    return lib.sdpa_last_error_string().decode()


def sdpa_version() -> int:
    return lib.sdpa_version()


def _check(status: int):
    if status != 0:
        raise SdpaError(status, sdpa_last_error_string())


_DTYPES = {}


def dtype_code(t) -> int:
    if not _DTYPES:
        import torch
        _DTYPES.update({torch.float16: DTYPE_F16, torch.bfloat16: DTYPE_BF16,
                        torch.float8_e4m3fn: DTYPE_E4M3, torch.float8_e5m2: DTYPE_E5M2})
    return _DTYPES[t.dtype]


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _st4(t):
    if t is None:
        return _NO_STRIDES
    if t.dim() != 4:
        raise ValueError("tensors are logical [b, h, s, d] views")
    return t.stride()


def _bst(t):
    """Strides of a [b|1, h|1, s_q, s_kv] bias view; size-1 batch/head dims broadcast."""
    if t is None:
        return (0, 0, 0, 0)
    st = list(t.stride())
    if t.shape[0] == 1:
        st[0] = 0
    if t.shape[1] == 1:
        st[1] = 0
    return st


def _p0(t) -> int:
    return 0 if t is None else t.data_ptr()


def make_problem(q, k, v, o=None, *, attn_scale: Optional[float] = None, causal=False,
                 dout=None, dq=None, dk=None, dv=None, descale_q=None, descale_k=None,
                 descale_v=None, seq_lens_q=None, seq_lens_kv=None, alibi=False,
                 alibi_slopes=None, dropout_p: float = 0.0, dropout_mask=None,
                 dropout_mask_t=None, descale_do=None, bias=None, dbias=None) -> Problem:
    """Fills an sdpa_problem_t from logical [b, h, s, d] torch tensors (no copies).

    ALiBi is on when ``alibi`` is true or ``alibi_slopes`` (fp32 CUDA tensor of h_q slopes)
    is given; without slopes the library uses 2^(-8 (h + 1) / h_q)."""
    b, h_q, s_q, d = q.shape
    h_kv, s_kv = k.shape[1], k.shape[2]
    in_dt = dtype_code(q)
    if o is not None:
        out_dt = dtype_code(o)
    else:
        out_dt = DTYPE_BF16 if in_dt == DTYPE_E4M3 else in_dt
    scale = (1.0 / math.sqrt(d)) if attn_scale is None else float(attn_scale)
    return Problem.from_buffer_copy(_PACK.pack(
        b, h_q, h_kv, s_q, s_kv, d, in_dt, out_dt, scale, causal_code(causal),
        *_st4(q), *_st4(k), *_st4(v), *_st4(o), *_st4(dout), *_st4(dq), *_st4(dk), *_st4(dv),
        _p0(descale_q), _p0(descale_k), _p0(descale_v), _p0(seq_lens_q), _p0(seq_lens_kv),
        1 if (alibi or alibi_slopes is not None) else 0, _p0(alibi_slopes),
        float(dropout_p), _p0(dropout_mask), _p0(dropout_mask_t),
        dtype_code(dout) if dout is not None else in_dt, _p0(descale_do),
        _p0(bias), *_bst(bias), _p0(dbias), *_bst(dbias)))


_RAW_STREAM = None


def _stream(stream, like=None) -> int:
    """The cudaStream_t to launch on: ``stream`` if given, else PyTorch's current stream on the
    device of tensor ``like`` (read through torch's raw accessor when it has one: a few µs
    cheaper per call than building a Stream object)."""
    global _RAW_STREAM
    if stream is not None:
        return int(stream)
    import torch
    if _RAW_STREAM is None:
        _RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", False)
    if _RAW_STREAM and like is not None and like.device.index is not None:
        return _RAW_STREAM(like.device.index)
    return torch.cuda.current_stream().cuda_stream


def sdpa_workspace_size(problem: Problem, is_backward: bool) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.sdpa_workspace_size(ctypes.byref(problem), 1 if is_backward else 0, ctypes.byref(n)))
    return n.value


def sdpa_fwd(q, k, v, o, lse=None, *, attn_scale: Optional[float] = None, causal=False,
             descale_q=None, descale_k=None, descale_v=None, workspace=None, stream=None,
             seq_lens_q=None, seq_lens_kv=None, alibi=False, alibi_slopes=None,
             dropout_p: float = 0.0, dropout_mask=None, bias=None) -> None:
    """O (and LSE when ``lse`` is given: fp32 [b, h_q, s_q] contiguous) from Q, K, V.

    seq_lens_q / seq_lens_kv: optional int32 CUDA tensors of b valid lengths.
    alibi / alibi_slopes: the linear position bias (see :func:`make_problem`).
    dropout_p / dropout_mask: dropout with the row-major keep bits of :func:`sdpa_dropout_mask`."""
    p = make_problem(q, k, v, o, attn_scale=attn_scale, causal=causal, descale_q=descale_q,
                     descale_k=descale_k, descale_v=descale_v, seq_lens_q=seq_lens_q,
                     seq_lens_kv=seq_lens_kv, alibi=alibi, alibi_slopes=alibi_slopes,
                     dropout_p=dropout_p, dropout_mask=dropout_mask, bias=bias)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.sdpa_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                        _ptr(workspace), ws_bytes, _stream(stream, q)))


def sdpa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, *, attn_scale: Optional[float] = None,
             causal=False, stream=None, seq_lens_q=None, seq_lens_kv=None, alibi=False,
             alibi_slopes=None, dropout_p: float = 0.0, dropout_mask_t=None, descale_q=None,
             descale_k=None, descale_v=None, descale_do=None, bias=None, dbias=None) -> None:
    """dQ, dK, dV (overwritten) for the incoming gradient ``dout``; the masking, lengths,
    ALiBi and dropout options must be those of the forward call that produced ``o`` and
    ``lse`` (dropout_mask_t: the transposed keep bits of the same draw).  FP8: E4M3 q, k, v
    and an E5M2 (or E4M3) dout with their fp32 CUDA descales; o, dq, dk, dv in BF16/F16."""
    p = make_problem(q, k, v, o, attn_scale=attn_scale, causal=causal, dout=dout, dq=dq, dk=dk,
                     dv=dv, seq_lens_q=seq_lens_q, seq_lens_kv=seq_lens_kv, alibi=alibi,
                     alibi_slopes=alibi_slopes, dropout_p=dropout_p, dropout_mask_t=dropout_mask_t,
                     descale_q=descale_q, descale_k=descale_k, descale_v=descale_v,
                     descale_do=descale_do, bias=bias, dbias=dbias)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.sdpa_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), ws_bytes, _stream(stream, q)))


def _mask_problem(b: int, h_q: int, s_q: int, s_kv: int, dropout_p: float, causal=False) -> Problem:
    p = Problem()
    p.b, p.h_q, p.s_q, p.s_kv = b, h_q, s_q, s_kv
    p.dropout_p = float(dropout_p)
    p.causal = causal_code(causal)
    return p


def sdpa_dropout_mask_size(b: int, h_q: int, s_q: int, s_kv: int):
    """(bytes of the row-major keep bits, bytes of the transposed ones)."""
    n, n_t = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib.sdpa_dropout_mask_size(ctypes.byref(_mask_problem(b, h_q, s_q, s_kv, 0.0)),
                                      ctypes.byref(n), ctypes.byref(n_t)))
    return n.value, n_t.value


def sdpa_dropout_mask(b: int, h_q: int, s_q: int, s_kv: int, dropout_p: float, seed: int,
                      offset: int, mask=None, mask_t=None, stream=None, causal=False) -> None:
    """Draws the Philox4x32-10 keep bits into ``mask`` (row-major, for sdpa_fwd) and/or
    ``mask_t`` (transposed, for sdpa_bwd): CUDA tensors of sdpa_dropout_mask_size bytes.
    With ``causal`` (no per-batch lengths) tiles above the diagonal are left unwritten."""
    p = _mask_problem(b, h_q, s_q, s_kv, dropout_p, causal)
    _check(lib.sdpa_dropout_mask(ctypes.byref(p), int(seed), int(offset), _ptr(mask), _ptr(mask_t),
                                 _stream(stream, mask if mask is not None else mask_t)))


NOALLOC_SCRATCH_BYTES = 32 << 20  # SDPA_NOALLOC_SCRATCH_BYTES in include/sdpa.h


def sdpa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, *, attn_scale: Optional[float] = None,
                     causal=False, stream=None) -> None:
    """sdpa_bwd without a workspace, for callers that cannot allocate device memory: the
    scratch is a fixed 32 MiB array inside the library, shared by every call (calls must not
    overlap on the GPU; larger problems raise SdpaError with SDPA_ERR_UNSUPPORTED)."""
    p = make_problem(q, k, v, o, attn_scale=attn_scale, causal=causal, dout=dout, dq=dq, dk=dk,
                     dv=dv)
    _check(lib.sdpa_bwd_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout),
                                _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream, q)))


def sdpa_device_error() -> int:
    """Synchronises the device and returns (and clears) the kernels' error word."""
    f = ctypes.c_uint32(0)
    _check(lib.sdpa_device_error(ctypes.byref(f)))
    return f.value
