"""Seeded synthetic inputs for the SDPA workloads.

This module only *draws and lays out* inputs.  It holds none of the attention
arithmetic, so both the fp64 oracle (``oracle/``) and the CUDA path (through
``attention_flashattention_sdpa_gb300``) can take their inputs from here without
sharing any of the method.

Recipe (the pages measure on synthetic tensors only: the cuDNN-in-Python post draws
``torch.randn(...).half()`` for its GPT-2-like problem; the attention codelab, §3
"Building Q, K, V test arrays", draws normal arrays of a fixed shape):

* one CPU ``torch.Generator`` seeded with ``seed`` (default 0);
* Q, K, V, dO drawn in that order as iid N(0, 1) fp32 over the *physical* buffer;
* cast to fp16 / bf16 with round-to-nearest-even (``Tensor.to``);
* layout ``"bhsd"``: contiguous [b, h, s, d]; layout ``"bshd"``: physical [b, s, h, d]
  viewed as logical BHSD with strides (s*h*d, d, h*d, 1), as in the GPT-2-like
  example of the cuDNN-in-Python post;
* FP8: each of Q, K, V is drawn as above in fp32, then quantised per tensor to
  OCP E4M3 (finite max 448) with ``scale = 448 / amax|x|``, ``descale = 1 / scale``
  (a single-step amax stands in for the amax history of the delayed-scaling recipe
  on the codelab's §10 "TransformerEngine and FP8").  The E4M3 bytes and the fp32
  descales are the inputs both sides see.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Tuple

import torch

E4M3_MAX = 448.0
E5M2_MAX = 57344.0


@dataclasses.dataclass(frozen=True)
class Workload:
    """One SDPA problem: logical BHSD shapes, dtype, layout and options."""
    name: str
    b: int
    h_q: int
    h_kv: int
    s_q: int
    s_kv: int
    d: int
    dtype: str            # "f16" | "bf16" | "e4m3"
    layout: str = "bhsd"  # "bhsd" | "bshd"
    causal: bool = False
    backward: bool = False
    stats: bool = True    # forward writes the per-row log-sum-exp
    attn_scale: Optional[float] = None
    alibi: bool = False   # ALiBi position bias with the default slopes
    dropout: float = 0.0  # dropout probability (0 = off)
    bias: bool = False    # an additive [1, h_q, s_q, s_kv] bias in the input dtype
    lens_q: Optional[Tuple[int, ...]] = None    # valid query rows per batch (padding mask)
    lens_kv: Optional[Tuple[int, ...]] = None   # valid keys per batch
    bottom_right: bool = False   # causal diagonal aligned to the end of each key sequence

    @property
    def scale(self) -> float:
        return self.attn_scale if self.attn_scale is not None else 1.0 / math.sqrt(self.d)

    def fwd_flops(self) -> float:
        """4*b*h_q*s_q*s_kv*d, halved for causal (the benchmark's counting rule).  Workloads
        with lengths or a bottom-right diagonal are counted by the benchmark itself."""
        f = 4.0 * self.b * self.h_q * self.s_q * self.s_kv * self.d
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops()


def tiny(causal: bool) -> Workload:
    return Workload("tiny" + ("_causal" if causal else ""), 1, 2, 2, 128, 128, 64, "f16",
                    causal=causal, backward=True)


def gpt2_inference() -> Workload:
    return Workload("gpt2_inference", 4, 12, 12, 1024, 1024, 64, "f16", layout="bshd",
                    causal=True, stats=False)


TRAINING_SEQ_LENS = (512, 1024, 2048, 4096, 8192, 16384)


def training(s: int) -> Workload:
    return Workload(f"training_s{s}", 2, 16, 16, s, s, 128, "bf16", causal=True, backward=True)


def fp8_large_head() -> Workload:
    return Workload("fp8_d256", 4, 16, 16, 4096, 4096, 256, "e4m3", causal=False, stats=False)


def grouped(h_kv: int) -> Workload:
    tag = {64: "mha", 8: "gqa", 1: "mqa"}.get(h_kv, f"hkv{h_kv}")
    return Workload(f"{tag}_70b", 1, 64, h_kv, 8192, 8192, 128, "bf16", causal=True, backward=True)


def training_alibi(s: int) -> Workload:
    """The training workload with the ALiBi bias on (default slopes)."""
    w = training(s)
    return Workload(f"training_alibi_bf16_causal_d128_s{s}", w.b, w.h_q, w.h_kv, s, s, w.d,
                    w.dtype, causal=True, backward=True, alibi=True)


def training_dropout(s: int, p: float = 0.1) -> Workload:
    """The training workload with attention dropout."""
    w = training(s)
    return Workload(f"training_dropout{p:g}_bf16_causal_d128_s{s}", w.b, w.h_q, w.h_kv, s, s, w.d,
                    w.dtype, causal=True, backward=True, dropout=p)


def training_fp8(s: int) -> Workload:
    """The training shape in FP8: E4M3 Q, K, V (bf16 O) and E5M2 dO."""
    w = training(s)
    return Workload(f"training_fp8_e4m3_causal_d128_s{s}", w.b, w.h_q, w.h_kv, s, s, w.d, "e4m3",
                    causal=True, backward=True)


def training_bias(s: int) -> Workload:
    """The training workload with a per-head additive bias broadcast over the batch."""
    w = training(s)
    return Workload(f"training_bias_bf16_causal_d128_s{s}", w.b, w.h_q, w.h_kv, s, s, w.d, w.dtype,
                    causal=True, backward=True, bias=True)


def backward_d256(causal: bool = True) -> Workload:
    """The large-head shape of the FP8 forward (b4 h16 s4096 d256) in bf16, forward with the
    statistics and then the backward pass."""
    return Workload(f"backward_d256_bf16{'_causal' if causal else ''}_s4096", 4, 16, 16, 4096, 4096, 256,
                    "bf16", causal=causal, backward=True)


def make_bias(w: Workload, seed: int = 3) -> torch.Tensor:
    """The additive bias of a ``bias`` workload: a [1, h_q, s_q, s_kv] tensor in the input
    dtype, broadcast over the batch, iid N(0, 1) from a CPU generator seeded with ``seed``,
    drawn head by head in fp32 and rounded to nearest even (as Q, K, V are)."""
    g = torch.Generator().manual_seed(seed)
    dt = _TORCH_DT[w.dtype]
    out = torch.empty(1, w.h_q, w.s_q, w.s_kv, dtype=dt)
    for h in range(w.h_q):
        out[0, h] = torch.randn(w.s_q, w.s_kv, generator=g, dtype=torch.float32).to(dt)
    return out


VARLEN_LENS = (8192, 7168, 6144, 5120, 4096, 3072, 2048, 1024)


def training_varlen() -> Workload:
    """A padded batch of eight sequences of 1K..8K tokens (4.5 full 8K sequences of work),
    self-attention with a causal mask, bf16 d=128, 16 heads."""
    n = len(VARLEN_LENS)
    return Workload("training_varlen_bf16_causal_d128_s1k-8k", n, 16, 16, 8192, 8192, 128, "bf16",
                    causal=True, backward=True, lens_q=VARLEN_LENS, lens_kv=VARLEN_LENS)


def prefill_bottom_right() -> Workload:
    """A 2K-token chunk attending to an 8K-token context (the chunk's rows see the whole
    prefix): bottom-right causal, s_q = 2048, s_kv = 8192, bf16 d=128, GQA 32/8 heads."""
    return Workload("prefill_bottom_right_bf16_d128_q2k_kv8k", 2, 32, 8, 2048, 8192, 128, "bf16",
                    causal=True, bottom_right=True, stats=False)


def all_workloads():
    out = [tiny(False), tiny(True), gpt2_inference()]
    out += [training(s) for s in TRAINING_SEQ_LENS]
    out += [fp8_large_head(), grouped(8), grouped(1), grouped(64), training_alibi(8192),
            training_dropout(8192), training_fp8(8192), training_bias(8192), training_varlen(),
            prefill_bottom_right(), backward_d256(True), backward_d256(False)]
    return out


_TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def _logical(buf: torch.Tensor, b: int, h: int, s: int, d: int, layout: str) -> torch.Tensor:
    if layout == "bhsd":
        return buf.view(b, h, s, d)
    if layout == "bshd":
        return buf.view(b, s, h, d).permute(0, 2, 1, 3)
    raise ValueError(f"unknown layout {layout!r}")


def _draw(g: torch.Generator, n: int) -> torch.Tensor:
    return torch.randn(n, generator=g, dtype=torch.float32)


def quantize_e5m2(x: torch.Tensor):
    """Per-tensor amax quantisation to E5M2, the gradient format (input preparation).

    Returns (bytes-as-float8 tensor with x's shape/strides, descale float)."""
    amax = float(x.abs().max())
    scale = E5M2_MAX / amax if amax > 0 else 1.0
    q8 = (x.float() * scale).clamp_(-E5M2_MAX, E5M2_MAX).to(torch.float8_e5m2)
    return q8, 1.0 / scale


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor amax quantisation to E4M3 (input preparation, not the method).

    Returns (bytes-as-float8 tensor with x's shape/strides, descale float)."""
    amax = float(x.abs().max())
    scale = E4M3_MAX / amax if amax > 0 else 1.0
    q8 = (x.float() * scale).clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q8, 1.0 / scale


@dataclasses.dataclass
class Inputs:
    """CPU tensors (logical BHSD views) plus FP8 descales when dtype is e4m3."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: Optional[torch.Tensor] = None
    descale_q: float = 1.0
    descale_k: float = 1.0
    descale_v: float = 1.0
    descale_do: float = 1.0


def make_inputs(w: Workload, seed: int = 0, with_do: Optional[bool] = None) -> Inputs:
    """Draw Q, K, V (and dO) for workload ``w`` following the recipe above."""
    if with_do is None:
        with_do = w.backward
    g = torch.Generator().manual_seed(seed)
    nq = w.b * w.h_q * w.s_q * w.d
    nkv = w.b * w.h_kv * w.s_kv * w.d
    qf, kf, vf = _draw(g, nq), _draw(g, nkv), _draw(g, nkv)
    dof = _draw(g, nq) if with_do else None
    if w.dtype == "e4m3":
        q8, dq_ = quantize_e4m3(qf)
        k8, dk_ = quantize_e4m3(kf)
        v8, dv_ = quantize_e4m3(vf)
        do8, ddo_ = quantize_e5m2(dof) if dof is not None else (None, 1.0)
        return Inputs(_logical(q8, w.b, w.h_q, w.s_q, w.d, w.layout),
                      _logical(k8, w.b, w.h_kv, w.s_kv, w.d, w.layout),
                      _logical(v8, w.b, w.h_kv, w.s_kv, w.d, w.layout),
                      _logical(do8, w.b, w.h_q, w.s_q, w.d, w.layout) if do8 is not None else None,
                      dq_, dk_, dv_, ddo_)
    dt = _TORCH_DT[w.dtype]
    mk = lambda f, h, s: _logical(f.to(dt), w.b, h, s, w.d, w.layout)
    return Inputs(mk(qf, w.h_q, w.s_q), mk(kf, w.h_kv, w.s_kv), mk(vf, w.h_kv, w.s_kv),
                  mk(dof, w.h_q, w.s_q) if dof is not None else None)


def sample_rows(w: Workload, n: int, seed: int = 1):
    """Seeded (b, h_q, row) triples for checking large shapes row by row.

    Always includes the first and last rows of the sequence (the causal edge cases)."""
    g = torch.Generator().manual_seed(seed)
    bs = torch.randint(0, w.b, (n,), generator=g).tolist()
    hs = torch.randint(0, w.h_q, (n,), generator=g).tolist()
    rs = torch.randint(0, w.s_q, (n,), generator=g).tolist()
    out = list(zip(bs, hs, rs))
    out[0] = (0, 0, 0)
    out[-1] = (w.b - 1, w.h_q - 1, w.s_q - 1)
    return out


def sample_kv_heads(w: Workload, n: int, seed: int = 2):
    """Seeded (b, kv-head) pairs for checking dK/dV of large shapes head by head."""
    g = torch.Generator().manual_seed(seed)
    pairs = {(0, 0), (w.b - 1, w.h_kv - 1)}
    while len(pairs) < min(n, w.b * w.h_kv):
        pairs.add((int(torch.randint(0, w.b, (1,), generator=g)),
                   int(torch.randint(0, w.h_kv, (1,), generator=g))))
    return sorted(pairs)
