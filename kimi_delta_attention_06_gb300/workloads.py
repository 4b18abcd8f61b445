"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module draws random tensors and nothing else: it holds none of the KDA
arithmetic, so both the CUDA path and the fp64 oracle can consume what it
produces without sharing any of the method's code.

Recipes (the shapes and value distributions of the workloads the Kimi K3
primer describes: median 142k-token agentic prompts and single-token decode,
SemiAnalysis wiki summary section 9 / InferenceX "Inference performance"):

* q, k, v ~ N(0, 1); q and k L2-normalised per (token, head), which the KDA
  module does before the recurrence (primer section 3);
* beta = sigmoid(N(0, 1));
* log_alpha = -softplus(N(0, 1) + shift) per channel (shift 0 for the tiny
  case, -2 for the 128-dim cases, so alpha is mostly 0.85..0.99);
* initial states ~ N(0, 0.02) fp32 where a case has one.

q, k, v and beta are handed to the GPU as bf16; log_alpha and states are
fp32.  The oracle receives exactly the same (rounded) values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import List, Optional

import torch
import torch.nn.functional as F


@dataclass
class PrefillCase:
    name: str
    q: torch.Tensor            # [T, H, Dk] bf16
    k: torch.Tensor            # [T, H, Dk] bf16
    v: torch.Tensor            # [T, H, Dv] bf16
    log_alpha: torch.Tensor    # [T, H, Dk] fp32
    beta: torch.Tensor         # [T, H] bf16
    init_state: Optional[torch.Tensor]   # [N, H, Dk, Dv] fp32 or None
    cu_seqlens: torch.Tensor   # [N+1] int32, host
    ckpt_stride: int

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def H(self) -> int:
        return int(self.q.shape[1])

    @property
    def Dk(self) -> int:
        return int(self.q.shape[2])

    @property
    def Dv(self) -> int:
        return int(self.v.shape[2])

    @property
    def N(self) -> int:
        return int(self.cu_seqlens.numel() - 1)


@dataclass
class DecodeCase:
    name: str
    state: torch.Tensor        # [N, H, Dk, Dv] fp32
    steps: List[dict]          # per step: q, k, v (bf16), log_alpha (fp32), beta (bf16)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _unit(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def _token_inputs(T: int, H: int, Dk: int, Dv: int, g, device, la_shift: float):
    q = _unit(torch.randn(T, H, Dk, generator=g, device=device)).to(torch.bfloat16)
    k = _unit(torch.randn(T, H, Dk, generator=g, device=device)).to(torch.bfloat16)
    v = torch.randn(T, H, Dv, generator=g, device=device).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn(T, H, generator=g, device=device)).to(torch.bfloat16)
    la = -F.softplus(torch.randn(T, H, Dk, generator=g, device=device) + la_shift)
    return q, k, v, la.contiguous(), beta


def prefill_case(lengths: List[int], H: int, D: int, seed: int, device="cpu",
                 la_shift: float = -2.0, s0_std: Optional[float] = 0.02,
                 s0_every_other: bool = False, ckpt_stride: int = 0,
                 name: str = "prefill") -> PrefillCase:
    """Packed prefill inputs for sequences of the given lengths."""
    g = _gen(seed, device)
    T = int(sum(lengths))
    q, k, v, la, beta = _token_inputs(T, H, D, D, g, device, la_shift)
    N = len(lengths)
    s0 = None
    if s0_std is not None:
        s0 = torch.randn(N, H, D, D, generator=g, device=device) * s0_std
        if s0_every_other:           # odd sequences start from zeros
            s0[1::2] = 0
    cu = torch.zeros(N + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return PrefillCase(name, q, k, v, la, beta, s0, cu, ckpt_stride)


def tiny_case(seed: int = 0, device="cpu") -> PrefillCase:
    """B=1, H=2, T=256, Dk=Dv=64: the case the oracle finishes in well under a second.

    q, k, v are drawn in fp32 and rounded to bf16 (the GPU's input type);
    log_alpha = -softplus(N(0,1)); zero initial state.
    """
    return prefill_case([256], H=2, D=64, seed=seed, device=device, la_shift=0.0,
                        s0_std=None, name="tiny_T256_H2_D64")


def single_case(T: int, seed: int = 1, device="cpu", H: int = 32, D: int = 128,
                ckpt_stride: int = 0) -> PrefillCase:
    """B=1 long prompt, H=32, D=128, fp32 N(0, 0.02) initial state."""
    return prefill_case([T], H=H, D=D, seed=seed, device=device, la_shift=-2.0,
                        s0_std=0.02, ckpt_stride=ckpt_stride, name=f"single_T{T}_H{H}_D{D}")


def varlen_lengths(seed: int, num_seqs: int = 16, lo: int = 1024, hi: int = 65536,
                   target=(270_000, 330_000)) -> (List[int], int):
    """Log-uniform lengths in [lo, hi]; the first seed >= ``seed`` whose total
    falls inside ``target`` (about 300k tokens) is used.  Returns (lengths, seed)."""
    s = int(seed)
    while True:
        g = torch.Generator().manual_seed(s)
        u = torch.rand(num_seqs, generator=g, dtype=torch.float64)
        lens = [int(math.floor(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo)))))
                for x in u]
        if target is None or target[0] <= sum(lens) <= target[1]:
            return lens, s
        s += 1


def varlen_case(seed: int = 3, device="cpu", H: int = 32, D: int = 128,
                ckpt_stride: int = 32768) -> PrefillCase:
    """16 packed sequences, log-uniform lengths in [1k, 64k] (~300k tokens);
    even-numbered sequences start from an N(0, 0.02) state (prefix-cache hit),
    odd ones from zeros."""
    lens, s = varlen_lengths(seed)
    c = prefill_case(lens, H=H, D=D, seed=s, device=device, la_shift=-2.0, s0_std=0.02,
                     s0_every_other=True, ckpt_stride=ckpt_stride)
    c.name = f"varlen16_T{sum(lens)}_H{H}_D{D}_seed{s}"
    return c


def decode_case(N: int = 512, H: int = 32, D: int = 128, steps: int = 64, seed: int = 4,
                device="cpu", la_shift: float = -2.0) -> DecodeCase:
    """N concurrent sequences x H heads, one token per step, fp32 N(0, 0.02) states."""
    g = _gen(seed, device)
    state = torch.randn(N, H, D, D, generator=g, device=device) * 0.02
    st = []
    for _ in range(steps):
        q, k, v, la, beta = _token_inputs(N, H, D, D, g, device, la_shift)
        st.append(dict(q=q, k=k, v=v, log_alpha=la, beta=beta))
    return DecodeCase(f"decode_N{N}_H{H}_D{D}", state, st)


@dataclass
class ModuleCase:
    """Raw inputs of the KDA module around the recurrence: the q, k, v projections before
    the short convolution, its depthwise taps, the gate pre-activations, and the output
    norm weight."""
    xq: torch.Tensor           # [T, H, D] bf16
    xk: torch.Tensor
    xv: torch.Tensor
    conv_w: torch.Tensor       # [3, H, D, 4] fp32
    a_raw: torch.Tensor        # [T, H, D] fp32 (alpha gate pre-activation)
    b_raw: torch.Tensor        # [T, H] bf16 (beta pre-activation)
    gamma: torch.Tensor        # [H, D] fp32 (output norm weight)
    cu_seqlens: torch.Tensor   # [2] int32, host


def module_case(T: int, H: int = 32, D: int = 128, seed: int = 5, device="cpu") -> ModuleCase:
    """One T-token prompt: projections ~ N(0, 1), taps ~ N(0, 0.5^2), alpha pre-activations
    ~ N(-2, 1) (so -softplus gives the decays of the prefill cases), beta pre-activations
    ~ N(0, 1), norm weight ~ U(0.5, 1.5)."""
    g = _gen(seed, device)
    xq, xk, xv = (torch.randn(T, H, D, generator=g, device=device).to(torch.bfloat16) for _ in range(3))
    w = torch.randn(3, H, D, 4, generator=g, device=device) * 0.5
    a = torch.randn(T, H, D, generator=g, device=device) - 2.0
    b = torch.randn(T, H, generator=g, device=device).to(torch.bfloat16)
    gamma = torch.rand(H, D, generator=g, device=device) + 0.5
    cu = torch.tensor([0, T], dtype=torch.int32)
    return ModuleCase(xq, xk, xv, w.contiguous(), a.contiguous(), b, gamma.contiguous(), cu)


def head_slice(case, h0: int, h1: int):
    """The same inputs restricted to heads [h0, h1): one rank's share when a prompt's
    heads are split over ranks.  Works on PrefillCase, DecodeCase and ModuleCase; every
    sliced tensor is made contiguous (the kernels take packed [.., H, ..] layouts)."""
    def cut(x, dim):
        return None if x is None else x.narrow(dim, h0, h1 - h0).contiguous()

    if isinstance(case, PrefillCase):
        return replace(case, name=f"{case.name}_heads{h0}-{h1}", q=cut(case.q, 1), k=cut(case.k, 1),
                       v=cut(case.v, 1), log_alpha=cut(case.log_alpha, 1), beta=cut(case.beta, 1),
                       init_state=cut(case.init_state, 1))
    if isinstance(case, DecodeCase):
        return DecodeCase(f"{case.name}_heads{h0}-{h1}", cut(case.state, 1),
                          [{k: cut(v, 1) for k, v in st.items()} for st in case.steps])
    if isinstance(case, ModuleCase):
        return replace(case, xq=cut(case.xq, 1), xk=cut(case.xk, 1), xv=cut(case.xv, 1),
                       conv_w=cut(case.conv_w, 1), a_raw=cut(case.a_raw, 1), b_raw=cut(case.b_raw, 1),
                       gamma=cut(case.gamma, 0))
    raise TypeError(f"no head layout known for {type(case).__name__}")
