"""Seeded synthetic inputs for the KDA mixer core.

This module only draws random numbers with the shapes and value
distributions of the five workloads below; it holds none of the method's
arithmetic, so both the CUDA path and the fp64 oracle may take their inputs
from it.

Distributions (``N(0, s)`` names the variance ``s``):
  raw q/k/v ~ N(0,1); conv weights ~ N(0,0.25); gate input z ~ N(0,1);
  dt_bias ~ N(0,0.5); A_log = log U(1,16) per head; beta logits b ~ N(0,1);
  output-gate logits ~ N(0,1); RMSNorm weight 1 + N(0,0.1); gate lower bound
  -5, L2 eps 1e-6, RMSNorm eps 1e-5.  bf16 workloads round every I/O tensor
  to bf16 once; both implementations read the same bits.

Workloads (seed = 1000 + workload index):
  0 "tiny"    B=1, T=64, H=2, fp32 I/O, zero state and ring
  1 "decode"  256 sessions x H=32, one token each, bf16; state and ring come
              from 512 warm-up tokens per session (drawn here, run by caller)
  2 "prefill" B=1, T=4096, H=32, bf16, zero state
  3 "long"    B=1, T=32768, H=96, bf16, zero state
  4 "varlen"  8 sequences, lengths ~ U_int[512, 16384], H=64, bf16; state and
              ring from 256 warm-up tokens per sequence
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

HEAD_DIM = 128

WORKLOADS = {
    0: dict(name="tiny", H=2, lens=[64], io="f32", warmup=0),
    1: dict(name="decode", H=32, lens=[1] * 256, io="bf16", warmup=512),
    2: dict(name="prefill", H=32, lens=[4096], io="bf16", warmup=0),
    3: dict(name="long", H=96, lens=[32768], io="bf16", warmup=0),
    4: dict(name="varlen", H=64, lens=None, io="bf16", warmup=256),
}


def describe(idx: int, H=None) -> str:
    w = WORKLOADS[idx]
    lens = w["lens"] if w["lens"] is not None else varlen_lengths()
    return (f"{w['name']}: {len(lens)} seq(s), {sum(lens)} tokens, H={H or w['H']}, d={HEAD_DIM}, "
            f"{w['io']} I/O, warm-up {w['warmup']} tokens/seq")


def varlen_lengths(seed: int = 1004, n: int = 8, lo: int = 512, hi: int = 16384):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def io_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(seed)


@dataclass
class Params:
    num_heads: int
    head_dim: int
    conv_w: torch.Tensor   # [3][H*D][4] fp32
    A_log: torch.Tensor    # [H] fp32
    dt_bias: torch.Tensor  # [H*D] fp32
    norm_w: torch.Tensor   # [D] fp32
    gate_lower_bound: float = -5.0
    l2_eps: float = 1e-6
    norm_eps: float = 1e-5
    q_scale: float = 0.0
    gate_kind: int = 0     # 0: lower-bounded sigmoid gate; 1: -exp(A_log) softplus(z + dt_bias)

    def to(self, device) -> "Params":
        return Params(self.num_heads, self.head_dim, self.conv_w.to(device), self.A_log.to(device),
                      self.dt_bias.to(device), self.norm_w.to(device), self.gate_lower_bound,
                      self.l2_eps, self.norm_eps, self.q_scale, self.gate_kind)

    def head_slice(self, heads) -> "Params":
        """Parameters of a subset of heads (heads are independent)."""
        D = self.head_dim
        idx = torch.tensor(heads, dtype=torch.long, device=self.A_log.device)
        ch = (idx[:, None] * D + torch.arange(D, device=idx.device)[None, :]).reshape(-1)
        return Params(len(heads), D, self.conv_w[:, ch, :].contiguous(), self.A_log[idx].contiguous(),
                      self.dt_bias[ch].contiguous(), self.norm_w.clone(), self.gate_lower_bound,
                      self.l2_eps, self.norm_eps, self.q_scale, self.gate_kind)


def draw_params(H: int, seed: int, device="cpu", D: int = HEAD_DIM) -> Params:
    g = _gen(seed, device)
    W = H * D
    conv_w = torch.randn(3, W, 4, generator=g, device=device) * 0.5
    A_log = torch.log(torch.rand(H, generator=g, device=device) * 15.0 + 1.0)
    dt_bias = torch.randn(W, generator=g, device=device) * math.sqrt(0.5)
    norm_w = 1.0 + torch.randn(D, generator=g, device=device) * math.sqrt(0.1)
    return Params(H, D, conv_w.float(), A_log.float(), dt_bias.float(), norm_w.float())


@dataclass
class Tokens:
    q: torch.Tensor     # [T][W]
    k: torch.Tensor
    v: torch.Tensor
    z: torch.Tensor
    b: torch.Tensor     # [T][H]
    gout: torch.Tensor  # [T][W]

    def fields(self):
        return (self.q, self.k, self.v, self.z, self.b, self.gout)

    def head_slice(self, heads, D: int = HEAD_DIM) -> "Tokens":
        idx = torch.tensor(heads, dtype=torch.long, device=self.q.device)
        ch = (idx[:, None] * D + torch.arange(D, device=idx.device)[None, :]).reshape(-1)
        return Tokens(self.q[:, ch], self.k[:, ch], self.v[:, ch], self.z[:, ch], self.b[:, idx],
                      self.gout[:, ch])


def draw_tokens(T: int, H: int, seed: int, dtype: torch.dtype, device="cpu",
                D: int = HEAD_DIM) -> Tokens:
    """Raw projections for T packed tokens, rounded once to ``dtype``."""
    g = _gen(seed, device)
    W = H * D

    def n(*shape):
        return torch.randn(*shape, generator=g, device=device).to(dtype)

    return Tokens(n(T, W), n(T, W), n(T, W), n(T, W), n(T, H), n(T, W))


@dataclass
class Workload:
    idx: int
    name: str
    params: Params
    tokens: Tokens
    cu_seqlens: list
    io: str
    warmup_tokens: Optional[Tokens] = None
    warmup_cu: Optional[list] = None
    meta: dict = field(default_factory=dict)

    @property
    def H(self):
        return self.params.num_heads

    @property
    def total_tokens(self):
        return self.cu_seqlens[-1]

    @property
    def n_seqs(self):
        return len(self.cu_seqlens) - 1


def cumsum0(lens):
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + int(L))
    return cu


def workload(idx: int, device="cpu", lens=None, H=None) -> Workload:
    """Draw workload ``idx`` on ``device``.  ``lens``/``H`` override the
    sequence lengths / head count (used for smaller cases of the same recipe)."""
    w = WORKLOADS[idx]
    seed = 1000 + idx
    H = H or w["H"]
    if lens is None:
        lens = w["lens"] if w["lens"] is not None else varlen_lengths()
    dtype = io_dtype(w["io"])
    params = draw_params(H, seed, device)
    cu = cumsum0(lens)
    tokens = draw_tokens(cu[-1], H, seed + 100_000, dtype, device)
    wt, wcu = None, None
    if w["warmup"]:
        wcu = cumsum0([w["warmup"]] * len(lens))
        wt = draw_tokens(wcu[-1], H, seed + 200_000, dtype, device)
    return Workload(idx, w["name"], params, tokens, cu, w["io"], wt, wcu)
