"""Large problems against the fp64 oracle.

- One sequence of 2^20 + 100 tokens (2 heads; AUTO runs its recurrence as
  segments).  The oracle cannot run a million tokens in a test, so its tail
  is checked.  With the bounded gate, every channel's summed log decay over
  4096 tokens is far below -200, so the state 4096 tokens back contributes
  less than e^-200 to the last 2048 tokens.  The oracle therefore restarts
  from a zero state 4096 tokens before the end, with the conv ring of the
  three raw rows before that point, and the last 2048 outputs and the final
  state must match.
- 512 heads (a 65536-wide row; more recurrence CTAs than SMs, several waves)
  on short sequences, sampled heads.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_04_gb300 as kda
import kda_synth
from kda_testlib import assert_close, head_cols, kda_params, oracle_run, tol_for

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_04_gb300 import build as kbuild
    kbuild.build()
    kda.lib()


def test_million_token_sequence_tail_against_oracle():
    T, H, io = (1 << 20) + 100, 2, "bf16"
    p = kda_synth.draw_params(H, 401)
    tk = kda_synth.draw_tokens(T, H, 402, torch.bfloat16, DEV)
    kp = kda_params(p, io)
    assert kda.kda_prefill_segments(kp, 1, T, kda.kda_prefill_workspace_bytes(kp, 1, T)) >= 5
    o, S, ring = kda.kda_prefill(kp, *tk.fields(), [0, T])
    torch.cuda.synchronize()
    # the oracle over the last 4096 tokens from zero state, ring = the 3 raw rows before
    t0 = T - 4096
    tail = kda_synth.Tokens(*[x[t0:].cpu() for x in tk.fields()])
    ring_in = torch.stack([torch.stack([pl[t0 - 3 + s] for s in range(3)]) for pl in (tk.q, tk.k, tk.v)])
    ring_in = ring_in[None].cpu()   # [1][3 planes][3 slots][W], slot 0 the oldest
    # the premise: every channel has decayed by far more than e^-200 over the first 2048
    # tokens of the tail (g <= 0 per token; summed in fp64 from the gate's definition)
    z = tail.z[:2048].double()
    x = torch.exp(p.A_log.double()).repeat_interleave(128)[None, :] * (z + p.dt_bias.double()[None, :])
    g = p.gate_lower_bound * torch.sigmoid(x)
    assert float(g.sum(0).max()) < -200.0
    ref = oracle_run(p, tail, [0, 4096], ring_in=ring_in)
    tol = tol_for(io)
    assert_close("o (last 2048 tokens)", o[T - 2048:], ref["o"][2048:], tol)
    assert_close("S", S, ref["S"], tol)
    np.testing.assert_array_equal(ring.double().cpu().numpy(), ref["ring"])


@pytest.mark.parametrize("lens", [[200, 1, 77], [1]])
def test_512_heads_sampled(lens):
    H, io = 512, "bf16"
    p = kda_synth.draw_params(H, 411)
    cu = kda_synth.cumsum0(lens)
    tk = kda_synth.draw_tokens(cu[-1], H, 412, torch.bfloat16)
    g = torch.Generator().manual_seed(413)
    n = len(lens)
    heads = [0, 255, 511]
    S0 = torch.randn(n, H, 128, 128, generator=g) * 0.05
    R0 = torch.randn(n, 3, 3, H * 128, generator=g).to(torch.bfloat16)
    kp = kda_params(p, io)
    o, S, ring = kda.kda_prefill(kp, *[t.to(DEV) for t in tk.fields()], cu, S_in=S0.to(DEV), ring_in=R0.to(DEV))
    torch.cuda.synchronize()
    ref = oracle_run(p, tk, cu, S_in=S0, ring_in=R0, heads=heads)
    cols = head_cols(heads).to(DEV)
    tol = tol_for(io)
    assert_close("o", o[:, cols], ref["o"], tol)
    assert_close("S", S[:, heads], ref["S"], tol)
    np.testing.assert_array_equal(ring[..., cols].double().cpu().numpy(), ref["ring"])
