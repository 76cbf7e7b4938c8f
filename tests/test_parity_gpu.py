"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Tolerances (GPU vs oracle, rel-L2 = |x - y|_2 / |y|_2 over the tensor):
fp32 I/O: rel-L2 <= 1e-4 on o and S; bf16 I/O with fp32 state: rel-L2 <= 2e-2
and max-abs <= 5e-2 on o and S.  The conv ring is a copy and must match
bit for bit.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_04_gb300 as kda
import kda_synth
from kda_testlib import (assert_close, head_cols, kda_params, oracle_run, tol_for)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_04_gb300 import build as kbuild
    kbuild.build()
    kda.lib()


def run_prefill(p, tokens, cu, io, algo="auto", S_in=None, ring_in=None, alias=False):
    kp = kda_params(p, io, algo)
    d = [t.to(DEV) for t in tokens.fields()]
    S_in_d = None if S_in is None else S_in.to(DEV).contiguous()
    ring_in_d = None if ring_in is None else ring_in.to(DEV).contiguous()
    if alias:
        o, S, ring = kda.kda_prefill(kp, *d, cu, S_in=S_in_d, S_out=S_in_d, ring_in=ring_in_d,
                                     ring_out=ring_in_d)
    else:
        o, S, ring = kda.kda_prefill(kp, *d, cu, S_in=S_in_d, ring_in=ring_in_d)
    torch.cuda.synchronize()
    return o, S, ring


def check_against_oracle(p, tokens, cu, io, o, S, ring, S_in=None, ring_in=None, heads=None):
    ref = oracle_run(p, tokens, cu, S_in=S_in, ring_in=ring_in, heads=heads)
    tol = tol_for(io)
    if heads is not None:
        cols = head_cols(heads).to(o.device)
        o = o[:, cols]
        S = S[:, torch.tensor(heads, device=S.device)]
        ring = ring[..., cols]
    assert_close("o", o, ref["o"], tol)
    assert_close("S", S, ref["S"], tol)
    np.testing.assert_array_equal(ring.double().cpu().numpy(), ref["ring"])
    return ref


# ---------------------------------------------------------------- config 0
@pytest.mark.parametrize("algo", ["auto", "scan"])
def test_tiny_f32_prefill(algo):
    w = kda_synth.workload(0)
    o, S, ring = run_prefill(w.params, w.tokens, w.cu_seqlens, w.io, algo)
    check_against_oracle(w.params, w.tokens, w.cu_seqlens, w.io, o, S, ring)


def test_tiny_f32_as_decode_steps():
    """Workload 0 run as 64 one-token decode steps equals the oracle's prefill."""
    w = kda_synth.workload(0)
    kp = kda_params(w.params, w.io)
    H = w.H
    S = torch.zeros(1, H, 128, 128, device=DEV)
    ring = torch.zeros(1, 3, 3, H * 128, device=DEV)
    d = [t.to(DEV) for t in w.tokens.fields()]
    outs = []
    for t in range(w.total_tokens):
        outs.append(kda.kda_decode(kp, *[x[t:t + 1] for x in d], S, ring))
    torch.cuda.synchronize()
    o = torch.cat(outs)
    check_against_oracle(w.params, w.tokens, w.cu_seqlens, w.io, o, S, ring)


# ---------------------------------------------------------------- config 2
@pytest.mark.parametrize("algo", ["auto", "scan"])
def test_prefill_T4096_H32_bf16(algo):
    w = kda_synth.workload(2, device=DEV)
    o, S, ring = run_prefill(w.params, w.tokens, w.cu_seqlens, w.io, algo)
    check_against_oracle(w.params.to("cpu"), w.tokens, w.cu_seqlens, w.io, o, S, ring)


# ---------------------------------------------------------------- config 3
def test_long_prefill_T32768_H96_sampled_heads():
    """Full-size workload in the benchmark's launch configuration; the oracle
    checks three heads (heads are independent)."""
    w = kda_synth.workload(3, device=DEV)
    o, S, ring = run_prefill(w.params, w.tokens, w.cu_seqlens, w.io)
    check_against_oracle(w.params.to("cpu"), w.tokens, w.cu_seqlens, w.io, o, S, ring, heads=[0, 47, 95])


# ---------------------------------------------------------------- config 4
def varlen_state(w, heads=None):
    """Initial state and ring from the oracle run over the warm-up tokens."""
    ref = oracle_run(w.params.to("cpu"), w.warmup_tokens, w.warmup_cu, heads=heads)
    return torch.from_numpy(ref["S"]).float(), torch.from_numpy(ref["ring"]).to(torch.bfloat16)


def test_varlen_continuing_sessions_sampled_heads():
    w = kda_synth.workload(4, device=DEV)
    heads = [0, 33, 63]
    S_h, ring_h = varlen_state(w, heads)
    # full-width state: oracle warm-up on the checked heads, zero elsewhere
    S_in = torch.zeros(w.n_seqs, w.H, 128, 128)
    S_in[:, torch.tensor(heads)] = S_h
    ring_in = torch.zeros(w.n_seqs, 3, 3, w.H * 128, dtype=torch.bfloat16)
    ring_in[..., head_cols(heads)] = ring_h
    o, S, ring = run_prefill(w.params, w.tokens, w.cu_seqlens, w.io, S_in=S_in, ring_in=ring_in)
    check_against_oracle(w.params.to("cpu"), w.tokens, w.cu_seqlens, w.io, o, S, ring,
                         S_in=S_in, ring_in=ring_in, heads=heads)


# ---------------------------------------------------------------- config 1
def test_decode_256_sessions_H32_bf16_sampled():
    """One decode step over 256 sessions x 32 heads; sessions 0, 97, 255 start
    from the oracle's state after 512 warm-up tokens and are checked."""
    w = kda_synth.workload(1, device=DEV)
    sessions = [0, 97, 255]
    kp = kda_params(w.params, w.io)
    # warm-up on the GPU gives every session a realistic state (timing input);
    # the checked sessions are then overwritten with the oracle's warm-up
    wcu = w.warmup_cu
    _, S, ring = kda.kda_prefill(kp, *[t for t in w.warmup_tokens.fields()], wcu)
    sub_cu = kda_synth.cumsum0([512] * len(sessions))
    rows = torch.cat([torch.arange(wcu[s], wcu[s + 1]) for s in sessions]).to(DEV)
    sub = kda_synth.Tokens(*[t[rows] for t in w.warmup_tokens.fields()])
    ref_w = oracle_run(w.params.to("cpu"), sub, sub_cu)
    idx = torch.tensor(sessions, device=DEV)
    S[idx] = torch.from_numpy(ref_w["S"]).float().to(DEV)
    ring[idx] = torch.from_numpy(ref_w["ring"]).to(torch.bfloat16).to(DEV)
    S0 = S[idx].cpu()
    ring0 = ring[idx].cpu()
    o = kda.kda_decode(kp, *[t for t in w.tokens.fields()], S, ring)
    torch.cuda.synchronize()
    step = kda_synth.Tokens(*[t[idx] for t in w.tokens.fields()])
    ref = oracle_run(w.params.to("cpu"), step, list(range(len(sessions) + 1)), S_in=S0, ring_in=ring0)
    tol = tol_for(w.io)
    assert_close("o", o[idx], ref["o"], tol)
    assert_close("S", S[idx], ref["S"], tol)
    np.testing.assert_array_equal(ring[idx].double().cpu().numpy(), ref["ring"])


# ---------------------------------------------------------------- edge cases
def small_case(io, lens, H=2, seed=5):
    p = kda_synth.draw_params(H, seed)
    cu = kda_synth.cumsum0(lens)
    tk = kda_synth.draw_tokens(cu[-1], H, seed + 1, kda_synth.io_dtype(io))
    return p, tk, cu


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_ragged_varlen_with_empty_and_short_sequences(io):
    """Lengths spanning several chunks, a ragged tail, empty and sub-ring
    sequences, with nonzero initial state and ring."""
    lens = [0, 1, 2, 3, 63, 64, 65, 200, 0, 129]
    p, tk, cu = small_case(io, lens)
    n, H = len(lens), p.num_heads
    g = torch.Generator().manual_seed(77)
    S_in = torch.randn(n, H, 128, 128, generator=g) * 0.05
    ring_in = torch.randn(n, 3, 3, H * 128, generator=g).to(kda_synth.io_dtype(io))
    o, S, ring = run_prefill(p, tk, cu, io, S_in=S_in, ring_in=ring_in)
    check_against_oracle(p, tk, cu, io, o, S, ring, S_in=S_in, ring_in=ring_in)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_in_place_state_and_ring(io):
    lens = [5, 70, 2]
    p, tk, cu = small_case(io, lens, seed=9)
    n, H = len(lens), p.num_heads
    g = torch.Generator().manual_seed(78)
    S_in = torch.randn(n, H, 128, 128, generator=g) * 0.05
    ring_in = torch.randn(n, 3, 3, H * 128, generator=g).to(kda_synth.io_dtype(io))
    o, S, ring = run_prefill(p, tk, cu, io, S_in=S_in.clone(), ring_in=ring_in.clone(), alias=True)
    check_against_oracle(p, tk, cu, io, o, S, ring, S_in=S_in, ring_in=ring_in)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_prefill_one_token_equals_decode(io):
    lens = [1, 1, 1]
    p, tk, cu = small_case(io, lens, seed=11)
    n, H = len(lens), p.num_heads
    g = torch.Generator().manual_seed(79)
    S_in = (torch.randn(n, H, 128, 128, generator=g) * 0.05).to(DEV)
    ring_in = torch.randn(n, 3, 3, H * 128, generator=g).to(kda_synth.io_dtype(io)).to(DEV)
    o_p, S_p, ring_p = run_prefill(p, tk, cu, io, algo="scan", S_in=S_in, ring_in=ring_in)
    kp = kda_params(p, io)
    S_d, ring_d = S_in.clone(), ring_in.clone()
    o_d = kda.kda_decode(kp, *[t.to(DEV) for t in tk.fields()], S_d, ring_d)
    torch.cuda.synchronize()
    assert torch.equal(ring_p, ring_d)
    rel = (torch.linalg.norm((o_p - o_d).double()) / torch.linalg.norm(o_d.double())).item()
    assert rel < (1e-5 if io == "f32" else 1e-2)
    rel = (torch.linalg.norm((S_p - S_d).double()) / torch.linalg.norm(S_d.double())).item()
    assert rel < 1e-5


def test_deterministic_repeat_runs():
    p, tk, cu = small_case("bf16", [300, 17], seed=13)
    a = run_prefill(p, tk, cu, "bf16")
    b = run_prefill(p, tk, cu, "bf16")
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_zero_tokens_copies_state():
    p, tk, cu = small_case("bf16", [0, 0], seed=15)
    n, H = 2, p.num_heads
    S_in = torch.randn(n, H, 128, 128)
    ring_in = torch.randn(n, 3, 3, H * 128).to(torch.bfloat16)
    kp = kda_params(p, "bf16")
    empty = torch.empty(0, H * 128, dtype=torch.bfloat16, device=DEV)
    emptyb = torch.empty(0, H, dtype=torch.bfloat16, device=DEV)
    o, S, ring = kda.kda_prefill(kp, empty, empty, empty, empty, emptyb, empty, cu,
                                 S_in=S_in.to(DEV), ring_in=ring_in.to(DEV), o=empty)
    torch.cuda.synchronize()
    assert torch.equal(S.cpu(), S_in)
    assert torch.equal(ring.cpu(), ring_in)


# ---------------------------------------------------------------- softplus gate
@pytest.mark.parametrize("io, algo, runs", [("f32", "auto", "scan"), ("bf16", "scan", "scan"),
                                            ("bf16", "auto", "chunked")])
def test_softplus_gate_prefill_and_verify(io, algo, runs):
    """The earlier Kimi-Linear gate (unbounded below) on the scan prefill and
    on the chunked form (bf16 I/O), and on a multi-token decode round
    continuing from it."""
    lens = [70, 3, 131]
    p, tk, cu = small_case(io, lens, seed=91)
    p.gate_kind = 1
    n, H = len(lens), p.num_heads
    kp = kda_params(p, io, algo)
    assert kda.kda_prefill_algo(kp) == runs
    g = torch.Generator().manual_seed(92)
    S_in = torch.randn(n, H, 128, 128, generator=g) * 0.05
    ring_in = torch.randn(n, 3, 3, H * 128, generator=g).to(kda_synth.io_dtype(io))
    o, S, ring = run_prefill(p, tk, cu, io, algo, S_in=S_in, ring_in=ring_in)
    ref = check_against_oracle(p, tk, cu, io, o, S, ring, S_in=S_in, ring_in=ring_in)
    # a 3-token round per session from the prefill's state
    n_tok = 3
    vt = kda_synth.draw_tokens(n * n_tok, H, 93, kda_synth.io_dtype(io))
    rounds = [t.reshape(n, n_tok, *t.shape[1:]).contiguous().to(DEV) for t in vt.fields()]
    o2 = kda.kda_decode_multi(kp, *rounds, S, ring)
    torch.cuda.synchronize()
    ref2 = oracle_run(p, vt, list(range(0, n * n_tok + 1, n_tok)), S_in=torch.from_numpy(ref["S"]).float(),
                      ring_in=torch.from_numpy(ref["ring"]).to(kda_synth.io_dtype(io)))
    tol = tol_for(io)
    assert_close("o", o2.reshape(n * n_tok, -1), ref2["o"], tol)
    assert_close("S", S, ref2["S"], tol)
