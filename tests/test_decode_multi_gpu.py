"""Multi-token decode (speculative verify rounds) over a state pool, through
the C ABI, against the fp64 oracle: a round of n_tokens per session equals
the recurrence over those tokens (a prefill with one sequence per session);
keeping the input state allows a rollback by replaying the accepted prefix;
pool slots index the state and ring."""
import numpy as np
import pytest
import torch

import gated_delta_rule_04_gb300 as kda
import kda_synth
from kda_testlib import assert_close, kda_params, oracle_run, tol_for

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_04_gb300 import build as kbuild
    kbuild.build()
    kda.lib()


def round_inputs(io, n, n_tok, H=2, seed=21):
    """Tokens of n sessions x n_tok, nonzero initial state and ring."""
    p = kda_synth.draw_params(H, seed)
    tk = kda_synth.draw_tokens(n * n_tok, H, seed + 1, kda_synth.io_dtype(io))
    g = torch.Generator().manual_seed(seed + 2)
    S0 = torch.randn(n, H, 128, 128, generator=g) * 0.05
    ring0 = torch.randn(n, 3, 3, H * 128, generator=g).to(kda_synth.io_dtype(io))
    return p, tk, S0, ring0


def as_rounds(t, n, n_tok):
    return t.reshape(n, n_tok, *t.shape[1:]).contiguous()


def first_tokens(tk, n, n_tok, j):
    """The first j tokens of every session, as flat [n*j][...] tensors."""
    return kda_synth.Tokens(*[as_rounds(t, n, n_tok)[:, :j].reshape(n * j, *t.shape[1:]) for t in tk.fields()])


def run_round(p, tk, n, n_tok, io, S_in, ring_in, separate=True, slots=None):
    kp = kda_params(p, io)
    d = [as_rounds(t, n, n_tok).to(DEV) for t in tk.fields()]
    S_in_d, ring_in_d = S_in.to(DEV), ring_in.to(DEV)
    S_out = torch.empty_like(S_in_d) if separate else None
    ring_out = torch.empty_like(ring_in_d) if separate else None
    if separate and slots is not None:
        S_out.copy_(S_in_d)
        ring_out.copy_(ring_in_d)
    o = kda.kda_decode_multi(kp, *d, S_in_d, ring_in_d, S_out=S_out, ring_out=ring_out,
                             slots=None if slots is None else torch.tensor(slots, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    S_res = S_in_d if S_out is None else S_out
    ring_res = ring_in_d if ring_out is None else ring_out
    return o.reshape(n * n_tok, -1), S_res, ring_res, S_in_d, ring_in_d


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_verify_round_matches_oracle_and_keeps_snapshot(io):
    n, n_tok = 3, 5
    p, tk, S0, ring0 = round_inputs(io, n, n_tok)
    o, S, ring, S_in_d, ring_in_d = run_round(p, tk, n, n_tok, io, S0, ring0)
    ref = oracle_run(p, tk, list(range(0, n * n_tok + 1, n_tok)), S_in=S0, ring_in=ring0)
    tol = tol_for(io)
    assert_close("o", o, ref["o"], tol)
    assert_close("S", S, ref["S"], tol)
    np.testing.assert_array_equal(ring.double().cpu().numpy(), ref["ring"])
    # the snapshot (inputs) is untouched
    assert torch.equal(S_in_d.cpu(), S0)
    assert torch.equal(ring_in_d.cpu(), ring0)


@pytest.mark.parametrize("keep", [1, 2, 4])
def test_rollback_replays_the_accepted_prefix(keep):
    io, n, n_tok = "bf16", 3, 5
    p, tk, S0, ring0 = round_inputs(io, n, n_tok, seed=31)
    run_round(p, tk, n, n_tok, io, S0, ring0)           # the full round, snapshot kept
    sub = first_tokens(tk, n, n_tok, keep)
    o, S, ring, _, _ = run_round(p, sub, n, keep, io, S0, ring0)
    ref = oracle_run(p, sub, list(range(0, n * keep + 1, keep)), S_in=S0, ring_in=ring0)
    tol = tol_for(io)
    assert_close("o", o, ref["o"], tol)
    assert_close("S", S, ref["S"], tol)
    np.testing.assert_array_equal(ring.double().cpu().numpy(), ref["ring"])


@pytest.mark.parametrize("n_tok, cuts", [(6, [2, 4]), (19, [3, 11])])
def test_round_equals_the_same_tokens_in_shorter_rounds(n_tok, cuts):
    """The in-kernel token loop carries state and ring exactly: a round of
    n_tok tokens (groups of 8, 8 and 3 for 19) equals, bit for bit, the same
    tokens cut into shorter rounds of two or more tokens, whatever the
    grouping inside each."""
    io, n = "bf16", 4
    p, tk, S0, ring0 = round_inputs(io, n, n_tok, seed=41)
    o_multi, S_multi, ring_multi, _, _ = run_round(p, tk, n, n_tok, io, S0, ring0, separate=False)
    kp = kda_params(p, io)
    S, ring = S0.to(DEV), ring0.to(DEV)
    rounds = [as_rounds(t, n, n_tok).to(DEV) for t in tk.fields()]
    edges = [0] + cuts + [n_tok]
    outs = [kda.kda_decode_multi(kp, *[x[:, lo:hi].contiguous() for x in rounds], S, ring)
            for lo, hi in zip(edges[:-1], edges[1:])]
    torch.cuda.synchronize()
    o_cut = torch.cat(outs, dim=1).reshape(n * n_tok, -1)
    assert torch.equal(o_multi, o_cut)
    assert torch.equal(S_multi, S)
    assert torch.equal(ring_multi, ring)


def test_round_matches_chained_single_token_decodes():
    """kda_decode one token at a time and a round over the same tokens agree
    to the bf16 tolerance (the two kernels sum over key rows in different
    orders)."""
    io, n, n_tok = "bf16", 4, 6
    p, tk, S0, ring0 = round_inputs(io, n, n_tok, seed=43)
    o_multi, S_multi, ring_multi, _, _ = run_round(p, tk, n, n_tok, io, S0, ring0, separate=False)
    kp = kda_params(p, io)
    S, ring = S0.to(DEV), ring0.to(DEV)
    rounds = [as_rounds(t, n, n_tok).to(DEV) for t in tk.fields()]
    outs = [kda.kda_decode(kp, *[x[:, t].contiguous() for x in rounds], S, ring) for t in range(n_tok)]
    torch.cuda.synchronize()
    o_single = torch.stack(outs, dim=1).reshape(n * n_tok, -1)
    tol = tol_for(io)
    assert_close("o", o_single.cpu(), o_multi.cpu().double().numpy(), tol)
    assert_close("S", S.cpu(), S_multi.cpu().double().numpy(), tol)
    assert torch.equal(ring_multi, ring)


def test_state_pool_slots():
    """Sessions mapped to pool slots: used slots advance, the others stay
    bit-identical, and an out-of-range slot skips its session."""
    io, n, n_tok, n_slots = "bf16", 3, 4, 6
    p, tk, _, _ = round_inputs(io, n, n_tok, seed=51)
    g = torch.Generator().manual_seed(52)
    S_pool = torch.randn(n_slots, 2, 128, 128, generator=g) * 0.05
    ring_pool = torch.randn(n_slots, 3, 3, 256, generator=g).to(torch.bfloat16)
    slots = [4, 0, 2]
    kp = kda_params(p, io)
    d = [as_rounds(t, n, n_tok).to(DEV) for t in tk.fields()]
    S_d, ring_d = S_pool.to(DEV), ring_pool.to(DEV)
    o = kda.kda_decode_multi(kp, *d, S_d, ring_d, slots=torch.tensor(slots, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    idx = torch.tensor(slots)
    ref = oracle_run(p, tk, list(range(0, n * n_tok + 1, n_tok)), S_in=S_pool[idx], ring_in=ring_pool[idx])
    tol = tol_for(io)
    assert_close("o", o.reshape(n * n_tok, -1), ref["o"], tol)
    assert_close("S", S_d.cpu()[idx], ref["S"], tol)
    np.testing.assert_array_equal(ring_d.cpu()[idx].double().numpy(), ref["ring"])
    for s in (1, 3, 5):
        assert torch.equal(S_d.cpu()[s], S_pool[s])
        assert torch.equal(ring_d.cpu()[s], ring_pool[s])
    # an out-of-range slot: that session's output rows, state and ring are untouched
    S_d2, ring_d2 = S_pool.to(DEV), ring_pool.to(DEV)
    o2 = torch.full_like(d[0], 7.0)
    kda.kda_decode_multi(kp, *d, S_d2, ring_d2, o=o2,
                         slots=torch.tensor([4, n_slots, 2], dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert torch.all(o2[1] == 7.0)
    assert torch.equal(S_d2.cpu()[0], S_pool[0])
    assert torch.equal(o2[0], o[0]) and torch.equal(o2[2], o[2])


def test_longest_round_f32():
    n_tok = kda.KDA_DECODE_MAX_TOKENS
    io, n = "f32", 2
    p, tk, S0, ring0 = round_inputs(io, n, n_tok, seed=61)
    o, S, ring, _, _ = run_round(p, tk, n, n_tok, io, S0, ring0)
    ref = oracle_run(p, tk, list(range(0, n * n_tok + 1, n_tok)), S_in=S0, ring_in=ring0)
    tol = tol_for(io)
    assert_close("o", o, ref["o"], tol)
    assert_close("S", S, ref["S"], tol)
    np.testing.assert_array_equal(ring.double().cpu().numpy(), ref["ring"])


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("n_tok", [1, 9, 17])
@pytest.mark.parametrize("gate_kind", [0, 1])
def test_round_lengths_across_groups_and_gates(io, n_tok, gate_kind):
    """Round lengths around the 8-token groups of the round kernel (9: a full
    group and a group of one; 17: two full groups and one) and one token (the
    one-token kernel), with the bounded and the softplus gate, against the
    oracle."""
    n = 2
    p, tk, S0, ring0 = round_inputs(io, n, n_tok, seed=71 + n_tok)
    p.gate_kind = gate_kind
    o, S, ring, _, _ = run_round(p, tk, n, n_tok, io, S0, ring0)
    ref = oracle_run(p, tk, list(range(0, n * n_tok + 1, n_tok)), S_in=S0, ring_in=ring0)
    tol = tol_for(io)
    assert_close("o", o, ref["o"], tol)
    assert_close("S", S, ref["S"], tol)
    np.testing.assert_array_equal(ring.double().cpu().numpy(), ref["ring"])
