"""The segmented recurrence (KDA_ALGO_CHUNKED_SEGMENTS): one sequence with few
heads runs its chunk recurrence as P segments whose affine maps S -> M S + B
are composed by a scan.  Checked against the single-pass schedule and the
oracle, on inputs with a long memory (a gate lower bound of -0.002 per token
and beta near 0.02), so that the starting state of every segment still
matters at its end."""
import numpy as np
import pytest
import torch

import gated_delta_rule_04_gb300 as kda
import kda_synth
from kda_testlib import assert_close, head_cols, kda_params, oracle_run, rel_l2, tol_for

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_04_gb300 import build as kbuild
    kbuild.build()
    kda.lib()


def _slow(p: kda_synth.Params) -> kda_synth.Params:
    p.gate_lower_bound = -0.002
    return p


def _tokens(T, H, seed):
    """Seeded tokens whose beta logits are shifted by -4 (beta ~ 0.02): the
    delta rule then removes little of the state per token."""
    tk = kda_synth.draw_tokens(T, H, seed, torch.bfloat16)
    tk.b = (tk.b.float() - 4.0).to(tk.b.dtype)
    return tk


@pytest.mark.parametrize("T, H, in_place", [(2048, 4, False), (4096 + 100, 8, True), (8192 + 37, 2, False)])
def test_segments_match_single_pass_and_oracle(T, H, in_place):
    io = "bf16"
    p = _slow(kda_synth.draw_params(H, 201))
    tk = _tokens(T, H, 202)
    g = torch.Generator().manual_seed(203)
    S0 = torch.randn(1, H, 128, 128, generator=g) * 0.05
    R0 = torch.randn(1, 3, 3, H * 128, generator=g).to(torch.bfloat16)
    cu = [0, T]
    d = [t.to(DEV) for t in tk.fields()]
    out = {}
    for algo in ("chunked", "chunked_segments"):
        kp = kda_params(p, io, algo=algo)
        assert kda.kda_prefill_algo(kp) == "chunked"
        ws = torch.empty(kda.kda_prefill_workspace_bytes(kp, 1, T), dtype=torch.uint8, device=DEV)
        S_in, ring_in = S0.to(DEV), R0.to(DEV)
        kw = dict(S_out=S_in, ring_out=ring_in) if in_place else {}
        o, S, ring = kda.kda_prefill(kp, *d, cu, S_in=S_in, ring_in=ring_in, workspace=ws, **kw)
        torch.cuda.synchronize()
        assert kda.kda_workspace_status(ws) == kda.KDA_OK
        out[algo] = (o.clone(), S.clone(), ring.clone())
    (o1, S1, r1), (o2, S2, r2) = out["chunked"], out["chunked_segments"]
    # the same records; only the order of the state products differs
    assert rel_l2(o2.double().cpu(), o1.double().cpu()) < 2e-3
    assert rel_l2(S2.double().cpu(), S1.double().cpu()) < 2e-3
    assert torch.equal(r1, r2)
    # the segmented schedule ran: its rounding differs from the single pass
    assert not torch.equal(S1, S2)
    heads = [0, H - 1]
    ref = oracle_run(p, tk, cu, S_in=S0, ring_in=R0, heads=heads)
    cols = head_cols(heads).to(DEV)
    tol = tol_for(io)
    assert_close("o", o2[:, cols], ref["o"], tol)
    assert_close("S", S2[:, heads], ref["S"], tol)
    np.testing.assert_array_equal(r2[..., cols].double().cpu().numpy(), ref["ring"])


def test_slow_gate_keeps_the_starting_state():
    """On these inputs the state 512 tokens (the shortest segment) on still
    depends on the state it started from: a segment that started from the
    wrong state would fail the oracle check."""
    T, H = 2048, 4
    p = _slow(kda_synth.draw_params(H, 201))
    tk = _tokens(T, H, 202)
    g = torch.Generator().manual_seed(203)
    S0 = torch.randn(1, H, 128, 128, generator=g) * 0.05
    a = oracle_run(p, tk, [0, T], S_in=S0, heads=[0])
    b = oracle_run(p, tk, [0, T], S_in=torch.zeros_like(S0), heads=[0])
    assert rel_l2(b["S"], a["S"]) > 0.1
    tail = slice(512, 640)
    assert rel_l2(b["o"][tail], a["o"][tail]) > 0.1


def test_segments_workspace_reserve():
    """The segmented schedule reserves its state slots in the workspace size
    (kda_prefill refuses a workspace one alignment unit short of it), and
    reports one window."""
    T, H, io = 4096, 8, "bf16"
    p = _slow(kda_synth.draw_params(H, 211))
    tk = _tokens(T, H, 212)
    kp_seg = kda_params(p, io, algo="chunked_segments")
    full = kda.kda_prefill_workspace_bytes(kp_seg, 1, T)
    # B_0..B_6, M_1..M_6 and X_2..X_7 for P = 8 segments of 8 heads
    assert full >= 19 * H * 128 * 128 * 4
    assert kda.kda_prefill_windows(kp_seg, 1, T, full) == 1
    d = [t.to(DEV) for t in tk.fields()]
    ws = torch.empty(full - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_prefill(kp_seg, *d, [0, T], workspace=ws)
    assert ei.value.status == kda.KDA_ERR_WORKSPACE


@pytest.mark.parametrize("H, T, auto_segments", [(8, 4096, True), (16, 32768, True), (32, 32768, False),
                                                 (8, 512, False), (32, 4096, True), (32, 8192 + 64, False),
                                                 (24, 16384, False)])
def test_auto_picks_segments(H, T, auto_segments):
    """kda_prefill with KDA_ALGO_AUTO runs one sequence as segments when at
    least five fit the SMs (2P - 3 CTAs per head, 8 chunks per segment), or
    three for 64 to 128 chunks; otherwise the overlapped windows where they
    apply."""
    p = kda_synth.draw_params(H, 221)
    auto = kda_params(p, "bf16", algo="auto")
    chunked = kda_params(p, "bf16", algo="chunked")
    big = 1 << 40
    if auto_segments:
        assert kda.kda_prefill_windows(auto, 1, T, big) == 1
        assert kda.kda_prefill_segments(auto, 1, T, big) >= 3
        assert kda.kda_prefill_segments(chunked, 1, T, big) == 0
        assert kda.kda_prefill_workspace_bytes(auto, 1, T) > kda.kda_prefill_workspace_bytes(chunked, 1, T)
    else:
        assert kda.kda_prefill_windows(auto, 1, T, big) == kda.kda_prefill_windows(chunked, 1, T, big)
        assert kda.kda_prefill_segments(auto, 1, T, big) == 0

