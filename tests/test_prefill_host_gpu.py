"""kda_prefill_host (inputs and output in host memory, token segments with
overlapped copies) against the fp64 oracle and against kda_prefill on the
device: segments that cut sequences anywhere (inside a chunk, inside the conv
window), empty sequences, nonzero initial state and ring, in place."""
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


def inputs(io, cu, H=2, seed=71, state=True):
    p = kda_synth.draw_params(H, seed)
    tk = kda_synth.draw_tokens(cu[-1], H, seed + 1, kda_synth.io_dtype(io))
    n = len(cu) - 1
    g = torch.Generator().manual_seed(seed + 2)
    S0 = torch.randn(n, H, 128, 128, generator=g) * 0.05 if state else None
    ring0 = torch.randn(n, 3, 3, H * 128, generator=g).to(kda_synth.io_dtype(io)) if state else None
    return p, tk, S0, ring0


def run_host(p, tk, cu, io, seg, S0, ring0, in_place=False, algo="auto"):
    kp = kda_params(p, io, algo)
    host = [t.pin_memory() for t in tk.fields()]
    S_in = None if S0 is None else S0.to(DEV)
    ring_in = None if ring0 is None else ring0.to(DEV)
    kw = dict(S_out=S_in, ring_out=ring_in) if in_place else {}
    stream = torch.cuda.Stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    o, S, ring = kda.kda_prefill_host(kp, *host, cu, S_in=S_in, ring_in=ring_in, segment_tokens=seg,
                                      stream=stream, h2d_stream=h2d, d2h_stream=d2h, **kw)
    stream.synchronize()
    return o, S, ring


@pytest.mark.parametrize("io, cu, seg", [
    ("bf16", [0, 300], 100),                       # segments cut inside a chunk
    ("bf16", [0, 70, 70, 200, 331, 333], 64),      # empty and 2-token sequences, cuts inside the conv window
    ("bf16", [0, 130, 260], 1),                    # one token per segment
    ("bf16", [0, 257], 1000),                      # one segment
    ("f32", [0, 90, 200], 37),                     # scan path
])
def test_host_prefill_matches_oracle(io, cu, seg):
    p, tk, S0, ring0 = inputs(io, cu)
    o, S, ring = run_host(p, tk, cu, io, seg, S0, ring0)
    ref = oracle_run(p, tk, cu, S_in=S0, ring_in=ring0)
    tol = tol_for(io)
    assert_close("o", o, ref["o"], tol)
    assert_close("S", S, ref["S"], tol)
    np.testing.assert_array_equal(ring.double().cpu().numpy(), ref["ring"])


def test_host_prefill_softplus_gate_matches_oracle():
    """The unbounded softplus gate through the host-buffer prefill (each
    segment on the chunked form), cuts inside chunks."""
    io, cu = "bf16", [0, 70, 300, 301]
    p, tk, S0, ring0 = inputs(io, cu, seed=85)
    p.gate_kind = 1
    o, S, ring = run_host(p, tk, cu, io, 100, S0, ring0)
    ref = oracle_run(p, tk, cu, S_in=S0, ring_in=ring0)
    tol = tol_for(io)
    assert_close("o", o, ref["o"], tol)
    assert_close("S", S, ref["S"], tol)
    np.testing.assert_array_equal(ring.double().cpu().numpy(), ref["ring"])


def test_host_prefill_segments_that_run_as_segmented_recurrences():
    """Host segments of 4096 tokens of one 8192-token sequence with 32 heads:
    each runs its recurrence as 3 segments (affine maps composed by a scan);
    sampled heads against the oracle."""
    io, cu, H = "bf16", [0, 8192], 32
    p, tk, S0, ring0 = inputs(io, cu, H=H, seed=89)
    kp = kda_params(p, io)
    assert kda.kda_prefill_segments(kp, 1, 4096, 1 << 40) == 3
    o, S, ring = run_host(p, tk, cu, io, 4096, S0, ring0)
    heads = [0, 31]
    ref = oracle_run(p, tk, cu, S_in=S0, ring_in=ring0, heads=heads)
    cols = head_cols(heads)
    tol = tol_for(io)
    assert_close("o", o[:, cols], ref["o"], tol)
    assert_close("S", S[:, heads], ref["S"], tol)
    np.testing.assert_array_equal(ring[..., cols].double().cpu().numpy(), ref["ring"])


def test_host_prefill_in_place_zero_start():
    """No initial state or ring (zeros), and the in-place form."""
    io, cu = "bf16", [0, 150, 400]
    p, tk, S0, ring0 = inputs(io, cu, seed=81)
    o, S, ring = run_host(p, tk, cu, io, 96, None, None)
    ref = oracle_run(p, tk, cu)
    tol = tol_for(io)
    assert_close("o", o, ref["o"], tol)
    assert_close("S", S, ref["S"], tol)
    np.testing.assert_array_equal(ring.double().cpu().numpy(), ref["ring"])
    o2, S2, ring2 = run_host(p, tk, cu, io, 96, S0, ring0, in_place=True)
    ref2 = oracle_run(p, tk, cu, S_in=S0, ring_in=ring0)
    assert_close("o", o2, ref2["o"], tol)
    assert_close("S", S2, ref2["S"], tol)
    np.testing.assert_array_equal(ring2.double().cpu().numpy(), ref2["ring"])


def test_host_prefill_segment_on_chunk_grid_equals_device_prefill():
    """Segments of whole 64-token chunks inside one sequence keep the chunk
    grid of a single kda_prefill call, so the two results agree to the last
    bit."""
    io, cu, H = "bf16", [0, 1024], 4
    p, tk, S0, ring0 = inputs(io, cu, H=H, seed=91)
    o, S, ring = run_host(p, tk, cu, io, 256, S0, ring0)
    kp = kda_params(p, io)
    o_d, S_d, ring_d = kda.kda_prefill(kp, *[t.to(DEV) for t in tk.fields()], cu, S_in=S0.to(DEV),
                                       ring_in=ring0.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(o, o_d.cpu())
    assert torch.equal(S.cpu(), S_d.cpu())
    assert torch.equal(ring.cpu(), ring_d.cpu())


def test_host_prefill_status_word_is_clear():
    io, cu = "bf16", [0, 500]
    p, tk, S0, ring0 = inputs(io, cu, seed=95)
    kp = kda_params(p, io)
    scratch = torch.empty(kda.kda_prefill_host_scratch_bytes(kp, cu, 128), dtype=torch.uint8, device=DEV)
    kda.kda_prefill_host(kp, *[t.pin_memory() for t in tk.fields()], cu, segment_tokens=128, scratch=scratch)
    assert kda.kda_workspace_status(scratch) == kda.KDA_OK


def test_host_prefill_segments_that_run_as_windows():
    """Segments long enough to run as overlapped windows (2560 tokens, 8
    heads), on the chunk grid: bit-identical to one kda_prefill of the whole
    sequence, and the oracle on one head."""
    io, cu, H = "bf16", [0, 5120], 8
    p, tk, S0, ring0 = inputs(io, cu, H=H, seed=97)
    kp = kda_params(p, io, "chunked")   # (auto would run 8 heads as segments)
    assert kda.kda_prefill_windows(kp, 1, 2560, 1 << 40) >= 2
    o, S, ring = run_host(p, tk, cu, io, 2560, S0, ring0, algo="chunked")
    o_d, S_d, ring_d = kda.kda_prefill(kp, *[t.to(DEV) for t in tk.fields()], cu, S_in=S0.to(DEV),
                                       ring_in=ring0.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(o, o_d.cpu())
    assert torch.equal(S.cpu(), S_d.cpu())
    assert torch.equal(ring.cpu(), ring_d.cpu())
    ref = oracle_run(p, tk, cu, S_in=S0, ring_in=ring0, heads=[3])
    cols = head_cols([3])
    tol = tol_for(io)
    assert_close("o", o[:, cols], ref["o"], tol)
    assert_close("S", S[:, [3]], ref["S"], tol)
