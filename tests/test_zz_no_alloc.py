"""kda_prefill_noalloc: the prefill for callers that cannot allocate device
memory while they run (for example a plugin inside an engine that owns all
device memory, or a serving loop that must not call cudaMalloc/cudaFree
because they can synchronise the whole device).

The entry point is called through the C ABI and must give the same results
as kda_prefill, within the tolerances of the other parity tests, on two calls
in a row (the second sees the scratch the first one left behind), and match
the fp64 oracle by itself.  A bounded-wait timeout inside it is read back with
kda_noalloc_status.

This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import gated_delta_rule_04_gb300 as kda
import kda_synth
from kda_testlib import assert_close, kda_params, oracle_run, tol_for

pytestmark = pytest.mark.gpu
DEV = "cuda"
_vp = ctypes.c_void_p


def noalloc_fn():
    from gated_delta_rule_04_gb300 import build as kbuild
    kbuild.build()
    L = kda.lib()
    f = L.kda_prefill_noalloc
    f.argtypes = ([ctypes.POINTER(kda.kda_params)] + [_vp] * 6 + [ctypes.POINTER(ctypes.c_int64),
                  ctypes.c_int32, ctypes.c_int64] + [_vp] * 5 + [_vp])
    f.restype = ctypes.c_int
    return f


def call_noalloc(f, kp, tokens, cu, S_in=None, ring_in=None):
    n = len(cu) - 1
    T = cu[-1]
    H = kp.num_heads
    q = tokens[0]
    o = torch.empty_like(q)
    S_out = torch.empty(n, H, 128, 128, device=DEV)
    ring_out = torch.empty(n, 3, 3, H * 128, dtype=q.dtype, device=DEV)
    arr = (ctypes.c_int64 * len(cu))(*cu)
    ptr = lambda t: None if t is None else t.data_ptr()
    st = f(kp.ref, *[t.data_ptr() for t in tokens], arr, n, T, ptr(S_in), S_out.data_ptr(),
           ptr(ring_in), ring_out.data_ptr(), o.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return st, o, S_out, ring_out


@pytest.mark.parametrize("io, algo, gate_kind", [("bf16", "auto", 0), ("f32", "scan", 0), ("bf16", "auto", 1)])
def test_noalloc_matches_kda_prefill_twice(io, algo, gate_kind):
    f = noalloc_fn()
    H = 4
    p = kda_synth.draw_params(H, 21)
    p.gate_kind = gate_kind   # 1: the softplus gate (chunked form with bf16 I/O)
    kp = kda_params(p, io, algo)
    g = torch.Generator().manual_seed(22)
    cases = [[130, 7, 64], [3, 200, 1, 65]]  # second call: other shapes, nonzero state and ring
    for call, lens in enumerate(cases):
        cu = kda_synth.cumsum0(lens)
        tk = [t.to(DEV) for t in kda_synth.draw_tokens(cu[-1], H, 23 + call, kda_synth.io_dtype(io)).fields()]
        S_in = ring_in = None
        if call == 1:
            S_in = (torch.randn(len(lens), H, 128, 128, generator=g) * 0.05).to(DEV)
            ring_in = torch.randn(len(lens), 3, 3, H * 128, generator=g).to(kda_synth.io_dtype(io)).to(DEV)
        st, o, S, ring = call_noalloc(f, kp, tk, cu, S_in, ring_in)
        assert st == kda.KDA_OK, kda.kda_status_str(st)
        o_ref, S_ref, ring_ref = kda.kda_prefill(kp, *tk, cu, S_in=S_in, ring_in=ring_in)
        torch.cuda.synchronize()
        tol = tol_for(io)
        assert_close(f"call {call} o", o, o_ref.double().cpu().numpy(), tol)
        assert_close(f"call {call} S", S, S_ref.double().cpu().numpy(), tol)
        assert torch.equal(ring, ring_ref)
        # and against the oracle, independently of kda_prefill
        ref = oracle_run(p, kda_synth.Tokens(*[t.cpu() for t in tk]), cu,
                         S_in=None if S_in is None else S_in.cpu(), ring_in=None if ring_in is None else ring_in.cpu())
        assert_close(f"call {call} o vs oracle", o, ref["o"], tol)
        assert_close(f"call {call} S vs oracle", S, ref["S"], tol)
        np.testing.assert_array_equal(ring.double().cpu().numpy(), ref["ring"])


def test_noalloc_rejects_problems_beyond_its_scratch():
    f = noalloc_fn()
    H = 32
    p = kda_synth.draw_params(H, 24)
    kp = kda_params(p, "bf16")
    T = 4096  # needs about 0.4 GB of scratch, far beyond the fixed array
    need = kda.kda_prefill_workspace_bytes(kp, 1, T)
    assert need > 64 << 20
    x = torch.empty(T, H * 128, dtype=torch.bfloat16, device=DEV)
    bb = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    st, *_ = call_noalloc(f, kp, [x, x, x, x, bb, x], [0, T])
    assert st == kda.KDA_ERR_WORKSPACE
    np.testing.assert_equal(st, kda.KDA_ERR_WORKSPACE)


def test_noalloc_status_reports_a_timeout_then_ok():
    """With the test hook that shortens the chunk preparation's pipeline waits
    to 1 us, a call through the no-allocation entry point times out;
    kda_noalloc_status reports it and clears the word; a normal call then
    succeeds."""
    f = noalloc_fn()
    L = kda.lib()
    L.kda_noalloc_status.argtypes = [_vp]
    L.kda_noalloc_status.restype = ctypes.c_int
    H = 1
    p = kda_synth.draw_params(H, 25)
    cu = [0, 128]
    tk = [t.to(DEV) for t in kda_synth.draw_tokens(128, H, 26, torch.bfloat16).fields()]
    stream = torch.cuda.current_stream().cuda_stream
    st, *_ = call_noalloc(f, kda_params(p, "bf16", wait_limit_us=1), tk, cu)
    assert st == kda.KDA_OK
    assert L.kda_noalloc_status(stream) == kda.KDA_ERR_TIMEOUT
    st, o, S, ring = call_noalloc(f, kda_params(p, "bf16"), tk, cu)
    assert st == kda.KDA_OK
    assert L.kda_noalloc_status(stream) == kda.KDA_OK
    ref = oracle_run(p, kda_synth.Tokens(*[t.cpu() for t in tk]), cu)
    assert_close("o", o, ref["o"], tol_for("bf16"))
