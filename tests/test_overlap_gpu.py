"""kda_prefill's overlapped windows (one long sequence whose recurrence leaves
SMs idle): the same bytes as the single pass, which kda_prefill runs when it
is given stage events, and the oracle on a head."""
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


@pytest.mark.parametrize("T, in_place", [(2048, False), (4096 + 100, True), (16384, False), (16384 + 4000, True)])
def test_windows_equal_single_pass(T, in_place):
    H, io = 8, "bf16"
    p = kda_synth.draw_params(H, 101)
    tk = kda_synth.draw_tokens(T, H, 102, torch.bfloat16)
    g = torch.Generator().manual_seed(103)
    S0 = torch.randn(1, H, 128, 128, generator=g) * 0.05
    R0 = torch.randn(1, 3, 3, H * 128, generator=g).to(torch.bfloat16)
    kp = kda_params(p, io, "chunked")   # (auto would run 8 heads as segments)
    cu = [0, T]
    ws = torch.empty(kda.kda_prefill_workspace_bytes(kp, 1, T), dtype=torch.uint8, device=DEV)
    assert kda.kda_prefill_windows(kp, 1, T, ws.numel()) >= 2
    d = [t.to(DEV) for t in tk.fields()]
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(kda.KDA_PREFILL_EVENTS)]
    results = []
    for stage_events in (None, evs):
        S_in, ring_in = S0.to(DEV), R0.to(DEV)
        kw = dict(S_out=S_in, ring_out=ring_in) if in_place else {}
        o, S, ring = kda.kda_prefill(kp, *d, cu, S_in=S_in, ring_in=ring_in, workspace=ws,
                                     stage_events=stage_events, **kw)
        torch.cuda.synchronize()
        results.append((o.clone(), S.clone(), ring.clone()))
    assert kda.kda_workspace_status(ws) == kda.KDA_OK
    (o1, S1, r1), (o2, S2, r2) = results
    assert torch.equal(o1, o2)
    assert torch.equal(S1, S2)
    assert torch.equal(r1, r2)
    ref = oracle_run(p, tk, cu, S_in=S0, ring_in=R0, heads=[5])
    cols = head_cols([5]).to(DEV)
    tol = tol_for(io)
    assert_close("o", o1[:, cols], ref["o"], tol)
    assert_close("S", S1[:, [5]], ref["S"], tol)
    np.testing.assert_array_equal(r1[..., cols].double().cpu().numpy(), ref["ring"])
