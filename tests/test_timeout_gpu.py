"""The bounded-wait timeout path of the chunk preparation, made to run out on
purpose without faulting or hanging anything.

Every in-kernel wait gives up after a limit; the kernel then records
KDA_ERR_TIMEOUT in the workspace's error word, lets its own copies and
tensor-core work finish, frees its tensor memory and returns.  The test hook
``wait_limit_us`` of kda_params shortens the limit of the waits between the
chunk preparation's two warp groups to one microsecond (an item takes several),
so the first hand-off wait runs out.  kda_workspace_status must report the
timeout; a normal call on the same workspace must then succeed and match the
oracle.
"""
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


@pytest.mark.parametrize("lens", [[128], [64, 200, 3]])
def test_pipeline_wait_timeout_is_reported_then_a_normal_call_recovers(lens):
    H = 1
    p = kda_synth.draw_params(H, 31)
    cu = kda_synth.cumsum0(lens)
    tk = kda_synth.draw_tokens(cu[-1], H, 32, torch.bfloat16)
    d = [t.to(DEV) for t in tk.fields()]
    short = kda_params(p, "bf16", wait_limit_us=1)
    assert kda.kda_prefill_algo(short) == "chunked"
    ws = torch.empty(kda.kda_prefill_workspace_bytes(short, len(lens), cu[-1]), dtype=torch.uint8, device=DEV)
    kda.kda_prefill(short, *d, cu, workspace=ws)
    torch.cuda.synchronize()
    assert kda.kda_workspace_status(ws) == kda.KDA_ERR_TIMEOUT
    # the status read cleared the word; the context is still usable
    normal = kda_params(p, "bf16")
    o, S, ring = kda.kda_prefill(normal, *d, cu, workspace=ws)
    torch.cuda.synchronize()
    assert kda.kda_workspace_status(ws) == kda.KDA_OK
    ref = oracle_run(p, tk, cu)
    tol = tol_for("bf16")
    assert_close("o", o, ref["o"], tol)
    assert_close("S", S, ref["S"], tol)
    np.testing.assert_array_equal(ring.double().cpu().numpy(), ref["ring"])
