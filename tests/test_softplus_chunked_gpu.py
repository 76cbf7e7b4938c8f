"""The unbounded softplus gate g = -e^A softplus(z + dt_bias) on the chunked
tensor-core form (bf16 I/O): the diagonal 16 x 16 blocks of A and P are
summed position by position, every other factor is one exponential of a
non-positive exponent.  Checked against the fp64 oracle on inputs whose
per-token log decay reaches -60 to -80, so that a 16-token sub-tile spans
e^-600 and more (far outside fp32 for any factorisation through one
reference point), and against
the fp32 scan of the same gate."""
import math

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


def softplus_params(H, seed, dt_shift=0.0, dt_scale=None):
    p = kda_synth.draw_params(H, seed)
    p.gate_kind = 1
    if dt_scale is not None:
        g = torch.Generator().manual_seed(seed + 7)
        p.dt_bias = torch.randn(p.dt_bias.shape, generator=g) * dt_scale
    p.dt_bias = p.dt_bias + dt_shift
    return p


def run(p, tk, cu, algo="auto", S_in=None, ring_in=None):
    kp = kda_params(p, "bf16", algo)
    d = [t.to(DEV) for t in tk.fields()]
    o, S, ring = kda.kda_prefill(kp, *d, cu, S_in=None if S_in is None else S_in.to(DEV),
                                 ring_in=None if ring_in is None else ring_in.to(DEV))
    torch.cuda.synchronize()
    return o, S, ring


def check(p, tk, cu, o, S, ring, S_in=None, ring_in=None, heads=None):
    ref = oracle_run(p, tk, cu, S_in=S_in, ring_in=ring_in, heads=heads)
    tol = tol_for("bf16")
    if heads is not None:
        cols = head_cols(heads).to(o.device)
        o, S, ring = o[:, cols], S[:, torch.tensor(heads, device=S.device)], ring[..., cols]
    assert_close("o", o, ref["o"], tol)
    assert_close("S", S, ref["S"], tol)
    np.testing.assert_array_equal(ring.double().cpu().numpy(), ref["ring"])
    return ref


@pytest.mark.parametrize("name, dt_shift, dt_scale", [
    ("drawn", 0.0, None),          # e^A in [1, 16]: g from about -0.02 to -40 per token
    ("strong", 3.0, None),         # g from about -0.3 to -63
    ("mixed", -2.0, 4.0),          # per channel from almost no decay to about -80
])
def test_softplus_chunked_varlen_vs_oracle(name, dt_shift, dt_scale):
    lens = [70, 3, 131, 64, 1, 200, 0, 65]
    H = 2
    p = softplus_params(H, 301, dt_shift, dt_scale)
    cu = kda_synth.cumsum0(lens)
    tk = kda_synth.draw_tokens(cu[-1], H, 302, torch.bfloat16)
    g = torch.Generator().manual_seed(303)
    n = len(lens)
    S_in = torch.randn(n, H, 128, 128, generator=g) * 0.05
    ring_in = torch.randn(n, 3, 3, H * 128, generator=g).to(torch.bfloat16)
    assert kda.kda_prefill_algo(kda_params(p, "bf16")) == "chunked"
    o, S, ring = run(p, tk, cu, S_in=S_in, ring_in=ring_in)
    check(p, tk, cu, o, S, ring, S_in=S_in, ring_in=ring_in)


def test_softplus_strong_decay_spans_beyond_fp32():
    """The inputs of the 'strong' case do reach decays that no single
    reference point could hold: some 16-token sub-tile has a channel whose
    cumulative log decay is below -88 (e^-88 is the smallest normal fp32)."""
    p = softplus_params(2, 301, 3.0)
    tk = kda_synth.draw_tokens(64, 2, 302, torch.bfloat16)
    z = tk.z.float()[:16]
    x = z + p.dt_bias[None, :]
    g = -torch.exp(p.A_log).repeat_interleave(128)[None, :] * torch.nn.functional.softplus(x)
    assert float(g.sum(0).min()) < -88.0


def test_softplus_chunked_equals_scan():
    """Chunked form and fp32 scan of the same gate and inputs agree to the
    bf16 tolerance (they share no kernel)."""
    lens = [300, 64, 17]
    H = 4
    p = softplus_params(H, 311)
    cu = kda_synth.cumsum0(lens)
    tk = kda_synth.draw_tokens(cu[-1], H, 312, torch.bfloat16)
    oc, Sc, rc = run(p, tk, cu, algo="chunked")
    os_, Ss, rs = run(p, tk, cu, algo="scan")
    assert rel_l2(oc.double().cpu(), os_.double().cpu()) < 1e-2
    assert rel_l2(Sc.double().cpu(), Ss.double().cpu()) < 1e-2
    assert torch.equal(rc, rs)


def test_softplus_chunked_long_sequence_sampled_heads():
    """One sequence of T = 4096 with 32 heads (overlapped windows and the
    multi-sub-tile chunk grid), sampled heads against the oracle."""
    T, H = 4096, 32
    p = softplus_params(H, 321)
    tk = kda_synth.draw_tokens(T, H, 322, torch.bfloat16)
    cu = [0, T]
    o, S, ring = run(p, tk, cu)
    assert torch.isfinite(o.float()).all()
    check(p, tk, cu, o, S, ring, heads=[0, 17, 31])


def test_softplus_chunked_segments_vs_oracle():
    """A few-head sequence that AUTO runs as segments, with the softplus gate."""
    T, H = 4096 + 64, 4
    p = softplus_params(H, 331, -6.0)   # weak decay: g about -0.01 to -0.07 per token
    tk = kda_synth.draw_tokens(T, H, 332, torch.bfloat16)
    g = torch.Generator().manual_seed(333)
    S_in = torch.randn(1, H, 128, 128, generator=g) * 0.05
    kp = kda_params(p, "bf16")
    assert kda.kda_prefill_windows(kp, 1, T, 1 << 40) == 1
    o, S, ring = run(p, tk, [0, T], S_in=S_in)
    check(p, tk, [0, T], o, S, ring, S_in=S_in, heads=[1, 3])
    assert math.isfinite(float(S.abs().max()))


def test_softplus_chunked_windows_vs_oracle():
    """The softplus gate under the overlapped windows (one sequence of 8256
    tokens, 8 heads, KDA_ALGO_CHUNKED), sampled heads against the oracle."""
    T, H = 8192 + 64, 8
    p = softplus_params(H, 341)
    tk = kda_synth.draw_tokens(T, H, 342, torch.bfloat16)
    kp = kda_params(p, "bf16", algo="chunked")
    assert kda.kda_prefill_windows(kp, 1, T, kda.kda_prefill_workspace_bytes(kp, 1, T)) >= 2
    o, S, ring = run(p, tk, [0, T], algo="chunked")
    check(p, tk, [0, T], o, S, ring, heads=[0, 7])

