"""Shared helpers of the parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import kda_synth
import oracle

TOL_F32 = dict(rel=1e-4, maxabs=None)
TOL_BF16 = dict(rel=2e-2, maxabs=5e-2)


def tol_for(io: str):
    return TOL_F32 if io == "f32" else TOL_BF16


def rel_l2(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def assert_close(name, got, want, tol):
    got = got.double().cpu().numpy() if hasattr(got, "cpu") else np.asarray(got)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    r = rel_l2(got, want)
    assert r <= tol["rel"], f"{name}: rel-L2 {r:.3e} > {tol['rel']}"
    if tol.get("maxabs") is not None:
        m = float(np.max(np.abs(got - want))) if got.size else 0.0
        assert m <= tol["maxabs"], f"{name}: max-abs {m:.3e} > {tol['maxabs']}"
    return r


def kda_params(p: kda_synth.Params, io: str, algo: str = "auto", device="cuda", wait_limit_us: int = 0):
    import gated_delta_rule_04_gb300 as kda
    return kda.make_params(p.conv_w.to(device), p.A_log.to(device), p.dt_bias.to(device),
                           p.norm_w.to(device), io_dtype=io, algo=algo,
                           gate_lower_bound=p.gate_lower_bound, l2_eps=p.l2_eps,
                           norm_eps=p.norm_eps, q_scale=p.q_scale,
                           gate=("bounded", "softplus")[p.gate_kind], wait_limit_us=wait_limit_us)


def oracle_run(p: kda_synth.Params, tokens: kda_synth.Tokens, cu, S_in=None, ring_in=None,
               heads=None, intermediates=False):
    """Oracle on all heads, or on the subset ``heads`` (heads are independent).
    S_in / ring_in are full-width tensors (or None)."""
    return oracle.run_synth(p, tokens, cu, S_in=S_in, ring_in=ring_in, heads=heads,
                            intermediates=intermediates)


def head_cols(heads):
    return torch.tensor([h * 128 + i for h in heads for i in range(128)], dtype=torch.long)
