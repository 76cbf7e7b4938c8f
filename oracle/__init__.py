"""fp64 CPU oracle of the KDA mixer core -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library and its Python binding never
do; the two implementations share no code.

The arithmetic lives in ``kda_oracle.c`` (plain C, double precision, token by
token); this module only marshals numpy arrays through ctypes.  Each entry
point states the passage it follows:

* ``mixer``  -- the whole layer core: short conv + SiLU, q/k L2 norm, q scale,
  lower-bounded gate (or the earlier Kimi-Linear softplus gate), beta, gated
  delta recurrence, RMSNormGated
  ("Kimi Delta Attention (KDA) -- analysis & C kernel plan", sections
  "The KDA layer, precisely" and "Recurrence"; "ferrox-models 0.8.0, module
  kda", module overview; "Kimi K3 - Retention gate", gate.py excerpt).
* ``core``   -- the recurrence alone on transformed inputs (section
  "Recurrence" of the KDA analysis page).
* ``chunked_core`` -- the chunked (UT transform, per-channel cumulative log
  gate) form of the same recurrence, with sub-tile reference points
  ("memra-engine 0.124.0, module kda", PREFILL DISPATCH; "Kimi K3 - Retention
  gate", section "Why").
* ``rmsnorm_gated`` -- the output norm alone.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


class _Params(ctypes.Structure):
    _fields_ = [
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("gate_lower_bound", ctypes.c_double),
        ("l2_eps", ctypes.c_double),
        ("norm_eps", ctypes.c_double),
        ("q_scale", ctypes.c_double),
        ("conv_w", _dp),
        ("A_log", _dp),
        ("dt_bias", _dp),
        ("norm_w", _dp),
        ("gate_kind", ctypes.c_int32),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/libkda_oracle.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i32, i64 = ctypes.c_int, ctypes.c_int64
        lib.kdao_core.argtypes = [i32, i32, i32] + [_dp] * 8 + [i32]
        lib.kdao_core.restype = i32
        lib.kdao_chunked_core.argtypes = [i32, i32, i32, i32, i32] + [_dp] * 8 + [i32]
        lib.kdao_chunked_core.restype = i32
        lib.kdao_mixer.argtypes = (
            [ctypes.POINTER(_Params), i32, ctypes.POINTER(ctypes.c_int64)] + [_dp] * 17 + [i32]
        )
        lib.kdao_mixer.restype = i32
        lib.kdao_rmsnorm_gated.argtypes = [i64, i32, i32, ctypes.c_double] + [_dp] * 4
        lib.kdao_rmsnorm_gated.restype = i32
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


@dataclass
class Params:
    """Mixer parameters (float64 numpy arrays).

    conv_w [3][H*D][4] (planes q, k, v; tap 3 weighs the current token),
    A_log [H], dt_bias [H*D], norm_w [D].
    """

    num_heads: int
    head_dim: int
    conv_w: np.ndarray
    A_log: np.ndarray
    dt_bias: np.ndarray
    norm_w: np.ndarray
    gate_lower_bound: float = -5.0
    l2_eps: float = 1e-6
    norm_eps: float = 1e-5
    q_scale: float = 0.0
    gate_kind: int = 0  # 0: lower-bounded sigmoid gate; 1: -exp(A_log) softplus(z + dt_bias)

    def _c(self):
        self._keep = [_f64(self.conv_w), _f64(self.A_log), _f64(self.dt_bias), _f64(self.norm_w)]
        cw, al, db, nw = self._keep
        return _Params(
            self.num_heads, self.head_dim, self.gate_lower_bound, self.l2_eps, self.norm_eps,
            self.q_scale, _ptr(cw), _ptr(al), _ptr(db), _ptr(nw), int(self.gate_kind),
        )


def core(q, k, v, g, beta, S0=None, nthreads=None):
    """Recurrence on transformed inputs.  q,k,v,g [T][H][D]; beta [T][H];
    S0 [H][D][D] (key rows) or None.  Returns (o [T][H][D], S [H][D][D])."""
    q, k, v, g, beta, S0 = map(_f64, (q, k, v, g, beta, S0))
    T, H, D = q.shape
    o = np.zeros((T, H, D))
    S = np.zeros((H, D, D))
    rc = _load().kdao_core(T, H, D, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0),
                           _ptr(S), _ptr(o), nthreads or default_threads())
    if rc:
        raise ValueError("kdao_core rejected its arguments")
    return o, S


def chunked_core(q, k, v, g, beta, S0=None, chunk=64, subtile=16, nthreads=None):
    """Chunked form of ``core`` (same arguments, chunk size ``chunk``)."""
    q, k, v, g, beta, S0 = map(_f64, (q, k, v, g, beta, S0))
    T, H, D = q.shape
    o = np.zeros((T, H, D))
    S = np.zeros((H, D, D))
    rc = _load().kdao_chunked_core(T, H, D, chunk, subtile, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                   _ptr(beta), _ptr(S0), _ptr(S), _ptr(o),
                                   nthreads or default_threads())
    if rc:
        raise ValueError("kdao_chunked_core rejected its arguments")
    return o, S


def mixer(params: Params, cu_seqlens, q, k, v, z, b, gout, S_in=None, ring_in=None,
          intermediates=False, nthreads=None):
    """Whole mixer core over packed varlen tokens.

    q,k,v,z,gout [T][H*D] raw (pre-conv) inputs; b [T][H]; cu_seqlens [n+1];
    S_in [n][H][D][D] or None (zero); ring_in [n][3][3][H*D] or None (zero).
    Returns dict with o, S, ring and, when ``intermediates``, qh, kh, vh, g,
    beta, o_core.
    """
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    n = cu.shape[0] - 1
    q, k, v, z, b, gout, S_in, ring_in = map(_f64, (q, k, v, z, b, gout, S_in, ring_in))
    H, D = params.num_heads, params.head_dim
    W = H * D
    T = q.shape[0]
    o = np.zeros((T, W))
    S = np.zeros((n, H, D, D))
    ring = np.zeros((n, 3, 3, W))
    inter = {}
    if intermediates:
        for name, shape in (("qh", (T, W)), ("kh", (T, W)), ("vh", (T, W)), ("g", (T, W)),
                            ("beta", (T, H)), ("o_core", (T, W))):
            inter[name] = np.zeros(shape)
    cp = params._c()
    rc = _load().kdao_mixer(
        ctypes.byref(cp), n, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(b), _ptr(gout), _ptr(S_in), _ptr(S),
        _ptr(ring_in), _ptr(ring), _ptr(o),
        _ptr(inter.get("qh")), _ptr(inter.get("kh")), _ptr(inter.get("vh")),
        _ptr(inter.get("g")), _ptr(inter.get("beta")), _ptr(inter.get("o_core")),
        nthreads or default_threads(),
    )
    if rc:
        raise ValueError("kdao_mixer rejected its arguments")
    out = {"o": o, "S": S, "ring": ring}
    out.update(inter)
    return out


def rmsnorm_gated(x, gate, w, num_heads, eps=1e-5):
    """RMSNormGated over [rows][H*D]: x / sqrt(mean_i x^2 + eps) * w[i] * sigmoid(gate)."""
    x, gate, w = map(_f64, (x, gate, w))
    rows = x.shape[0]
    D = w.shape[0]
    o = np.zeros_like(x)
    _load().kdao_rmsnorm_gated(rows, num_heads, D, eps, _ptr(x), _ptr(gate), _ptr(w), _ptr(o))
    return o


def run_synth(p, tokens, cu, S_in=None, ring_in=None, heads=None, intermediates=False, nthreads=None):
    """``mixer`` on the seeded inputs of ``kda_synth`` (a ``kda_synth.Params``
    and ``kda_synth.Tokens``, torch tensors on any device), on all heads or on
    the subset ``heads`` (heads are independent).  S_in / ring_in are the
    full-width tensors or None.  Marshalling only: every step of the
    arithmetic is in ``mixer``."""
    import torch

    def arr(t):
        return None if t is None else t.detach().to("cpu").double().numpy()

    if heads is not None:
        p = p.head_slice(heads)
        tokens = tokens.head_slice(heads)
        idx = torch.tensor(heads, dtype=torch.long)
        if S_in is not None:
            S_in = S_in[:, idx.to(S_in.device)]
        if ring_in is not None:
            ch = (idx[:, None] * p.head_dim + torch.arange(p.head_dim)[None, :]).reshape(-1).to(ring_in.device)
            ring_in = ring_in[..., ch]
    op = Params(p.num_heads, p.head_dim, arr(p.conv_w), arr(p.A_log), arr(p.dt_bias), arr(p.norm_w),
                p.gate_lower_bound, p.l2_eps, p.norm_eps, p.q_scale, p.gate_kind)
    return mixer(op, cu, *[arr(t) for t in tokens.fields()], S_in=arr(S_in), ring_in=arr(ring_in),
                 intermediates=intermediates, nthreads=nthreads)
