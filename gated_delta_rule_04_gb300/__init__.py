"""Python binding of the GB300 KDA mixer-core library (``libkda.so``).

Argument marshalling only: every step of the mixer runs in the CUDA kernels
behind the C ABI declared in ``include/kda.h``; PyTorch supplies device
memory and the stream.  The functions carry the C names:

    kda_prefill_algo, kda_prefill_workspace_bytes, kda_prefill_windows, kda_prefill_segments, kda_prefill,
    kda_prefill_with_events (as kda_prefill(..., stage_events=...)),
    kda_prefill_host_scratch_bytes, kda_prefill_host, kda_decode, kda_decode_multi,
    kda_workspace_status, kda_status_str

There is no fallback: if ``libkda.so`` is missing the import of this package
still succeeds, but the first call raises ``KdaLibraryMissing``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE, KDA_ERR_CUDA, KDA_ERR_TIMEOUT = range(6)
KDA_DTYPE_F32, KDA_DTYPE_BF16 = 0, 1
KDA_ALGO_AUTO, KDA_ALGO_SCAN, KDA_ALGO_CHUNKED, KDA_ALGO_CHUNKED_SEGMENTS = 0, 1, 2, 3
_ALGOS = {"auto": KDA_ALGO_AUTO, "scan": KDA_ALGO_SCAN, "chunked": KDA_ALGO_CHUNKED,
          "chunked_segments": KDA_ALGO_CHUNKED_SEGMENTS}

_vp = ctypes.c_void_p


class KdaLibraryMissing(RuntimeError):
    pass


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kda_status_str(status)} (status {status})")


class kda_params(ctypes.Structure):
    _fields_ = [
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("conv_kernel", ctypes.c_int32),
        ("io_dtype", ctypes.c_int32),
        ("algo", ctypes.c_int32),
        ("gate_lower_bound", ctypes.c_float),
        ("l2_eps", ctypes.c_float),
        ("norm_eps", ctypes.c_float),
        ("q_scale", ctypes.c_float),
        ("conv_w", _vp),
        ("A_log", _vp),
        ("dt_bias", _vp),
        ("norm_w", _vp),
        ("gate_kind", ctypes.c_int32),
        ("wait_limit_us", ctypes.c_uint32),
    ]


_lib = None


def lib():
    """The loaded ``libkda.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise KdaLibraryMissing(
                f"{LIB_PATH} is missing; build it with `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(kda_params)
        i32, i64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        L.kda_prefill_algo.argtypes = [P]
        L.kda_prefill_algo.restype = i32
        L.kda_prefill_workspace_bytes.argtypes = [P, i32, i64]
        L.kda_prefill_workspace_bytes.restype = sz
        L.kda_prefill_windows.argtypes = [P, i32, i64, sz]
        L.kda_prefill_windows.restype = i32
        L.kda_prefill_segments.argtypes = [P, i32, i64, sz]
        L.kda_prefill_segments.restype = i32
        L.kda_prefill.argtypes = [P] + [_vp] * 6 + [ctypes.POINTER(ctypes.c_int64), i32, i64] + [_vp] * 5 + [_vp, sz, _vp]
        L.kda_prefill.restype = ctypes.c_int
        L.kda_prefill_with_events.argtypes = L.kda_prefill.argtypes + [ctypes.POINTER(_vp)]
        L.kda_prefill_with_events.restype = ctypes.c_int
        L.kda_decode.argtypes = [P, i32] + [_vp] * 6 + [_vp] * 3 + [_vp]
        L.kda_decode.restype = ctypes.c_int
        L.kda_decode_multi.argtypes = [P, i32, i32] + [_vp] * 6 + [_vp, i32] + [_vp] * 5 + [_vp]
        L.kda_decode_multi.restype = ctypes.c_int
        L.kda_prefill_host_scratch_bytes.argtypes = [P, ctypes.POINTER(ctypes.c_int64), i32, i64, i64]
        L.kda_prefill_host_scratch_bytes.restype = sz
        L.kda_prefill_host.argtypes = ([P] + [_vp] * 6 + [ctypes.POINTER(ctypes.c_int64), i32, i64] + [_vp] * 5
                                       + [i64, _vp, sz, _vp, _vp, _vp])
        L.kda_prefill_host.restype = ctypes.c_int
        L.kda_workspace_status.argtypes = [_vp, _vp]
        L.kda_workspace_status.restype = ctypes.c_int
        L.kda_status_str.argtypes = [ctypes.c_int]
        L.kda_status_str.restype = ctypes.c_char_p
        _lib = L
    return _lib


def kda_status_str(status: int) -> str:
    return lib().kda_status_str(int(status)).decode()


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


@dataclass
class Params:
    """Holds the device parameter tensors and the C struct that points at them."""

    struct: kda_params
    tensors: tuple
    num_heads: int
    io_dtype: int

    @property
    def ref(self):
        return ctypes.byref(self.struct)


KDA_GATE_BOUNDED, KDA_GATE_SOFTPLUS = 0, 1
_GATES = {"bounded": KDA_GATE_BOUNDED, "softplus": KDA_GATE_SOFTPLUS}


def make_params(conv_w, A_log, dt_bias, norm_w, *, io_dtype: str = "bf16", algo: str = "auto",
                gate_lower_bound: float = -5.0, l2_eps: float = 1e-6, norm_eps: float = 1e-5,
                q_scale: float = 0.0, gate: str = "bounded", wait_limit_us: int = 0) -> Params:
    """conv_w [3][H*128][4], A_log [H], dt_bias [H*128], norm_w [128]: fp32 CUDA tensors.
    gate: "bounded" (g = lb sigmoid(e^A (z + dt_bias))) or "softplus"
    (g = -e^A softplus(z + dt_bias), unbounded below).  wait_limit_us: the
    test hook of kda_params (0 in normal use)."""
    H = int(A_log.shape[0])
    dt = {"f32": KDA_DTYPE_F32, "bf16": KDA_DTYPE_BF16}[io_dtype]
    tensors = tuple(t.contiguous() for t in (conv_w, A_log, dt_bias, norm_w))
    st = kda_params(H, 128, 4, dt, _ALGOS[algo], gate_lower_bound, l2_eps, norm_eps, q_scale,
                    *[t.data_ptr() for t in tensors], _GATES[gate], int(wait_limit_us))
    return Params(st, tensors, H, dt)


def kda_prefill_algo(params: Params) -> str:
    """'scan' or 'chunked': the prefill algorithm these parameters select."""
    a = int(lib().kda_prefill_algo(params.ref))
    if a < 0:
        raise KdaError(KDA_ERR_INVALID_ARG, "kda_prefill_algo")
    return {KDA_ALGO_SCAN: "scan", KDA_ALGO_CHUNKED: "chunked"}[a]


def kda_prefill_workspace_bytes(params: Params, n_seqs: int, total_tokens: int) -> int:
    return int(lib().kda_prefill_workspace_bytes(params.ref, int(n_seqs), int(total_tokens)))


def kda_prefill_windows(params: Params, n_seqs: int, total_tokens: int, workspace_bytes: int) -> int:
    """How many overlapped windows kda_prefill runs (1 = single pass)."""
    return int(lib().kda_prefill_windows(params.ref, int(n_seqs), int(total_tokens), int(workspace_bytes)))


def kda_prefill_segments(params: Params, n_seqs: int, total_tokens: int, workspace_bytes: int) -> int:
    """How many segments kda_prefill runs one sequence's recurrence as (0 = none)."""
    return int(lib().kda_prefill_segments(params.ref, int(n_seqs), int(total_tokens), int(workspace_bytes)))


def _cu_array(cu_seqlens: Sequence[int]):
    vals = [int(x) for x in cu_seqlens]
    return (ctypes.c_int64 * len(vals))(*vals), len(vals) - 1, vals[-1]


KDA_PREFILL_EVENTS = 6


def kda_prefill(params: Params, q, k, v, z, b, gout, cu_seqlens, S_in=None, S_out=None,
                ring_in=None, ring_out=None, o=None, workspace=None, stream=None, stage_events=None):
    """Varlen prefill.  Tensors are CUDA tensors in the layouts of ``include/kda.h``;
    ``cu_seqlens`` is a host sequence of n+1 ints.  Missing outputs and the
    workspace are allocated with torch.  ``stage_events`` (optional) is a list
    of KDA_PREFILL_EVENTS torch.cuda.Event objects recorded at the stage
    boundaries (kda_prefill_with_events).  Returns (o, S_out, ring_out)."""
    import torch
    cu, n, T = _cu_array(cu_seqlens)
    H = params.num_heads
    dev = q.device
    if o is None:
        o = torch.empty_like(q)
    if S_out is None:
        S_out = torch.empty(n, H, 128, 128, dtype=torch.float32, device=dev)
    if ring_out is None:
        ring_out = torch.empty(n, 3, 3, H * 128, dtype=q.dtype, device=dev)
    if workspace is None:
        nbytes = kda_prefill_workspace_bytes(params, n, T)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    args = (params.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(b), _ptr(gout),
            cu, n, T, _ptr(S_in), _ptr(S_out), _ptr(ring_in), _ptr(ring_out), _ptr(o),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if stage_events is None:
        st = lib().kda_prefill(*args)
    else:
        handles = []
        for e in stage_events:
            if e is not None and not e.cuda_event:
                e.record()  # torch creates the underlying cudaEvent_t lazily
            handles.append(None if e is None else e.cuda_event)
        evs = (_vp * KDA_PREFILL_EVENTS)(*handles)
        st = lib().kda_prefill_with_events(*args, evs)
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill")
    return o, S_out, ring_out


def kda_prefill_host_scratch_bytes(params: Params, cu_seqlens, segment_tokens: int) -> int:
    cu, n, T = _cu_array(cu_seqlens)
    return int(lib().kda_prefill_host_scratch_bytes(params.ref, cu, n, T, int(segment_tokens)))


def kda_prefill_host(params: Params, q, k, v, z, b, gout, cu_seqlens, S_in=None, S_out=None,
                     ring_in=None, ring_out=None, o=None, segment_tokens: int = 4096, scratch=None,
                     stream=None, h2d_stream=None, d2h_stream=None, device=None):
    """Prefill from HOST tensors (page-locked for the copies to overlap): the
    library copies token segments in on ``h2d_stream``, runs them on
    ``stream`` and copies the output back on ``d2h_stream``.  S_in / ring_in /
    S_out / ring_out and ``scratch`` are CUDA tensors; missing ones are
    allocated (``o`` as pinned host memory).  Synchronise ``stream`` before
    reading ``o``.  Returns (o, S_out, ring_out)."""
    import torch
    cu, n, T = _cu_array(cu_seqlens)
    H = params.num_heads
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if o is None:
        o = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    if S_out is None:
        S_out = torch.empty(n, H, 128, 128, dtype=torch.float32, device=dev)
    if ring_out is None:
        ring_out = torch.empty(n, 3, 3, H * 128, dtype=q.dtype, device=dev)
    if scratch is None:
        nbytes = int(lib().kda_prefill_host_scratch_bytes(params.ref, cu, n, T, int(segment_tokens)))
        scratch = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    st = lib().kda_prefill_host(params.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(b), _ptr(gout),
                                cu, n, T, _ptr(S_in), _ptr(S_out), _ptr(ring_in), _ptr(ring_out), _ptr(o),
                                int(segment_tokens), _ptr(scratch), scratch.numel() * scratch.element_size(),
                                _stream(stream), None if h2d_stream is None else _stream(h2d_stream),
                                None if d2h_stream is None else _stream(d2h_stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill_host")
    return o, S_out, ring_out


def kda_decode(params: Params, q, k, v, z, b, gout, S, ring, o=None, stream=None):
    """One token per session; S and ring are updated in place.  Returns o."""
    import torch
    n = int(q.shape[0])
    if o is None:
        o = torch.empty_like(q)
    st = lib().kda_decode(params.ref, n, _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(b), _ptr(gout),
                          _ptr(S), _ptr(ring), _ptr(o), _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode")
    return o


KDA_DECODE_MAX_TOKENS = 64


def kda_decode_multi(params: Params, q, k, v, z, b, gout, S_in, ring_in, S_out=None, ring_out=None,
                     slots=None, o=None, stream=None):
    """n_tokens consecutive tokens per session (a speculative verify round).
    q, k, v, z, gout: [n][n_tokens][H*128]; b: [n][n_tokens][H].  S_in /
    ring_in are state / ring pools [n_slots][...]; S_out / ring_out default to
    them (in-place).  ``slots`` (int32 CUDA tensor [n]) maps sessions to pool
    slots.  Keeping S_in / ring_in (separate outputs) allows a rollback: call
    again with the accepted prefix of the tokens.  Returns o."""
    import torch
    n, n_tok = int(q.shape[0]), int(q.shape[1])
    S_out = S_in if S_out is None else S_out
    ring_out = ring_in if ring_out is None else ring_out
    if o is None:
        o = torch.empty_like(q)
    n_slots = int(S_in.shape[0])
    st = lib().kda_decode_multi(params.ref, n, n_tok, _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(b), _ptr(gout),
                                _ptr(slots), n_slots, _ptr(S_in), _ptr(S_out), _ptr(ring_in), _ptr(ring_out),
                                _ptr(o), _stream(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_multi")
    return o


def kda_workspace_status(workspace, stream=None) -> int:
    return int(lib().kda_workspace_status(_ptr(workspace), _stream(stream)))
