"""The C ABI on the host: the library loads without a GPU, exports every
function include/kda.h declares, and rejects bad arguments before it
enqueues anything (every case here fails validation, so no kernel runs)."""
import ctypes
import os
import re

import pytest

import gated_delta_rule_04_gb300 as kda
from gated_delta_rule_04_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")

FAKE = 0x10000  # aligned non-null address; never dereferenced on these paths


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return kda.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"kda_prefill", "kda_decode", "kda_prefill_workspace_bytes", "kda_status_str",
            "kda_workspace_status"} <= set(names)
    for name in names:
        assert hasattr(L, name), f"libkda.so does not export {name}"


def test_status_strings(L):
    for s in range(6):
        assert kda.kda_status_str(s)
    assert kda.kda_status_str(99) == "unknown status"


def params(**kw):
    d = dict(num_heads=2, head_dim=128, conv_kernel=4, io_dtype=kda.KDA_DTYPE_BF16,
             algo=kda.KDA_ALGO_AUTO, gate_lower_bound=-5.0, l2_eps=1e-6, norm_eps=1e-5, q_scale=0.0,
             conv_w=FAKE, A_log=FAKE, dt_bias=FAKE, norm_w=FAKE)
    d.update(kw)
    return kda.kda_params(**d)


def prefill(L, p, cu, T=None, ws_bytes=1 << 40, ws=FAKE, **ptrs):
    arr = (ctypes.c_int64 * len(cu))(*cu)
    n = len(cu) - 1
    T = cu[-1] if T is None else T
    a = dict(q=FAKE, k=FAKE, v=FAKE, z=FAKE, b=FAKE, gout=FAKE, S_in=None, S_out=FAKE,
             ring_in=None, ring_out=FAKE, o=FAKE)
    a.update(ptrs)
    return L.kda_prefill(ctypes.byref(p), a["q"], a["k"], a["v"], a["z"], a["b"], a["gout"], arr, n, T,
                         a["S_in"], a["S_out"], a["ring_in"], a["ring_out"], a["o"], ws, ws_bytes, None)


def test_algo_query(L):
    assert L.kda_prefill_algo(ctypes.byref(params(algo=kda.KDA_ALGO_SCAN))) == kda.KDA_ALGO_SCAN
    assert L.kda_prefill_algo(ctypes.byref(params(io_dtype=kda.KDA_DTYPE_F32))) == kda.KDA_ALGO_SCAN
    assert L.kda_prefill_algo(ctypes.byref(params(head_dim=64))) == -1
    assert L.kda_prefill_algo(None) == -1


def test_workspace_query(L):
    p = params()
    small = L.kda_prefill_workspace_bytes(ctypes.byref(p), 1, 64)
    big = L.kda_prefill_workspace_bytes(ctypes.byref(p), 1, 64 * 1000)
    assert 0 < small < big
    assert L.kda_prefill_workspace_bytes(ctypes.byref(p), 0, 0) == 0
    assert L.kda_prefill_workspace_bytes(None, 1, 64) == 0
    assert L.kda_prefill_workspace_bytes(ctypes.byref(params(head_dim=64)), 1, 64) == 0
    assert L.kda_prefill_workspace_bytes(ctypes.byref(p), -1, 64) == 0


@pytest.mark.parametrize("kw, want", [
    (dict(head_dim=64), kda.KDA_ERR_UNSUPPORTED),
    (dict(conv_kernel=3), kda.KDA_ERR_UNSUPPORTED),
    (dict(num_heads=0), kda.KDA_ERR_INVALID_ARG),
    (dict(io_dtype=7), kda.KDA_ERR_INVALID_ARG),
    (dict(algo=9), kda.KDA_ERR_INVALID_ARG),
    (dict(gate_lower_bound=0.5), kda.KDA_ERR_INVALID_ARG),
    (dict(gate_lower_bound=float("nan")), kda.KDA_ERR_INVALID_ARG),
    (dict(l2_eps=-1.0), kda.KDA_ERR_INVALID_ARG),
    (dict(conv_w=None), kda.KDA_ERR_INVALID_ARG),
    (dict(dt_bias=FAKE + 4), kda.KDA_ERR_INVALID_ARG),
    (dict(algo=kda.KDA_ALGO_CHUNKED, io_dtype=kda.KDA_DTYPE_F32), kda.KDA_ERR_UNSUPPORTED),
    (dict(algo=kda.KDA_ALGO_CHUNKED, gate_lower_bound=-8.0), kda.KDA_ERR_UNSUPPORTED),
])
def test_bad_params(L, kw, want):
    assert prefill(L, params(**kw), [0, 64]) == want


@pytest.mark.parametrize("cu, T", [
    ([1, 64], 64),        # cu[0] != 0
    ([0, 64, 32], 32),    # decreasing
    ([0, 64], 65),        # cu[n] != total
    ([0, 10], -1),
])
def test_bad_cu_seqlens(L, cu, T):
    assert prefill(L, params(), cu, T=T) == kda.KDA_ERR_INVALID_ARG


def test_null_cu_seqlens(L):
    p = params()
    assert L.kda_prefill(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 64, None,
                         FAKE, None, FAKE, FAKE, FAKE, 1 << 40, None) == kda.KDA_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["q", "k", "v", "z", "gout", "o", "b", "S_out"])
def test_null_token_pointers(L, name):
    assert prefill(L, params(), [0, 64], **{name: None}) == kda.KDA_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["q", "o", "S_out", "S_in", "ring_in", "ring_out"])
def test_misaligned_pointers(L, name):
    assert prefill(L, params(), [0, 64], **{name: FAKE + 8}) == kda.KDA_ERR_INVALID_ARG


def test_workspace_errors(L):
    p = params()
    need = L.kda_prefill_workspace_bytes(ctypes.byref(p), 1, 64)
    assert prefill(L, p, [0, 64], ws_bytes=need - 1) == kda.KDA_ERR_WORKSPACE
    assert prefill(L, p, [0, 64], ws=None) == kda.KDA_ERR_WORKSPACE
    assert prefill(L, p, [0, 64], ws=FAKE + 16) == kda.KDA_ERR_WORKSPACE


def test_empty_batch_is_a_no_op(L):
    assert prefill(L, params(), [0], T=0) == kda.KDA_OK


def test_decode_validation(L):
    p = params()
    f = FAKE
    assert L.kda_decode(ctypes.byref(p), 0, f, f, f, f, f, f, f, f, f, None) == kda.KDA_OK
    assert L.kda_decode(ctypes.byref(p), -1, f, f, f, f, f, f, f, f, f, None) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_decode(ctypes.byref(p), 4, f, f, f, f, f, f, None, f, f, None) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_decode(ctypes.byref(p), 4, f, f, f, f, None, f, f, f, f, None) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_decode(ctypes.byref(p), 4, f + 2, f, f, f, f, f, f, f, f, None) == kda.KDA_ERR_INVALID_ARG
    bad = params(head_dim=96)
    assert L.kda_decode(ctypes.byref(bad), 4, f, f, f, f, f, f, f, f, f, None) == kda.KDA_ERR_UNSUPPORTED


def test_workspace_status_rejects_bad_pointer(L):
    assert L.kda_workspace_status(None, None) == kda.KDA_ERR_WORKSPACE
    assert L.kda_workspace_status(FAKE + 16, None) == kda.KDA_ERR_WORKSPACE


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(kda, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(kda, "_lib", None)
    with pytest.raises(kda.KdaLibraryMissing):
        kda.lib()


def test_decode_multi_validation(L):
    p = params()
    f = FAKE

    def call(n=4, n_tok=3, slots=None, n_slots=4, S_in=f, S_out=f, ring_in=f, ring_out=f, q=f, b=f):
        return L.kda_decode_multi(ctypes.byref(p), n, n_tok, q, f, f, f, b, f, slots, n_slots, S_in, S_out,
                                  ring_in, ring_out, f, None)

    assert call(n=0) == kda.KDA_OK
    assert call(n_tok=0) == kda.KDA_ERR_INVALID_ARG
    assert call(n_tok=kda.KDA_DECODE_MAX_TOKENS + 1) == kda.KDA_ERR_INVALID_ARG
    assert call(n=-1) == kda.KDA_ERR_INVALID_ARG
    assert call(n_slots=3) == kda.KDA_ERR_INVALID_ARG          # identity slots need n_slots >= n
    assert call(S_in=None) == kda.KDA_ERR_INVALID_ARG
    assert call(ring_out=None) == kda.KDA_ERR_INVALID_ARG
    assert call(S_out=f + 8) == kda.KDA_ERR_INVALID_ARG
    assert call(b=None) == kda.KDA_ERR_INVALID_ARG
    bad = params(head_dim=64)
    assert L.kda_decode_multi(ctypes.byref(bad), 4, 3, f, f, f, f, f, f, None, 4, f, f, f, f, f,
                              None) == kda.KDA_ERR_UNSUPPORTED


def test_gate_kind_validation(L):
    # the softplus gate runs the chunked form with bf16 I/O (diagonal blocks by
    # position pairs) and the scan with fp32 I/O
    assert L.kda_prefill_algo(ctypes.byref(params(gate_kind=1))) == kda.KDA_ALGO_CHUNKED
    assert L.kda_prefill_algo(ctypes.byref(params(gate_kind=1, io_dtype=kda.KDA_DTYPE_F32))) == kda.KDA_ALGO_SCAN
    assert prefill(L, params(gate_kind=1, algo=kda.KDA_ALGO_CHUNKED, io_dtype=kda.KDA_DTYPE_F32),
                   [0, 64]) == kda.KDA_ERR_UNSUPPORTED
    assert prefill(L, params(gate_kind=2), [0, 64]) == kda.KDA_ERR_INVALID_ARG
    # the lower bound is not used by the softplus gate
    assert L.kda_prefill_algo(ctypes.byref(params(gate_kind=1, gate_lower_bound=0.5))) == kda.KDA_ALGO_CHUNKED
    assert L.kda_prefill_algo(ctypes.byref(params(gate_kind=1, gate_lower_bound=-80.0))) == kda.KDA_ALGO_CHUNKED


# ---------------------------------------------------------------- kda_prefill_host
STAGE_ALIGN = 256


def _up(x):
    return (x + STAGE_ALIGN - 1) // STAGE_ALIGN * STAGE_ALIGN


def segment_piece_counts(cu, seg):
    """Sequences that hold tokens of each segment [t0, t0 + seg), with the
    empty sequences that start inside it: the piece count of every segment."""
    T = cu[-1]
    out = []
    for t0 in range(0, T, seg):
        t1 = min(T, t0 + seg)
        first = next(i for i in range(len(cu) - 1) if cu[i + 1] > t0)
        last = max(i for i in range(len(cu) - 1) if i == first or cu[i] < t1)
        out.append((last - first + 1, t1 - t0))
    return out


def host_scratch(L, p, cu, seg):
    arr = (ctypes.c_int64 * len(cu))(*cu)
    return L.kda_prefill_host_scratch_bytes(ctypes.byref(p), arr, len(cu) - 1, cu[-1], seg)


@pytest.mark.parametrize("cu, seg", [
    ([0, 64], 64), ([0, 300], 100), ([0, 10, 10, 200, 700], 128), ([0, 5, 9, 13, 1000], 4),
    ([0, 0, 0, 130, 130], 64),
])
def test_host_scratch_bytes(L, cu, seg):
    """Scratch = the largest per-segment workspace + three staging sets."""
    p = params()
    H, es = 2, 2
    ws = max(L.kda_prefill_workspace_bytes(ctypes.byref(p), n, t) for n, t in segment_piece_counts(cu, seg))
    s = min(seg, cu[-1])
    stage = 6 * _up(s * H * 128 * es) + _up(s * H * es)
    assert host_scratch(L, p, cu, seg) == _up(ws) + 3 * stage


def test_host_scratch_bytes_rejects(L):
    p = params()
    assert host_scratch(L, p, [0, 64], 0) == 0
    assert host_scratch(L, p, [0], 64) == 0
    assert host_scratch(L, params(head_dim=64), [0, 64], 64) == 0
    assert host_scratch(L, p, [0, 64, 32], 64) == 0


def prefill_host(L, p, cu, T=None, seg=64, scratch=FAKE, scratch_bytes=1 << 40, **ptrs):
    arr = (ctypes.c_int64 * len(cu))(*cu)
    n = len(cu) - 1
    T = cu[-1] if T is None else T
    a = dict(q=FAKE, k=FAKE, v=FAKE, z=FAKE, b=FAKE, gout=FAKE, S_in=None, S_out=FAKE,
             ring_in=None, ring_out=FAKE, o=FAKE)
    a.update(ptrs)
    return L.kda_prefill_host(ctypes.byref(p), a["q"], a["k"], a["v"], a["z"], a["b"], a["gout"], arr, n, T,
                              a["S_in"], a["S_out"], a["ring_in"], a["ring_out"], a["o"], seg, scratch,
                              scratch_bytes, None, None, None)


@pytest.mark.parametrize("kw, want", [
    (dict(head_dim=64), kda.KDA_ERR_UNSUPPORTED),
    (dict(num_heads=0), kda.KDA_ERR_INVALID_ARG),
    (dict(algo=kda.KDA_ALGO_CHUNKED, io_dtype=kda.KDA_DTYPE_F32), kda.KDA_ERR_UNSUPPORTED),
])
def test_host_bad_params(L, kw, want):
    assert prefill_host(L, params(**kw), [0, 64]) == want


def test_host_validation(L):
    p = params()
    assert prefill_host(L, p, [1, 64]) == kda.KDA_ERR_INVALID_ARG
    assert prefill_host(L, p, [0, 64], T=65) == kda.KDA_ERR_INVALID_ARG
    assert prefill_host(L, p, [0, 64], seg=0) == kda.KDA_ERR_INVALID_ARG
    assert prefill_host(L, p, [0, 64], seg=1 << 40) == kda.KDA_ERR_UNSUPPORTED
    for name in ("S_out", "ring_out", "q", "b", "gout", "o"):
        assert prefill_host(L, p, [0, 64], **{name: None}) == kda.KDA_ERR_INVALID_ARG, name
    for name in ("S_out", "ring_out", "S_in", "ring_in"):
        assert prefill_host(L, p, [0, 64], **{name: FAKE + 8}) == kda.KDA_ERR_INVALID_ARG, name
    need = host_scratch(L, p, [0, 64], 64)
    assert prefill_host(L, p, [0, 64], scratch_bytes=need - 1) == kda.KDA_ERR_WORKSPACE
    assert prefill_host(L, p, [0, 64], scratch=None) == kda.KDA_ERR_WORKSPACE
    assert prefill_host(L, p, [0, 64], scratch=FAKE + 16) == kda.KDA_ERR_WORKSPACE
    assert prefill_host(L, p, [0], T=0) == kda.KDA_OK


def test_prefill_windows_query(L):
    p = params()
    assert L.kda_prefill_windows(ctypes.byref(params(head_dim=64)), 1, 32768, 1 << 40) == -1
    assert L.kda_prefill_windows(ctypes.byref(p), -1, 32768, 1 << 40) == -1
    # several sequences, short ones, or the scan path: always the single pass
    assert L.kda_prefill_windows(ctypes.byref(p), 2, 32768, 1 << 40) == 1
    assert L.kda_prefill_windows(ctypes.byref(p), 1, 2047, 1 << 40) == 1
    assert L.kda_prefill_windows(ctypes.byref(params(algo=kda.KDA_ALGO_SCAN)), 1, 32768, 1 << 40) == 1
    assert L.kda_prefill_windows(ctypes.byref(p), 1, 32768, 1 << 40) >= 1   # needs a device for more


def test_prefill_segments_query(L):
    p = params()
    assert L.kda_prefill_segments(ctypes.byref(params(head_dim=64)), 1, 32768, 1 << 40) == -1
    assert L.kda_prefill_segments(ctypes.byref(p), -1, 32768, 1 << 40) == -1
    # several sequences, the scan path, or the plain chunked schedule: no segments
    assert L.kda_prefill_segments(ctypes.byref(p), 2, 32768, 1 << 40) == 0
    assert L.kda_prefill_segments(ctypes.byref(params(algo=kda.KDA_ALGO_SCAN)), 1, 32768, 1 << 40) == 0
    assert L.kda_prefill_segments(ctypes.byref(params(algo=kda.KDA_ALGO_CHUNKED)), 1, 32768, 1 << 40) == 0
    assert L.kda_prefill_segments(ctypes.byref(p), 1, 32768, 1 << 40) in (0, 9)   # 2 heads: 9 with a device


@pytest.mark.parametrize("H", [8, 48, 64, 96])
@pytest.mark.parametrize("T", [2048, 4096 + 37, 16384, 20384, 32768, 32768 + 64 * 7 + 5])
def test_workspace_covers_overlapped_windows(L, T, H):
    """A single sequence may run as up to 4 windows (3 above 48 heads; at least
    1024 tokens per window up to 64 heads, 8192 with more), the last one 1/d as
    long as the others (d = 6 above 64 heads, 4 above 32, 2 up to 32); the
    workspace query covers two windows' records (window sizes round up to whole
    64-token chunks)."""
    import bench
    rec = bench.REC_BYTES   # equal to the layout header's (tests/test_record_layout.py)
    p = params(num_heads=H)
    need = L.kda_prefill_workspace_bytes(ctypes.byref(p), 1, T)
    windows = min(3 if H > 48 else 4, T // (1024 if H <= 64 else 8192))
    if windows >= 2:
        d = 6 if H > 64 else 4 if H > 32 else 2
        seg = -(-(d * T) // (d * windows - d + 1))
        seg_chunks = -(-seg // 64)
        assert (windows - 1) * seg_chunks * 64 < T <= windows * seg_chunks * 64   # no empty last window
        assert need >= 2 * seg_chunks * H * rec
    # and never less than the single pass needs for several sequences' worth of chunks
    assert need >= (T // 64 + 1) * H * rec


def noalloc(L, p, cu, T=None, **ptrs):
    f = L.kda_prefill_noalloc
    arr = (ctypes.c_int64 * len(cu))(*cu)
    n = len(cu) - 1
    T = cu[-1] if T is None else T
    a = dict(q=FAKE, k=FAKE, v=FAKE, z=FAKE, b=FAKE, gout=FAKE, S_in=None, S_out=FAKE,
             ring_in=None, ring_out=FAKE, o=FAKE)
    a.update(ptrs)
    f.restype = ctypes.c_int
    return f(ctypes.byref(p), *[ctypes.c_void_p(a[x]) if a[x] else None for x in ("q", "k", "v", "z", "b", "gout")],
             arr, ctypes.c_int32(n), ctypes.c_int64(T),
             *[ctypes.c_void_p(a[x]) if a[x] else None for x in ("S_in", "S_out", "ring_in", "ring_out", "o")],
             None)


@pytest.mark.parametrize("kw, cu", [
    (dict(head_dim=64), [0, 64]),
    (dict(conv_w=0, algo=kda.KDA_ALGO_CHUNKED), [0, 64]),
    (dict(num_heads=0, head_dim=96), [0, 64]),
    (dict(gate_kind=1, algo=kda.KDA_ALGO_CHUNKED, io_dtype=kda.KDA_DTYPE_F32), [0, 64]),
    (dict(l2_eps=-1.0), [0, 64]),
    (dict(), [0, 70, 60]),
    (dict(), [1, 64]),
])
def test_noalloc_rejects_exactly_as_kda_prefill(L, kw, cu):
    """The no-allocation entry point runs kda_prefill's checks and returns the
    same status for every rejected argument set (no kernel runs)."""
    p = params(**kw)
    want = prefill(L, p, cu)
    assert want != kda.KDA_OK
    assert noalloc(L, p, cu) == want


def test_noalloc_rejects_more_than_512_sequences(L):
    """The sequence order is sorted on the host stack, so one call takes at
    most 512 sequences; the check runs before anything is enqueued."""
    cu = list(range(0, 514))   # 513 one-token sequences
    assert noalloc(L, params(), cu) == kda.KDA_ERR_UNSUPPORTED
