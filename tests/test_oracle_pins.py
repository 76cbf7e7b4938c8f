"""Pins of the fp64 oracle against facts fixed by the sources and by
mathematics, independent of the oracle's own code.

Sources: "Kimi Delta Attention (KDA) -- analysis & C kernel plan" (sections
"The KDA layer, precisely", "Recurrence"); "ferrox-models 0.8.0, module kda"
(module overview); "Kimi K3 - Retention gate - OpenModelAtlas" (gate formula,
gate.py excerpt); "memra-engine 0.124.0, module kda" (PREFILL DISPATCH, the
chunked form).
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    return x * sig(x)


def rand_core(rng, T, H, D, unit_keys=True, g_lo=-5.0):
    q = rng.standard_normal((T, H, D))
    k = rng.standard_normal((T, H, D))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, D))
    g = rng.uniform(g_lo, 0.0, (T, H, D))
    beta = rng.uniform(0.05, 0.95, (T, H))
    return q, k, v, g, beta


def rand_params(rng, H, D, **kw):
    return oracle.Params(
        num_heads=H, head_dim=D,
        conv_w=rng.standard_normal((3, H * D, 4)) * 0.5,
        A_log=np.log(rng.uniform(1, 16, H)),
        dt_bias=rng.standard_normal(H * D) * math.sqrt(0.5),
        norm_w=1 + rng.standard_normal(D) * math.sqrt(0.1), **kw)


def rand_tokens(rng, T, H, D):
    W = H * D
    return dict(q=rng.standard_normal((T, W)), k=rng.standard_normal((T, W)),
                v=rng.standard_normal((T, W)), z=rng.standard_normal((T, W)),
                b=rng.standard_normal((T, H)), gout=rng.standard_normal((T, W)))


# --------------------------------------------------------------------- core
def test_p1_one_token_zero_state():
    """From a zero state one token gives S = beta k v^T and o = beta (q.k) v."""
    rng = np.random.default_rng(1)
    q, k, v, g, beta = rand_core(rng, 1, 3, 8, unit_keys=False)
    o, S = oracle.core(q, k, v, g, beta)
    for h in range(3):
        np.testing.assert_allclose(S[h], beta[0, h] * np.outer(k[0, h], v[0, h]), rtol=0, atol=1e-14)
        np.testing.assert_allclose(o[0, h], beta[0, h] * (q[0, h] @ k[0, h]) * v[0, h], rtol=0, atol=1e-14)


def test_p2_beta_zero_only_decays():
    """With beta = 0 the state only decays by exp(g) along the key axis."""
    rng = np.random.default_rng(2)
    T, H, D = 9, 2, 6
    q, k, v, g, _ = rand_core(rng, T, H, D)
    beta = np.zeros((T, H))
    S0 = rng.standard_normal((H, D, D))
    o, S = oracle.core(q, k, v, g, beta, S0)
    csum = np.cumsum(g, axis=0)
    for h in range(H):
        np.testing.assert_allclose(S[h], np.exp(csum[-1, h])[:, None] * S0[h], rtol=1e-13, atol=1e-15)
        for t in range(T):
            St = np.exp(csum[t, h])[:, None] * S0[h]
            np.testing.assert_allclose(o[t, h], St.T @ q[t, h], rtol=1e-12, atol=1e-14)


def test_p3_orthonormal_keys_store_and_overwrite():
    """g = 0, beta = 1, orthonormal keys: the state returns every stored value
    exactly, from any initial state; writing a key again overwrites its value."""
    rng = np.random.default_rng(3)
    D, T = 8, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((D, D)))
    keys = Qm.T[:T]
    vals = rng.standard_normal((T, D))
    S0 = rng.standard_normal((1, D, D))
    zeros = np.zeros((T, 1, D))
    o, S = oracle.core(zeros, keys[:, None, :], vals[:, None, :], zeros, np.ones((T, 1)), S0)
    for j in range(T):
        np.testing.assert_allclose(S[0].T @ keys[j], vals[j], atol=1e-13)
    # overwrite key 2
    newv = rng.standard_normal(D)
    one = np.zeros((1, 1, D))
    _, S2 = oracle.core(one, keys[2][None, None], newv[None, None], one, np.ones((1, 1)), S)
    np.testing.assert_allclose(S2[0].T @ keys[2], newv, atol=1e-13)
    for j in (0, 1, 3, 4, 5):
        np.testing.assert_allclose(S2[0].T @ keys[j], vals[j], atol=1e-13)


def load_p4():
    rows = []
    with open(os.path.join(GOLDEN, "p4_three_token_recurrence.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            a, b, c = line.split("|")
            rows.append(([float(x) for x in a.split()], [float(x) for x in b.split()],
                          [float(x) for x in c.split()]))
    return rows


def test_p4_hand_derived_three_tokens():
    rows = load_p4()
    T = len(rows)
    k = np.array([[r[0][1:3]] for r in rows])
    v = np.array([[r[0][3:5]] for r in rows])
    q = np.array([[r[0][5:7]] for r in rows])
    beta = np.array([[r[0][7]] for r in rows])
    g = np.log(np.array([[r[0][8:10]] for r in rows]))
    for t in range(1, T + 1):
        o, S = oracle.core(q[:t], k[:t], v[:t], g[:t], beta[:t])
        np.testing.assert_allclose(o[t - 1, 0], rows[t - 1][1], rtol=0, atol=1e-15)
        np.testing.assert_allclose(S[0].reshape(-1), rows[t - 1][2], rtol=0, atol=1e-15)


def test_p11_transition_matrix_form():
    """Brute force on tiny inputs through the equivalent matrix form
    S_t = (I - beta k k^T) Diag(e^g) S_{t-1} + beta k v^T, o_t = S_t^T q_t."""
    rng = np.random.default_rng(11)
    for T in (1, 2, 3, 4):
        D = 3
        q, k, v, g, beta = rand_core(rng, T, 1, D, unit_keys=False)
        S0 = rng.standard_normal((1, D, D))
        o, S = oracle.core(q, k, v, g, beta, S0)
        St = S0[0].copy()
        for t in range(T):
            kt = k[t, 0][:, None]
            M = (np.eye(D) - beta[t, 0] * kt @ kt.T) @ np.diag(np.exp(g[t, 0]))
            St = M @ St + beta[t, 0] * kt @ v[t, 0][None, :]
            np.testing.assert_allclose(o[t, 0], St.T @ q[t, 0], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(S[0], St, rtol=1e-13, atol=1e-14)


def test_p7_retrieval_invariant():
    """After any step: S_t^T k_t = (1 - beta |k|^2) S'^T k_t + beta |k|^2 v_t."""
    rng = np.random.default_rng(7)
    T, H, D = 12, 2, 8
    q, k, v, g, beta = rand_core(rng, T, H, D, unit_keys=False)
    S0 = rng.standard_normal((H, D, D))
    for t in (0, 5, 11):
        _, Sprev = oracle.core(q[:t], k[:t], v[:t], g[:t], beta[:t], S0) if t else (None, S0)
        _, St = oracle.core(q[:t + 1], k[:t + 1], v[:t + 1], g[:t + 1], beta[:t + 1], S0)
        for h in range(H):
            Sp = np.exp(g[t, h])[:, None] * Sprev[h]
            kk = k[t, h] @ k[t, h]
            lhs = St[h].T @ k[t, h]
            rhs = (1 - beta[t, h] * kk) * (Sp.T @ k[t, h]) + beta[t, h] * kk * v[t, h]
            np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("C", [1, 2, 4, 16, 64])
def test_p6_chunked_equals_sequential(C):
    """The chunked form (per-channel cumulative log gate, sub-tile reference
    points, UT solve, state GEMMs) equals the sequential recurrence."""
    rng = np.random.default_rng(60 + C)
    T, H, D = 100, 2, 16
    q, k, v, g, beta = rand_core(rng, T, H, D)
    S0 = rng.standard_normal((H, D, D)) * 0.3
    o_ref, S_ref = oracle.core(q, k, v, g, beta, S0)
    o_c, S_c = oracle.chunked_core(q, k, v, g, beta, S0, chunk=C, subtile=16)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel(o_c, o_ref) < 1e-12
    assert rel(S_c, S_ref) < 1e-12


def test_p6_chunked_strong_decay_in_range():
    """Every gate at the -5 bound over 64-token chunks: a whole-chunk
    reference point would need factors up to e^{320} (beyond fp32 and bf16);
    with 16-token sub-tile references no factor exceeds e^{80} and the
    chunked form still equals the sequential one."""
    rng = np.random.default_rng(66)
    T, H, D = 130, 1, 8
    q, k, v, _, beta = rand_core(rng, T, H, D)
    g = np.full((T, H, D), -4.999)
    o_ref, S_ref = oracle.core(q, k, v, g, beta)
    o_c, S_c = oracle.chunked_core(q, k, v, g, beta, chunk=64, subtile=16)
    assert np.all(np.isfinite(o_c))
    np.testing.assert_allclose(o_c, o_ref, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(S_c, S_ref, rtol=1e-9, atol=1e-12)


# -------------------------------------------------------------------- mixer
def test_p1_mixer_one_token_closed_form():
    """One token from zero state and zero ring: only tap 3 sees data, so
    conv = w[3] x; then o_core = beta (q.k) v with the normalised q, k."""
    rng = np.random.default_rng(101)
    H, D = 3, 8
    p = rand_params(rng, H, D)
    tk = rand_tokens(rng, 1, H, D)
    out = oracle.mixer(p, [0, 1], **tk, intermediates=True)
    for h in range(H):
        sl = slice(h * D, (h + 1) * D)
        a = [silu(p.conv_w[pl, sl, 3] * tk[name][0, sl]) for pl, name in enumerate("qkv")]
        qn = a[0] / np.sqrt(a[0] @ a[0] + 1e-6) / math.sqrt(D)
        kn = a[1] / np.sqrt(a[1] @ a[1] + 1e-6)
        beta = sig(tk["b"][0, h])
        oc = beta * (qn @ kn) * a[2]
        np.testing.assert_allclose(out["o_core"][0, sl], oc, rtol=1e-13, atol=1e-15)
        rms = np.sqrt(np.mean(oc ** 2) + 1e-5)
        np.testing.assert_allclose(out["o"][0, sl], oc / rms * p.norm_w * sig(tk["gout"][0, sl]),
                                   rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(out["S"][0, h], beta * np.outer(kn, a[2]), rtol=1e-13, atol=1e-15)


def _taps(p, taps):
    p.conv_w = np.broadcast_to(np.array(taps, dtype=np.float64), p.conv_w.shape).copy()
    return p


def test_p5_conv_identity_tap():
    """Taps (0,0,0,1) make the conv the identity: v_hat_t = SiLU(v_t)."""
    rng = np.random.default_rng(51)
    H, D, T = 2, 4, 5
    p = _taps(rand_params(rng, H, D), (0, 0, 0, 1))
    tk = rand_tokens(rng, T, H, D)
    out = oracle.mixer(p, [0, T], **tk, intermediates=True)
    np.testing.assert_allclose(out["vh"], silu(tk["v"]), rtol=0, atol=1e-15)
    # P9: |k_hat|^2 = s / (s + eps) with s = sum SiLU(k)^2 per head
    a = silu(tk["k"]).reshape(T, H, D)
    s = (a ** 2).sum(-1)
    kn2 = (out["kh"].reshape(T, H, D) ** 2).sum(-1)
    np.testing.assert_allclose(kn2, s / (s + 1e-6), rtol=1e-14)
    aq = silu(tk["q"]).reshape(T, H, D)
    sq = (aq ** 2).sum(-1)
    qn2 = (out["qh"].reshape(T, H, D) ** 2).sum(-1)
    np.testing.assert_allclose(qn2, sq / (sq + 1e-6) / D, rtol=1e-14)


def test_p5_conv_oldest_tap_and_ring():
    """Taps (1,0,0,0) give x_{t-3}: zero for t < 3 from a zero ring, the ring
    slots (oldest first) from a nonzero ring."""
    rng = np.random.default_rng(52)
    H, D, T = 2, 4, 5
    W = H * D
    p = _taps(rand_params(rng, H, D), (1, 0, 0, 0))
    tk = rand_tokens(rng, T, H, D)
    out = oracle.mixer(p, [0, T], **tk, intermediates=True)
    np.testing.assert_allclose(out["vh"][:3], 0.0, atol=0)
    np.testing.assert_allclose(out["vh"][3:], silu(tk["v"][:2]), atol=1e-15)
    ring = rng.standard_normal((1, 3, 3, W))
    out = oracle.mixer(p, [0, T], **tk, ring_in=ring, intermediates=True)
    for t in range(3):
        np.testing.assert_allclose(out["vh"][t], silu(ring[0, 2, t]), atol=1e-15)
    # the final ring holds the last three raw inputs per plane
    for pl, name in enumerate("qkv"):
        np.testing.assert_array_equal(out["ring"][0, pl], tk[name][T - 3:])


def test_p5_short_sequence_ring_carry():
    """A sequence shorter than the ring shifts the old ring: slot s of the
    result is the raw input at local index L-3+s, from ring_in when negative."""
    rng = np.random.default_rng(53)
    H, D = 1, 4
    p = rand_params(rng, H, D)
    for L in (0, 1, 2):
        tk = rand_tokens(rng, L, H, D)
        ring = rng.standard_normal((1, 3, 3, H * D))
        out = oracle.mixer(p, [0, L], **tk, ring_in=ring)
        for pl, name in enumerate("qkv"):
            for s in range(3):
                src = L - 3 + s
                want = tk[name][src] if src >= 0 else ring[0, pl, 3 + src]
                np.testing.assert_array_equal(out["ring"][0, pl, s], want)


def test_p5_prefill_equals_decode_steps_and_split():
    """prefill(5) == five one-token steps == prefill(2) then prefill(3), with
    state and ring handed over (the five-position check of the ferrox page)."""
    rng = np.random.default_rng(54)
    H, D, T = 2, 8, 5
    p = rand_params(rng, H, D)
    tk = rand_tokens(rng, T, H, D)
    full = oracle.mixer(p, [0, T], **tk)
    S, ring, outs = None, None, []
    for t in range(T):
        one = {k_: v_[t:t + 1] for k_, v_ in tk.items()}
        r = oracle.mixer(p, [0, 1], **one, S_in=S, ring_in=ring)
        S, ring = r["S"], r["ring"]
        outs.append(r["o"][0])
    np.testing.assert_allclose(np.stack(outs), full["o"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S, full["S"], rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(ring, full["ring"])
    a = oracle.mixer(p, [0, 2], **{k_: v_[:2] for k_, v_ in tk.items()})
    b = oracle.mixer(p, [0, 3], **{k_: v_[2:] for k_, v_ in tk.items()}, S_in=a["S"], ring_in=a["ring"])
    np.testing.assert_allclose(np.concatenate([a["o"], b["o"]]), full["o"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(b["S"], full["S"], rtol=1e-12, atol=1e-14)


def test_p8_gate_bounds_and_special_values():
    """g = lb * sigmoid(exp(A_log) (z + dt_bias)) in (lb, 0); z = -dt_bias gives
    lb/2; g(z) + g(-z - 2 dt_bias) = lb; exp(A_log)(z + dt_bias) = ln 3 gives 3/4 lb."""
    rng = np.random.default_rng(8)
    H, D, T = 3, 4, 4
    W = H * D
    p = rand_params(rng, H, D)
    tk = rand_tokens(rng, T, H, D)
    tk["z"][1] = -p.dt_bias
    tk["z"][2] = -tk["z"][0] - 2 * p.dt_bias
    ea = np.repeat(np.exp(p.A_log), D)
    tk["z"][3] = np.log(3.0) / ea - p.dt_bias
    out = oracle.mixer(p, [0, T], **tk, intermediates=True)
    g = out["g"]
    # open interval in exact arithmetic; sigmoid saturates to 0 or 1 in fp64
    # once its argument passes about 37, so the rounded bounds are closed
    assert np.all(g >= -5.0) and np.all(g <= 0.0)
    arg = ea * (tk["z"] + p.dt_bias)
    mid = np.abs(arg) < 30
    assert np.all(g[mid] > -5.0) and np.all(g[mid] < 0.0)
    np.testing.assert_allclose(g[1], -2.5, rtol=0, atol=1e-15)
    np.testing.assert_allclose(g[0] + g[2], -5.0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(g[3], -3.75, rtol=0, atol=1e-14)
    np.testing.assert_allclose(out["beta"], sig(tk["b"]), rtol=1e-15)
    assert g.shape == (T, W)


def test_p8b_softplus_gate_special_values():
    """The earlier Kimi-Linear gate g = -exp(A_log) softplus(z + dt_bias):
    z = -dt_bias gives -exp(A_log) ln 2; z + dt_bias = ln(e - 1) gives
    -exp(A_log) (softplus = 1); far below zero g is -exp(A_log) e^{z + dt_bias}
    to first order; far above it is -exp(A_log) (z + dt_bias); always < 0."""
    rng = np.random.default_rng(81)
    H, D, T = 2, 4, 5
    p = rand_params(rng, H, D, gate_kind=1)
    tk = rand_tokens(rng, T, H, D)
    ea = np.repeat(np.exp(p.A_log), D)
    tk["z"][0] = -p.dt_bias
    tk["z"][1] = np.log(np.e - 1.0) - p.dt_bias
    tk["z"][2] = -40.0 - p.dt_bias
    tk["z"][3] = 60.0 - p.dt_bias
    out = oracle.mixer(p, [0, T], **tk, intermediates=True)
    g = out["g"]
    np.testing.assert_allclose(g[0], -ea * math.log(2.0), rtol=1e-15)
    np.testing.assert_allclose(g[1], -ea, rtol=1e-14)
    np.testing.assert_allclose(g[2], -ea * math.exp(-40.0), rtol=1e-15)   # e^x - e^{2x}/2 + ...
    np.testing.assert_allclose(g[3], -ea * 60.0, rtol=1e-15)              # x + e^{-x} - ...
    assert np.all(g < 0.0)
    # unbounded below: far past the -5 bound of the other gate
    assert np.all(g[3] < -5.0)


def test_p8c_softplus_gate_decay_only():
    """With beta = 0 and the softplus gate, the state only decays: after T
    tokens S = Diag(e^{sum_t g_t}) S0, with every g_t at a closed-form point:
    z + dt_bias = ln(e - 1) gives g = -exp(A_log), z + dt_bias = 0 gives
    g = -exp(A_log) ln 2."""
    rng = np.random.default_rng(82)
    H, D, T = 2, 4, 4
    p = rand_params(rng, H, D, gate_kind=1)
    tk = rand_tokens(rng, T, H, D)
    tk["b"][:] = -1e4                      # sigmoid underflows to exactly 0 in fp64
    tk["z"][0::2] = np.log(np.e - 1.0) - p.dt_bias
    tk["z"][1::2] = -p.dt_bias
    S0 = rng.standard_normal((1, H, D, D))
    out = oracle.mixer(p, [0, T], **tk, S_in=S0)
    ea = np.exp(p.A_log)
    for h in range(H):
        G = -ea[h] * (2 * 1.0 + 2 * math.log(2.0))   # two tokens of each kind
        np.testing.assert_allclose(out["S"][0, h], math.exp(G) * S0[0, h], rtol=1e-13)


def test_p9_rmsnorm_gated_constant_and_scale():
    """Constant input a with w = 1 and gate logit 0 gives a / sqrt(a^2+eps) / 2."""
    H, D = 2, 8
    for a in (0.5, -3.0, 1e-3):
        x = np.full((1, H * D), a)
        o = oracle.rmsnorm_gated(x, np.zeros_like(x), np.ones(D), H, eps=1e-5)
        np.testing.assert_allclose(o, a / math.sqrt(a * a + 1e-5) * 0.5, rtol=1e-14)
    # the normalised part has RMS sqrt(m / (m + eps)) for any w, gate
    rng = np.random.default_rng(9)
    x = rng.standard_normal((3, H * D))
    gate = rng.standard_normal((3, H * D))
    w = 1 + 0.3 * rng.standard_normal(D)
    o = oracle.rmsnorm_gated(x, gate, w, H, eps=1e-5)
    y = (o.reshape(3, H, D) / (w * sig(gate.reshape(3, H, D))))
    m = np.mean(x.reshape(3, H, D) ** 2, -1)
    np.testing.assert_allclose(np.sqrt(np.mean(y ** 2, -1)), np.sqrt(m / (m + 1e-5)), rtol=1e-13)


def test_p10_varlen_equals_separate_runs():
    rng = np.random.default_rng(10)
    H, D = 2, 8
    W = H * D
    p = rand_params(rng, H, D)
    lens = [7, 0, 3, 12, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    tk = rand_tokens(rng, int(cu[-1]), H, D)
    n = len(lens)
    S0 = rng.standard_normal((n, H, D, D)) * 0.2
    ring = rng.standard_normal((n, 3, 3, W))
    packed = oracle.mixer(p, cu, **tk, S_in=S0, ring_in=ring)
    for i in range(n):
        sl = slice(cu[i], cu[i + 1])
        one = oracle.mixer(p, [0, lens[i]], **{k_: v_[sl] for k_, v_ in tk.items()},
                           S_in=S0[i:i + 1], ring_in=ring[i:i + 1])
        np.testing.assert_array_equal(one["o"], packed["o"][sl])
        np.testing.assert_array_equal(one["S"][0], packed["S"][i])
        np.testing.assert_array_equal(one["ring"][0], packed["ring"][i])
    # a zero-length sequence hands its state and ring through unchanged
    np.testing.assert_array_equal(packed["S"][1], S0[1])
    np.testing.assert_array_equal(packed["ring"][1], ring[1])


def test_p10_head_permutation():
    rng = np.random.default_rng(12)
    H, D, T = 3, 4, 6
    p = rand_params(rng, H, D)
    tk = rand_tokens(rng, T, H, D)
    perm = np.array([2, 0, 1])
    ch = (perm[:, None] * D + np.arange(D)[None]).reshape(-1)
    p2 = oracle.Params(H, D, p.conv_w[:, ch], p.A_log[perm], p.dt_bias[ch], p.norm_w)
    tk2 = {k_: (v_[:, perm] if k_ == "b" else v_[:, ch]) for k_, v_ in tk.items()}
    a = oracle.mixer(p, [0, T], **tk)
    b = oracle.mixer(p2, [0, T], **tk2)
    np.testing.assert_array_equal(b["o"], a["o"][:, ch])
    np.testing.assert_array_equal(b["S"][0], a["S"][0][perm])


def test_p12_deterministic_and_thread_independent():
    rng = np.random.default_rng(13)
    H, D = 4, 16
    p = rand_params(rng, H, D)
    cu = [0, 20, 33]
    tk = rand_tokens(rng, 33, H, D)
    a = oracle.mixer(p, cu, **tk, nthreads=1)
    b = oracle.mixer(p, cu, **tk, nthreads=8)
    c = oracle.mixer(p, cu, **tk, nthreads=3)
    for key in ("o", "S", "ring"):
        np.testing.assert_array_equal(a[key], b[key])
        np.testing.assert_array_equal(a[key], c[key])


def test_ring_in_place_alias():
    """ring_out may alias ring_in (the CUDA ABI allows it; the oracle too)."""
    rng = np.random.default_rng(14)
    H, D = 1, 4
    p = rand_params(rng, H, D)
    tk = rand_tokens(rng, 2, H, D)
    ring = rng.standard_normal((1, 3, 3, H * D))
    ref = oracle.mixer(p, [0, 2], **tk, ring_in=ring.copy())
    np.testing.assert_array_equal(ref["ring"][0, :, 0], ring[0, :, 2])

def test_p13_recurrence_is_affine_in_its_starting_state():
    """The segment maps of a context-parallel split rest on this: over any run
    of tokens the final state is M S_0 + B with M independent of S_0 and of the
    values, and B independent of S_0 (each step is S <- (I - beta k k^T)
    Diag(e^g) S + beta k v^T).  Checked on the oracle's recurrence: the
    difference to the zero start is linear in S_0, unchanged when the values
    change, and the zero-start run is the values' part alone."""
    rng = np.random.default_rng(13)
    T, H, D = 24, 2, 8
    q, k, v, g, beta = rand_core(rng, T, H, D, g_lo=-0.05)
    beta = 0.2 * beta   # a long memory, so that the start still matters at the end
    S1, S2 = rng.standard_normal((2, H, D, D))
    zero = np.zeros((H, D, D))
    _, B = oracle.core(q, k, v, g, beta, zero)
    _, E1 = oracle.core(q, k, v, g, beta, S1)
    _, E2 = oracle.core(q, k, v, g, beta, S2)
    _, E12 = oracle.core(q, k, v, g, beta, 2.0 * S1 - 3.0 * S2)
    # linear part: M S for S1, S2 and a combination
    np.testing.assert_allclose(E12 - B, 2.0 * (E1 - B) - 3.0 * (E2 - B), rtol=0, atol=1e-12)
    # M does not depend on the values: the same difference with other values
    v2 = rng.standard_normal(v.shape)
    _, B2 = oracle.core(q, k, v2, g, beta, zero)
    _, E1b = oracle.core(q, k, v2, g, beta, S1)
    np.testing.assert_allclose(E1b - B2, E1 - B, rtol=0, atol=1e-12)
    # the part of the values alone: zero values give a zero offset
    _, B0 = oracle.core(q, k, np.zeros_like(v), g, beta, zero)
    np.testing.assert_allclose(B0, 0.0, atol=0)
    # the linear part is not trivial on these inputs (the start still matters)
    assert np.linalg.norm(E1 - B) > 0.1 * np.linalg.norm(S1)
    # and composing two runs' maps gives the whole run
    half = T // 2
    _, Bh1 = oracle.core(q[:half], k[:half], v[:half], g[:half], beta[:half], zero)
    _, Bh2 = oracle.core(q[half:], k[half:], v[half:], g[half:], beta[half:], zero)
    _, Eh2 = oracle.core(q[half:], k[half:], v[half:], g[half:], beta[half:], Bh1)
    np.testing.assert_allclose(Eh2, B, rtol=0, atol=1e-12)
    # the maps compose: M S_1 = M_2 (M_1 S_1), with M_i X the run from X minus
    # the run from zero (B_2 is what a context-parallel rank would send)
    _, E1h1 = oracle.core(q[:half], k[:half], v[:half], g[:half], beta[:half], S1)
    _, M2M1 = oracle.core(q[half:], k[half:], v[half:], g[half:], beta[half:], E1h1 - Bh1)
    np.testing.assert_allclose(M2M1 - Bh2, E1 - B, rtol=0, atol=1e-12)
