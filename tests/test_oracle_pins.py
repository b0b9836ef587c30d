"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test checks one oracle function against a hand-worked case, a closed form, an
invariant of the gated delta rule, a library routine, or brute force on tiny inputs,
chosen so that a dropped term, a wrong sign or index, or a transposed operand fails.
"""
import math
import os
import re

import numpy as np
import pytest
import scipy.special

import oracle
from gated_deltanet_layer_conv1d_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- golden cases
def _read_cases(path):
    """Parse the hand-worked fixture: `key value...` lines grouped by `case N`."""
    safe = {"sqrt": math.sqrt, "__builtins__": {}}

    def ev(tok):
        if not re.fullmatch(r"[0-9+\-*/(). sqrt]+", tok):
            raise ValueError(tok)
        return float(eval(tok, safe))  # noqa: S307 - fixture expressions: digits, + - * / sqrt

    cases, cur = [], None
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {}
                cases.append(cur)
            elif "|" in rest:
                cur[key] = np.array([[ev(t) for t in row.split()] for row in rest.split("|")])
            else:
                cur[key] = np.array([ev(t) for t in rest.split()])
    return cases


@pytest.mark.parametrize("idx", [0, 1])
def test_handworked_d4(idx):
    c = _read_cases(os.path.join(GOLDEN, "delta_rule_d4_handworked.txt"))[idx]
    S0 = c["S0"]
    # The oracle stores H = S^T ([d_k][d_v]).
    H1, o = oracle.delta_step(S0.T, c["q"], c["k"], c["v"], c["alpha"][0], c["beta"][0])
    np.testing.assert_allclose(H1.T, c["S1"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(o, c["o"], rtol=0, atol=1e-15)


# ---------------------------------------------------------------- a4 invariants
def _rand_head(rng, dk, dv):
    H = rng.standard_normal((dk, dv))
    q, k = rng.standard_normal(dk), rng.standard_normal(dk)
    v = rng.standard_normal(dv)
    return H, q, k, v


def test_beta0_alpha1_keeps_state():
    rng = np.random.default_rng(1)
    H, q, k, v = _rand_head(rng, 6, 5)
    H1, o = oracle.delta_step(H, q, k, v, 1.0, 0.0)
    np.testing.assert_array_equal(H1, H)
    np.testing.assert_allclose(o, H.T @ q, rtol=1e-14, atol=1e-14)


def test_alpha0_resets_state():
    rng = np.random.default_rng(2)
    H, q, k, v = _rand_head(rng, 6, 5)
    H1, o = oracle.delta_step(H, q, k, v, 0.0, 0.7)
    S1 = 0.7 * np.outer(v, k)
    np.testing.assert_allclose(H1.T, S1, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(o, S1 @ q, rtol=1e-13, atol=1e-13)


def test_delta_rule_stores_v_exactly():
    # With a unit key, beta = 1 and alpha = 1, reading the state at k returns v.
    rng = np.random.default_rng(3)
    H, q, k, v = _rand_head(rng, 8, 8)
    k = k / np.linalg.norm(k)
    H1, _ = oracle.delta_step(H, q, k, v, 1.0, 1.0)
    np.testing.assert_allclose(H1.T @ k, v, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("beta", [0.0, 0.5, 1.0, 1.5, 2.0])
def test_projection_is_contraction(beta):
    # For a unit k and beta in [0, 2], I - beta k k^T has spectral norm <= 1, so with
    # v = 0 and alpha = 1 the state's Frobenius norm cannot grow.
    rng = np.random.default_rng(4)
    H, q, k, _ = _rand_head(rng, 7, 9)
    k = k / np.linalg.norm(k)
    H1, _ = oracle.delta_step(H, q, k, np.zeros(9), 1.0, beta)
    assert np.linalg.norm(H1) <= np.linalg.norm(H) * (1 + 1e-14)


@pytest.mark.parametrize("dk,dv,Hk,Hv", [(4, 4, 1, 1), (3, 5, 1, 2), (4, 6, 2, 4)])
def test_recurrence_brute_force_matrix_form(dk, dv, Hk, Hv):
    # Explicit d x d matrix products: S <- alpha S (I - beta k k^T) + beta v k^T, o = S q,
    # with value head h reading key head h // (Hv // Hk).
    rng = np.random.default_rng(5)
    T = 8
    dims = oracle.Dims(Hk, Hv, dk, dv, 4, 1.0, 1e-6, 1e-6)
    qn = rng.standard_normal((T, Hk, dk))
    kn = rng.standard_normal((T, Hk, dk))
    v = rng.standard_normal((T, Hv, dv))
    alpha = rng.uniform(0.05, 1.0, (T, Hv))
    beta = rng.uniform(0.0, 2.0, (T, Hv))
    H0 = rng.standard_normal((Hv, dk, dv))
    H, o, snap = oracle.recurrence(dims, qn, kn, v, alpha, beta, H0, snapshots=True)
    G = Hv // Hk
    for h in range(Hv):
        S = H0[h].T.copy()
        for t in range(T):
            k, q = kn[t, h // G], qn[t, h // G]
            S = alpha[t, h] * S @ (np.eye(dk) - beta[t, h] * np.outer(k, k)) \
                + beta[t, h] * np.outer(v[t, h], k)
            np.testing.assert_allclose(o[t, h], S @ q, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(snap[t, h].T, S, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(H[h].T, S, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- a1 gates
def test_gates_closed_form_at_zero_logit():
    # a = -dt_bias makes softplus(0) = ln 2, so alpha = 2 ** (-exp(A_log)); sigmoid(0) = 1/2.
    A_log = np.array([-1.0, -0.3, 0.0, 0.9])
    dt_bias = np.array([0.0, 0.5, -1.25, 2.0])
    a = -dt_bias[None, :]
    b = np.zeros((1, 4))
    alpha, beta = oracle.gates(a, b, A_log, dt_bias)
    np.testing.assert_allclose(alpha[0], 2.0 ** (-np.exp(A_log)), rtol=1e-15)
    np.testing.assert_array_equal(beta[0], 0.5)


def test_gates_against_library_softplus_sigmoid():
    rng = np.random.default_rng(6)
    a = rng.standard_normal((50, 8)) * 30.0  # includes the far tails of softplus
    b = rng.standard_normal((50, 8)) * 5.0
    A_log = rng.uniform(-1, 1, 8)
    dt_bias = rng.standard_normal(8)
    alpha, beta = oracle.gates(a, b, A_log, dt_bias)
    sp = np.logaddexp(0.0, a + dt_bias)  # library softplus
    np.testing.assert_allclose(alpha, np.exp(-np.exp(A_log) * sp), rtol=1e-13, atol=0)
    np.testing.assert_allclose(beta, scipy.special.expit(b), rtol=1e-15)
    assert oracle.softplus(800.0) == 800.0
    assert oracle.softplus(-800.0) == 0.0


# ---------------------------------------------------------------- a2 conv
def test_conv_matches_numpy_convolve():
    rng = np.random.default_rng(7)
    T, C, W = 13, 5, 4
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, W))
    state0 = rng.standard_normal((C, W))
    out, st, _ = oracle.conv(w, state0, x)
    for c in range(C):
        # The window of token t is (x[t-W+1] .. x[t]); inputs before t = 0 come from the
        # state's newest W - 1 entries.
        ext = np.concatenate([state0[c, 1:], x[:, c]])
        pre = np.convolve(ext, w[c, ::-1], mode="valid")  # library 1-D convolution
        np.testing.assert_allclose(out[:, c], scipy.special.expit(pre) * pre, rtol=1e-13,
                                   atol=1e-14)
        np.testing.assert_array_equal(st[c], x[-W:, c])


def test_conv_delta_input_reproduces_reversed_weights():
    T, C, W = 8, 3, 4
    w = np.arange(1.0, C * W + 1).reshape(C, W) / 10.0
    x = np.zeros((T, C))
    x[2, :] = 1.0
    out, _, _ = oracle.conv(w, np.zeros((C, W)), x)
    silu = lambda z: z * scipy.special.expit(z)
    for c in range(C):
        np.testing.assert_allclose(out[2:2 + W, c], silu(w[c, ::-1]), rtol=1e-15)
        np.testing.assert_array_equal(out[:2, c], 0.0)
        np.testing.assert_array_equal(out[2 + W:, c], 0.0)


def test_conv_state_rotation_exact_and_snapshots():
    rng = np.random.default_rng(8)
    C, W = 6, 4
    x = rng.standard_normal((3, C))
    s0 = rng.standard_normal((C, W))
    _, st, snap = oracle.conv(rng.standard_normal((C, W)), s0, x, snapshots=True)
    np.testing.assert_array_equal(snap[0], np.concatenate([s0[:, 1:], x[:1].T], axis=1))
    np.testing.assert_array_equal(snap[1], np.concatenate([s0[:, 2:], x[:2].T], axis=1))
    np.testing.assert_array_equal(st, np.concatenate([s0[:, 3:], x[:3].T], axis=1))


# ---------------------------------------------------------------- a3 / a7 norms
def test_l2norm_closed_form_and_split():
    dims = oracle.Dims(2, 4, 8, 3, 4, q_scale=0.25, l2_eps=0.0, norm_eps=1e-6)
    T = 2
    xc = np.zeros((T, dims.conv_dim))
    xc[:, 0:8] = -3.0            # q of key head 0: constant vector
    xc[:, 8:16] = np.arange(8)   # q of key head 1
    xc[:, 16:24] = 2.0           # k of key head 0
    xc[:, 24:32] = 1.0           # k of key head 1
    xc[:, 32:] = np.arange(12)   # v
    qn, kn, v = oracle.l2norm_split(dims, xc)
    np.testing.assert_allclose(qn[:, 0], -0.25 / math.sqrt(8), rtol=1e-15)
    np.testing.assert_allclose(qn[:, 1], np.tile(0.25 * np.arange(8) / math.sqrt(140), (T, 1)),
                               rtol=1e-14)
    np.testing.assert_allclose(kn[:, 0], 1 / math.sqrt(8), rtol=1e-15)
    np.testing.assert_allclose(kn[:, 1], 1 / math.sqrt(8), rtol=1e-15)
    np.testing.assert_array_equal(v[0].reshape(-1), np.arange(12))


def test_l2norm_eps():
    dims = oracle.Dims(1, 1, 4, 4, 4, q_scale=1.0, l2_eps=1e-6, norm_eps=1e-6)
    xc = np.zeros((1, dims.conv_dim))
    xc[0, 0:4] = 1e-3
    qn, _, _ = oracle.l2norm_split(dims, xc)
    np.testing.assert_allclose(qn[0, 0], 1e-3 / math.sqrt(4e-6 + 1e-6), rtol=1e-15)


def test_gated_rmsnorm_closed_forms():
    dv, eps = 8, 1e-6
    w = np.linspace(0.5, 1.5, dv)
    z = np.linspace(-3, 3, dv)
    silu = z * scipy.special.expit(z)
    for c in (-2.0, 0.5, 3.0):
        o = np.full((1, 1, dv), c)
        y = oracle.gated_rmsnorm(o, z[None], w, eps)
        np.testing.assert_allclose(y[0], c / math.sqrt(c * c + eps) * w * silu, rtol=1e-14)
    o = np.array([1.0, -1.0] * (dv // 2)).reshape(1, 1, dv) * 5.0
    y = oracle.gated_rmsnorm(o, z[None], w, eps)
    np.testing.assert_allclose(y[0], o[0, 0] / math.sqrt(25 + eps) * w * silu, rtol=1e-14)


def test_gated_rmsnorm_sigmoid_gate_closed_forms():
    """The gdn_norm_sigmoid models' gate (layer_struct.rs, gated_rms_norm_f32_strided_k):
    sigmoid(z) in place of SiLU(z); with a constant o the norm part is sign(c) up to eps."""
    dv, eps = 8, 1e-6
    w = np.linspace(0.5, 1.5, dv)
    z = np.linspace(-3, 3, dv)
    for c in (-2.0, 0.5, 3.0):
        o = np.full((1, 1, dv), c)
        y = oracle.gated_rmsnorm(o, z[None], w, eps, gate=1)
        np.testing.assert_allclose(y[0], c / math.sqrt(c * c + eps) * w * scipy.special.expit(z),
                                   rtol=1e-14)
    # z = 0 halves the normalised row under the sigmoid gate and zeroes it under SiLU
    o = np.random.default_rng(5).standard_normal((3, 2, dv))
    zero = np.zeros((3, 2 * dv))
    y1 = oracle.gated_rmsnorm(o, zero, w, eps, gate=1).reshape(3, 2, dv)
    rms = np.sqrt((o * o).mean(-1, keepdims=True) + eps)
    np.testing.assert_allclose(y1, 0.5 * o / rms * w, rtol=1e-14)
    assert not oracle.gated_rmsnorm(o, zero, w, eps, gate=0).any()


def test_mixer_norm_gate_option_reaches_the_norm():
    """Through the whole mixer, SiLU(z) = z sigmoid(z) ties the two gates' outputs:
    y_silu = z * y_sigmoid element by element, with o and the state unchanged."""
    shape = wl.TINY
    rng = np.random.default_rng(17)
    T = 6
    toks = wl.make_tokens(rng, shape, T, bf16=False)
    wts = wl.make_weights(rng, shape)
    conv0 = rng.standard_normal((shape.conv_dim, shape.d_conv))
    H0 = rng.standard_normal((shape.n_v_heads, shape.d_k, shape.d_v)) * 0.1
    base = dict(n_k_heads=shape.n_k_heads, n_v_heads=shape.n_v_heads, d_k=shape.d_k,
                d_v=shape.d_v, d_conv=shape.d_conv, q_scale=shape.q_scale, l2_eps=1e-6,
                norm_eps=1e-6)
    r0 = oracle.mixer(oracle.Dims(**base), wts, toks["qkv"], toks["z"], toks["a"], toks["b"],
                      conv0.copy(), H0.copy())
    r1 = oracle.mixer(oracle.Dims(**base, norm_gate=1), wts, toks["qkv"], toks["z"], toks["a"],
                      toks["b"], conv0.copy(), H0.copy())
    np.testing.assert_array_equal(r0.o, r1.o)
    np.testing.assert_array_equal(r0.H, r1.H)
    np.testing.assert_allclose(r0.y, toks["z"] * r1.y, rtol=1e-12, atol=1e-300)


# ---------------------------------------------------------------- chunked == loop
def _prepared(rng, dims, T, alpha_lo=0.05):
    qn = rng.standard_normal((T, dims.n_k_heads, dims.d_k))
    kn = rng.standard_normal((T, dims.n_k_heads, dims.d_k))
    kn /= np.linalg.norm(kn, axis=-1, keepdims=True)
    qn /= np.linalg.norm(qn, axis=-1, keepdims=True)
    v = rng.standard_normal((T, dims.n_v_heads, dims.d_v))
    alpha = rng.uniform(alpha_lo, 1.0, (T, dims.n_v_heads))
    beta = rng.uniform(0.0, 1.0, (T, dims.n_v_heads))
    H0 = rng.standard_normal((dims.n_v_heads, dims.d_k, dims.d_v)) * 0.3
    return qn, kn, v, alpha, beta, H0


@pytest.mark.parametrize("C", [1, 2, 4, 64])
@pytest.mark.parametrize("dk,dv", [(16, 16), (8, 12)])
def test_chunked_equals_token_loop(C, dk, dv):
    rng = np.random.default_rng(9)
    dims = oracle.Dims(1, 2, dk, dv, 4, 1.0, 1e-6, 1e-6)
    T = 70  # not a multiple of any C above 2: the last chunk is ragged
    qn, kn, v, alpha, beta, H0 = _prepared(rng, dims, T)
    H_seq, o_seq, _ = oracle.recurrence(dims, qn, kn, v, alpha, beta, H0)
    H_ch, o_ch = oracle.chunked(dims, C, qn, kn, v, alpha, beta, H0)
    np.testing.assert_allclose(o_ch, o_seq, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(H_ch, H_seq, rtol=1e-10, atol=1e-11)


def test_chunked_strong_decay_stays_finite():
    # Cumulative log decay inside one 64-token chunk reaches about -440: every ratio must be
    # formed as exp(g_r - g_s) with r >= s.
    rng = np.random.default_rng(10)
    dims = oracle.Dims(1, 2, 16, 16, 4, 1.0, 1e-6, 1e-6)
    T = 64
    qn, kn, v, alpha, beta, H0 = _prepared(rng, dims, T)
    alpha[:] = 1e-3
    alpha[::7] = 0.999
    H_seq, o_seq, _ = oracle.recurrence(dims, qn, kn, v, alpha, beta, H0)
    H_ch, o_ch = oracle.chunked(dims, 64, qn, kn, v, alpha, beta, H0)
    assert np.isfinite(o_ch).all() and np.isfinite(H_ch).all()
    np.testing.assert_allclose(o_ch, o_seq, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(H_ch, H_seq, rtol=1e-9, atol=1e-12)


def test_chunked_bf16_operand_emulation_is_close_not_exact():
    rng = np.random.default_rng(11)
    dims = oracle.Dims(1, 2, 16, 16, 4, 1.0, 1e-6, 1e-6)
    qn, kn, v, alpha, beta, H0 = _prepared(rng, dims, 64, alpha_lo=0.5)
    H_seq, o_seq, _ = oracle.recurrence(dims, qn, kn, v, alpha, beta, H0)
    H_r, o_r = oracle.chunked(dims, 64, qn, kn, v, alpha, beta, H0, round_operands=True)
    rel = np.linalg.norm(o_r - o_seq) / np.linalg.norm(o_seq)
    assert 1e-5 < rel < 2e-2


# ---------------------------------------------------------------- mixer composition
def _tiny_mixer_inputs(T, shape=wl.TINY, seed=12, zero=False):
    rng = np.random.default_rng(seed)
    w = wl.make_weights(rng, shape)
    w["dt_bias"] = rng.standard_normal(shape.n_v_heads).astype(np.float32)
    H0, c0 = wl.make_states(rng, shape, 1, bf16=False, zero=zero)
    tok = wl.make_tokens(rng, shape, T, bf16=False)
    dims = oracle.Dims(shape.n_k_heads, shape.n_v_heads, shape.d_k, shape.d_v, shape.d_conv,
                       shape.q_scale, shape.l2_eps, shape.norm_eps)
    return dims, w, H0[0], c0[0], tok


def test_mixer_token_at_a_time_equals_block():
    T = 9
    dims, w, H0, c0, tok = _tiny_mixer_inputs(T)
    full = oracle.mixer(dims, w, tok["qkv"], tok["z"], tok["a"], tok["b"], c0, H0,
                        snapshots=True)
    H, cs = H0, c0
    for t in range(T):
        r = oracle.mixer(dims, w, tok["qkv"][t:t + 1], tok["z"][t:t + 1], tok["a"][t:t + 1],
                         tok["b"][t:t + 1], cs, H)
        H, cs = r.H, r.conv_state
        # verify semantics: the intermediate after t+1 tokens equals t+1 single steps
        np.testing.assert_array_equal(full.H_snap[t], H)
        np.testing.assert_array_equal(full.conv_snap[t], cs)
        np.testing.assert_array_equal(full.y[t], r.y[0])
    np.testing.assert_array_equal(full.H, H)
    np.testing.assert_array_equal(full.conv_state, cs)


@pytest.mark.parametrize("Hk,Hv", [(1, 2), (2, 4)])
def test_mixer_brute_force_numpy(Hk, Hv):
    """An independent numpy version of the whole mixer (library convolution, explicit
    matrix-form recurrence, direct norms) at tiny sizes."""
    shape = wl.LayerShape(Hk, Hv, 4, 5, 4, q_scale=0.7)
    T = 6
    dims, w, H0, c0, tok = _tiny_mixer_inputs(T, shape)
    r = oracle.mixer(dims, w, tok["qkv"], tok["z"], tok["a"], tok["b"], c0, H0)
    # Widen every input exactly to float64 before the numpy arithmetic.
    w = {k: v.astype(np.float64) for k, v in w.items()}
    tok = {k: v.astype(np.float64) for k, v in tok.items()}
    H0, c0 = H0.astype(np.float64), c0.astype(np.float64)
    dk, dv, W = 4, 5, 4
    C = shape.conv_dim
    sig = scipy.special.expit
    x = tok["qkv"].astype(np.float64)
    xc = np.empty((T, C))
    for c in range(C):
        ext = np.concatenate([c0[c, 1:], x[:, c]])
        pre = np.convolve(ext, w["conv_w"][c, ::-1].astype(np.float64), mode="valid")
        xc[:, c] = pre * sig(pre)
    S = [H0[h].T.astype(np.float64) for h in range(Hv)]
    G = Hv // Hk
    for t in range(T):
        for h in range(Hv):
            kh = h // G
            q = xc[t, kh * dk:(kh + 1) * dk]
            k = xc[t, Hk * dk + kh * dk:Hk * dk + (kh + 1) * dk]
            vv = xc[t, 2 * Hk * dk + h * dv:2 * Hk * dk + (h + 1) * dv]
            q = q / np.sqrt(q @ q + 1e-6) * 0.7
            k = k / np.sqrt(k @ k + 1e-6)
            al = np.exp(-np.exp(w["A_log"][h]) * np.logaddexp(0, tok["a"][t, h] + w["dt_bias"][h]))
            be = sig(tok["b"][t, h])
            S[h] = al * S[h] @ (np.eye(dk) - be * np.outer(k, k)) + be * np.outer(vv, k)
            o = S[h] @ q
            np.testing.assert_allclose(r.o[t, h], o, rtol=1e-12, atol=1e-13)
            zz = tok["z"][t, h * dv:(h + 1) * dv].astype(np.float64)
            y = o / np.sqrt(np.mean(o * o) + 1e-6) * w["norm_w"] * zz * sig(zz)
            np.testing.assert_allclose(r.y[t, h * dv:(h + 1) * dv], y, rtol=1e-12, atol=1e-13)
    for h in range(Hv):
        np.testing.assert_allclose(r.H[h].T, S[h], rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(r.conv_state, x[-W:].T)  # T >= W: last W raw inputs


def test_mixer_batch_matches_single():
    shape = wl.TINY
    seqs = []
    for i, T in enumerate([3, 1, 7]):
        dims, w, H0, c0, tok = _tiny_mixer_inputs(T, seed=20 + i)
        seqs.append(dict(tok, conv_state=c0, H=H0))
    res = oracle.mixer_batch(dims, w, seqs, snapshots=True)
    for s, r in zip(seqs, res):
        one = oracle.mixer(dims, w, s["qkv"], s["z"], s["a"], s["b"], s["conv_state"], s["H"],
                           snapshots=True)
        np.testing.assert_array_equal(r.y, one.y)
        np.testing.assert_array_equal(r.H, one.H)
        np.testing.assert_array_equal(r.H_snap, one.H_snap)
        np.testing.assert_array_equal(r.conv_state, one.conv_state)


def test_workload_bf16_rounding_is_ties_to_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.0000001, 3.0e-39], np.float32)
    r = wl.round_bf16(x)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even gives 1.
    assert r[0] == 1.0 and r[1] == 1.0 and r[2] == np.float32(1.015625)
    assert r[3] == -2.0
    assert (r.view(np.uint32) & 0xFFFF).max() == 0


# ---------------------------------------------------------------- binary16 state storage
def test_round_fp16_matches_numpy_half_conversion():
    rng = np.random.default_rng(11)
    xs = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 6, 4000),  # normals, subnormals
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e6, 2.0 ** -24,
                  2.0 ** -25, 3 * 2.0 ** -25, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25]),
    ])
    got = np.array([oracle.round_fp16(x) for x in xs])
    with np.errstate(over="ignore"):  # values past 65504 become inf, as they should
        ref = xs.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(got, ref)


def test_round_fp16_ties_go_to_even():
    u = 2.0 ** -10  # spacing of binary16 just above 1
    assert oracle.round_fp16(1.0 + u / 2) == 1.0            # tie between 1 and 1+u: even is 1
    assert oracle.round_fp16(1.0 + 3 * u / 2) == 1.0 + 2 * u  # tie: 1+2u has the even significand
    assert oracle.round_fp16(2.0 ** -25) == 0.0              # half the smallest subnormal
    assert oracle.round_fp16(3 * 2.0 ** -25) == 2.0 ** -23
    assert math.isinf(oracle.round_fp16(65520.0))            # the tie above 65504 overflows


def test_fp16_state_storage_rounds_every_stored_state_and_stays_close():
    rng = np.random.default_rng(12)
    dims = oracle.Dims(2, 4, 16, 16, 4, 0.25, 1e-6, 1e-6)
    dims16 = oracle.Dims(2, 4, 16, 16, 4, 0.25, 1e-6, 1e-6, h_fp16=True)
    T = 64
    qn = rng.standard_normal((T, 2, 16)); qn /= np.linalg.norm(qn, axis=-1, keepdims=True)
    kn = rng.standard_normal((T, 2, 16)); kn /= np.linalg.norm(kn, axis=-1, keepdims=True)
    v = rng.standard_normal((T, 4, 16))
    al = rng.uniform(0.5, 1.0, (T, 4))
    be = rng.uniform(0.0, 1.0, (T, 4))
    H0 = rng.standard_normal((4, 16, 16)).astype(np.float16).astype(np.float64)
    H, o, _ = oracle.recurrence(dims, qn, kn, v, al, be, H0)
    H16, o16, snap = oracle.recurrence(dims16, qn, kn, v, al, be, H0, snapshots=True)
    # every stored state is a binary16 value
    np.testing.assert_array_equal(snap, snap.astype(np.float16).astype(np.float64))
    np.testing.assert_array_equal(H16, snap[-1])
    # one rounding per token: far from exact, and within 64 half-ulps of the exact result
    e = np.linalg.norm(H16 - H) / np.linalg.norm(H)
    assert 1e-5 < e < 64 * 2.0 ** -11
    # the first output uses the unrounded update, so it equals the exact path's
    np.testing.assert_allclose(o16[0], o[0], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- projections
def test_proj_against_brute_force_loops():
    """layer_struct.rs, the bf16 in_proj / out_proj GEMMs: c[m][n] = sum_k x[m][k] w[n][k]
    (w holds one output feature per row); a non-square case so a transposed operand fails."""
    rng = np.random.default_rng(61)
    x = rng.standard_normal((3, 5))
    w = rng.standard_normal((7, 5))
    c = oracle.proj(x, w)
    assert c.shape == (3, 7)
    for m in range(3):
        for n in range(7):
            s = 0.0
            for k in range(5):
                s += x[m, k] * w[n, k]
            assert abs(c[m, n] - s) <= 1e-14 * (1.0 + abs(s))
    # a selection matrix copies the chosen features
    sel = np.zeros((2, 5))
    sel[0, 3] = sel[1, 0] = 1.0
    np.testing.assert_array_equal(oracle.proj(x, sel), x[:, [3, 0]])


def test_split_in_proj_layout():
    """[Q | K | V | Z | b | a]: every column lands in exactly one piece, in that order."""
    dims = oracle.Dims(2, 4, 8, 3, 4, 1.0, 1e-6, 1e-6)  # conv_dim 2*2*8 + 4*3 = 44
    width = oracle.in_proj_width(dims)
    assert width == 44 + 12 + 2 * 4
    rows = np.arange(2 * width, dtype=float).reshape(2, width)
    s = oracle.split_in_proj(dims, rows)
    assert [s[k].shape[1] for k in ("qkv", "z", "b", "a")] == [44, 12, 4, 4]
    np.testing.assert_array_equal(
        np.concatenate([s["qkv"], s["z"], s["b"], s["a"]], axis=1), rows)
    assert oracle.in_proj_width(dims) == wl.in_proj_width(
        wl.LayerShape(2, 4, 8, 3, 4, q_scale=1.0))
    # padding columns after a are not inputs
    padded = np.concatenate([rows, np.full((2, 8), 7.0)], axis=1)
    sp = oracle.split_in_proj(dims, padded)
    for k in ("qkv", "z", "b", "a"):
        np.testing.assert_array_equal(sp[k], s[k])


@pytest.mark.parametrize("shape", [wl.TINY, wl.LayerShape(2, 4, 16, 16, 4, q_scale=0.25)])
def test_woa_fold_of_the_stash_equals_the_state_after_m_tokens(shape):
    """Write-on-accept reading: replaying the stashed per-token factors of the first m draft
    tokens gives the state the token loop reaches after m tokens (the copy fold's state), for
    every m; the factors satisfy S_t = alpha_t S_{t-1} + delta_t k_hat_t^T exactly."""
    rng = np.random.default_rng(81)
    w = wl.make_weights(rng, shape)
    k = 9
    tok = wl.make_tokens(rng, shape, k, bf16=True)
    conv0 = wl.round_bf16(rng.standard_normal((shape.conv_dim, 4)).astype(np.float32) * 0.3)
    H0 = rng.standard_normal((shape.n_v_heads, shape.d_k, shape.d_v)) * 0.3
    d = oracle.Dims(shape.n_k_heads, shape.n_v_heads, shape.d_k, shape.d_v, 4,
                    float(np.float32(shape.q_scale)), 1e-6, 1e-6)
    r = oracle.mixer(d, w, tok["qkv"], tok["z"], tok["a"], tok["b"], conv0, H0, snapshots=True)
    alpha, k_hat, delta = oracle.woa_factors(d, w, tok["qkv"], tok["a"], tok["b"], conv0, H0)
    np.testing.assert_allclose(np.linalg.norm(k_hat, axis=-1), 1.0, rtol=1e-5)
    for m in range(1, k + 1):
        got = oracle.woa_fold(d, H0, alpha, k_hat, delta, m)
        np.testing.assert_allclose(got, r.H_snap[m - 1], rtol=1e-12, atol=1e-12)
    assert np.array_equal(oracle.woa_fold(d, H0, alpha, k_hat, delta, 0), H0)
    # a wrong sign or a dropped decay in the replay fails: replaying with alpha = 1 does not
    # reach the state after two tokens
    assert not np.allclose(oracle.woa_fold(d, H0, np.ones_like(alpha), k_hat, delta, 2),
                           r.H_snap[1], rtol=1e-6)
