"""Pins of the CPU oracle to facts other than itself (CPU only).

Each test ties one step of the oracle to something the pages or the
mathematics fix: a hand-derived fixture under tests/golden/, a closed form, a
special case that reduces to a library routine, or an algebraically
independent restatement (the Householder product form of the recurrence and
the dense chunked WY/UT form).  They are chosen so that a dropped term, a sign
or index slip or a transposed operand anywhere in the oracle fails one of them.
"""
import math

import numpy as np
import pytest
import torch

from conftest import golden_rows, rel_l2


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------- gates
def test_gates_hand_fixture(oracle_mod):
    rows = [list(map(float, r.split())) for r in golden_rows("gates_hand.txt")]
    a = np.array([[r[0]] for r in rows])
    dt_bias = np.array([r[1] for r in rows])
    A_log = np.array([r[2] for r in rows])
    b = np.array([[r[3]] for r in rows])
    for i, r in enumerate(rows):
        g, beta = oracle_mod.gates(a[i:i + 1], b[i:i + 1], A_log[i:i + 1], dt_bias[i:i + 1])
        assert g[0, 0] == pytest.approx(r[4], rel=1e-14, abs=0)
        assert beta[0, 0] == pytest.approx(r[5], rel=1e-15, abs=0)


def test_softplus_branches_continuous_and_finite(oracle_mod):
    a = np.array([[19.999999], [20.0], [20.000001], [-800.0], [800.0]])
    z = np.zeros((1,))
    g, beta = oracle_mod.gates(a, np.array([[0.0]] * 5), z, z)
    assert np.all(np.isfinite(g))
    # both sides of the switch agree to far below an f32 ulp at 20 (1.9e-6)
    assert abs(g[1, 0] - g[2, 0]) < 2e-6 and abs(g[0, 0] - g[1, 0]) < 2e-6
    assert g[3, 0] <= 0.0 and g[3, 0] > -1e-300  # large negative: g -> -0, no NaN
    assert g[4, 0] == -800.0
    b = np.array([[-np.inf], [np.inf]])
    _, beta = oracle_mod.gates(np.zeros((2, 1)), b, z, z)
    assert beta[0, 0] == 0.0 and beta[1, 0] == 1.0


# --------------------------------------------------------------------------- l2norm
def test_l2norm_hand_fixture(oracle_mod):
    for r in golden_rows("l2norm_hand.txt"):
        lhs, rhs = r.split("|")
        x = np.array([list(map(float, lhs.split()))])
        want = np.array([list(map(float, rhs.split()))])
        got = oracle_mod.l2norm(x)
        np.testing.assert_allclose(got, want, rtol=1e-15, atol=0)
    assert np.all(oracle_mod.l2norm(np.zeros((3, 128))) == 0.0)


# --------------------------------------------------------------------------- conv
def _conv_case(seed, lengths, C=6, K=4, state=True):
    r = _rng(seed)
    T = sum(lengths)
    x = r.standard_normal((T, C))
    w = r.standard_normal((C, K))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    st = r.standard_normal((len(lengths), C, K - 1)) if state else None
    return x, w, cu, st


def test_conv_onehot_current_tap_is_silu_of_input(oracle_mod):
    x, w, cu, st = _conv_case(1, [5, 1, 9])
    w[:] = 0.0
    w[:, 3] = 1.0
    y, _, _ = oracle_mod.conv1d(x, w, cu, st, apply_silu=True)
    np.testing.assert_allclose(y, x / (1.0 + np.exp(-x)), rtol=4e-16, atol=0)


def test_conv_onehot_oldest_tap_exposes_state_columns(oracle_mod):
    x, w, cu, st = _conv_case(2, [2, 7])
    w[:] = 0.0
    w[:, 0] = 1.0
    y, _, _ = oracle_mod.conv1d(x, w, cu, st, apply_silu=False)
    # sequence 0 has 2 tokens: y_t = column t of its state (col 0 oldest)
    np.testing.assert_array_equal(y[0], st[0, :, 0])
    np.testing.assert_array_equal(y[1], st[0, :, 1])
    # sequence 1: first 3 outputs are its state columns, then x delayed by 3
    for t in range(3):
        np.testing.assert_array_equal(y[2 + t], st[1, :, t])
    np.testing.assert_array_equal(y[5:9], x[2:6])


@pytest.mark.parametrize("state", [True, False])
def test_conv_random_matches_numpy_correlate(oracle_mod, state):
    lengths = [1, 2, 3, 17, 64]
    x, w, cu, st = _conv_case(3, lengths, C=5, state=state)
    y, so, _ = oracle_mod.conv1d(x, w, cu, st, apply_silu=False)
    K = w.shape[1]
    for i in range(len(lengths)):
        xs = x[cu[i]:cu[i + 1]]
        for c in range(x.shape[1]):
            head = st[i, c] if state else np.zeros(K - 1)
            ext = np.concatenate([head, xs[:, c]])
            ref = np.correlate(ext, w[c], mode="valid")  # cross-correlation, len L
            np.testing.assert_allclose(y[cu[i]:cu[i + 1], c], ref, rtol=1e-13, atol=1e-13)
            # state out = the K-1 newest raw values of [state | x], bit-exact
            np.testing.assert_array_equal(so[i, c], ext[-(K - 1):])


def test_conv_checkpoints_are_raw_inputs_at_multiples(oracle_mod):
    lengths = [130, 64, 63, 200]
    x, w, cu, st = _conv_case(4, lengths, C=3)
    N = 64
    _, _, ck = oracle_mod.conv1d(x, w, cu, st, ckpt_every=N)
    row = 0
    for i, L in enumerate(lengths):
        for m in range(1, L // N + 1):
            end = cu[i] + m * N
            np.testing.assert_array_equal(ck[row], x[end - 3:end].T)
            row += 1
    assert row == ck.shape[0] == 2 + 1 + 0 + 3


# --------------------------------------------------------------------------- delta rule
def _dr_case(seed, T, H_k=1, H_v=1, d_k=4, d_v=3, N=1, with_S0=True, g_scale=0.3):
    r = _rng(seed)
    q = r.standard_normal((T, H_k, d_k))
    k = r.standard_normal((T, H_k, d_k))
    v = r.standard_normal((T, H_v, d_v))
    g = -g_scale * r.random((T, H_v))
    beta = r.random((T, H_v))
    S0 = r.standard_normal((N, H_v, d_k, d_v)) if with_S0 else None
    return q, k, v, g, beta, S0


def test_decay_closed_form_when_beta_zero(oracle_mod):
    """beta = 0: the state only decays, S_T = exp(sum g) S0 and
    o_t = exp(G_t) S0^T (scale * q_hat_t)."""
    q, k, v, g, beta, S0 = _dr_case(5, T=9, d_k=5, d_v=3)
    beta[:] = 0.0
    scale = 0.37
    o, S, _ = oracle_mod.delta_rule(q, k, v, g, beta, S0=S0, scale=scale)
    G = np.cumsum(g[:, 0])
    np.testing.assert_allclose(S[0, 0], math.exp(G[-1]) * S0[0, 0], rtol=1e-13)
    qh = q[:, 0] / np.sqrt((q[:, 0] ** 2).sum(-1, keepdims=True) + 1e-6)
    want = np.exp(G)[:, None] * (qh @ S0[0, 0]) * scale
    np.testing.assert_allclose(o[:, 0], want, rtol=1e-12, atol=1e-14)


def test_retrieval_query_equal_to_key_returns_value(oracle_mod):
    """g = 0, beta = 1, unit keys, scale 1, no l2norm: S^T k + |k|^2 (v - S^T k)
    = v, so a query equal to the token's own key reads back its value for any
    starting state."""
    q, k, v, g, beta, S0 = _dr_case(6, T=7, d_k=6, d_v=4)
    k[:, 0] /= np.linalg.norm(k[:, 0], axis=-1, keepdims=True)
    q[:] = k
    g[:] = 0.0
    beta[:] = 1.0
    o, _, _ = oracle_mod.delta_rule(q, k, v, g, beta, S0=S0, scale=1.0, l2norm_qk=False)
    np.testing.assert_allclose(o, v, rtol=1e-12, atol=1e-12)


def test_retrieval_orthonormal_keys_from_zero_state(oracle_mod):
    d = 8
    r = _rng(7)
    basis, _ = np.linalg.qr(r.standard_normal((d, d)))
    keys = basis.T  # rows orthonormal
    vals = r.standard_normal((d, 5))
    perm = r.permutation(d)
    # d writes (beta=1), then d reads (beta=0) in another order
    T = 2 * d
    k = np.zeros((T, 1, d))
    q = np.zeros((T, 1, d))
    v = np.zeros((T, 1, 5))
    beta = np.zeros((T, 1))
    k[:d, 0] = keys
    v[:d, 0] = vals
    beta[:d] = 1.0
    q[d:, 0] = keys[perm]
    k[d:, 0] = keys[0]  # irrelevant: beta = 0 on read tokens
    o, S, _ = oracle_mod.delta_rule(q, k, v, np.zeros((T, 1)), beta, scale=1.0, l2norm_qk=False)
    np.testing.assert_allclose(o[d:, 0], vals[perm], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S[0, 0], keys.T @ vals, rtol=1e-12, atol=1e-12)


def test_scalar_d1_hand_fixture(oracle_mod):
    rows = golden_rows("scalar_recurrence_d1.txt")
    s0 = float(rows[0].split()[1])
    data = np.array([list(map(float, r.split())) for r in rows[1:]])
    T = len(data)
    g = data[:, 0:1]
    k = data[:, 1].reshape(T, 1, 1)
    v = data[:, 2].reshape(T, 1, 1)
    beta = data[:, 3:4]
    q = data[:, 4].reshape(T, 1, 1)
    o, S, _ = oracle_mod.delta_rule(q, k, v, g, beta, S0=np.full((1, 1, 1, 1), s0), scale=1.0,
                                    l2norm_qk=False)
    np.testing.assert_allclose(o[:, 0, 0], data[:, 6], rtol=1e-15, atol=1e-15)
    assert S[0, 0, 0, 0] == pytest.approx(data[-1, 5], rel=1e-15)
    # every intermediate state via prefixes
    for t in range(T):
        _, St, _ = oracle_mod.delta_rule(q[:t + 1], k[:t + 1], v[:t + 1], g[:t + 1],
                                         beta[:t + 1], S0=np.full((1, 1, 1, 1), s0), scale=1.0,
                                         l2norm_qk=False)
        assert St[0, 0, 0, 0] == pytest.approx(data[t, 5], rel=1e-15)


def _householder(q, k, v, g, beta, S0):
    """Independent form: S_t = e^g (I - beta k k^T) S_{t-1} + beta k v^T."""
    S = S0.copy()
    out = []
    I = np.eye(S.shape[0])
    for t in range(len(g)):
        S = math.exp(g[t]) * (I - beta[t] * np.outer(k[t], k[t])) @ S + beta[t] * np.outer(k[t], v[t])
        out.append(S.T @ q[t])
    return np.array(out), S


@pytest.mark.parametrize("d_k,d_v,T", [(1, 1, 5), (2, 2, 4), (2, 3, 5), (3, 2, 3)])
def test_tiny_bruteforce_householder_form(oracle_mod, d_k, d_v, T):
    q, k, v, g, beta, S0 = _dr_case(10 + d_k * 7 + d_v, T=T, d_k=d_k, d_v=d_v)
    o, S, _ = oracle_mod.delta_rule(q, k, v, g, beta, S0=S0, scale=1.0, l2norm_qk=False)
    o2, S2 = _householder(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0[0, 0])
    np.testing.assert_allclose(o[:, 0], o2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(S[0, 0], S2, rtol=1e-13, atol=1e-13)


def chunked_dense(q, k, v, g, beta, S0, C, inverse=None):
    """Dense chunked (WY/UT) restatement of the delta rule for one head with
    pre-normalised q, k: per chunk, G = cumsum(g); A_ij = beta_i e^{G_i-G_j}
    k_i.k_j (j < i); T = (I + A)^-1 diag(beta); W = T diag(e^G) K; U = T V;
    U' = U - W S; O = diag(e^G) Q S + [(Q K^T) o e^{G_i-G_j} 1(j<=i)] U';
    S <- e^{G_n} S + (diag(e^{G_n - G_j}) K)^T U'.  numpy.linalg.solve does the
    triangular system, or `inverse(A)` = (I + A)^-1 when given."""
    L = len(g)
    S = S0.copy()
    O = np.zeros((L, v.shape[1]))
    for c0 in range(0, L, C):
        sl = slice(c0, min(c0 + C, L))
        Q, K, V, gg, bb = q[sl], k[sl], v[sl], g[sl], beta[sl]
        n = len(gg)
        G = np.cumsum(gg)
        low = np.tril(np.ones((n, n), dtype=bool))
        Dm = np.exp(np.where(low, G[:, None] - G[None, :], -np.inf))
        A = np.tril(bb[:, None] * Dm * (K @ K.T), -1)
        Tm = (np.linalg.solve(np.eye(n) + A, np.diag(bb)) if inverse is None
              else inverse(A) @ np.diag(bb))
        W = Tm @ (np.exp(G)[:, None] * K)
        Up = Tm @ V - W @ S
        O[sl] = np.exp(G)[:, None] * (Q @ S) + ((Q @ K.T) * Dm) @ Up
        S = math.exp(G[-1]) * S + (np.exp(G[-1] - G)[:, None] * K).T @ Up
    return O, S


@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_chunked_dense_restatement_equals_recurrence(oracle_mod, C):
    lengths = [100, 37, 64]
    T = sum(lengths)
    q, k, v, g, beta, S0 = _dr_case(20, T=T, H_k=1, H_v=2, d_k=16, d_v=8, N=3, g_scale=0.5)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    o, S, _ = oracle_mod.delta_rule(q, k, v, g, beta, cu, S0=S0, scale=0.25)
    qn = q / np.sqrt((q ** 2).sum(-1, keepdims=True) + 1e-6) * 0.25
    kn = k / np.sqrt((k ** 2).sum(-1, keepdims=True) + 1e-6)
    for i in range(3):
        sl = slice(cu[i], cu[i + 1])
        for h in range(2):
            O2, S2 = chunked_dense(qn[sl, 0], kn[sl, 0], v[sl, h], g[sl, h], beta[sl, h],
                                   S0[i, h], C)
            assert rel_l2(o[sl, h], O2) < 1e-12
            assert rel_l2(S[i, h], S2) < 1e-12


def test_head_map_is_repeat_interleave(oracle_mod):
    H_k, H_v = 2, 6
    q, k, v, g, beta, S0 = _dr_case(30, T=12, H_k=H_k, H_v=H_v, d_k=4, d_v=4)
    o, S, _ = oracle_mod.delta_rule(q, k, v, g, beta, S0=S0)
    kmap = torch.repeat_interleave(torch.arange(H_k), H_v // H_k).tolist()
    assert kmap == [0, 0, 0, 1, 1, 1]
    for h in range(H_v):
        kh = kmap[h]
        o1, S1, _ = oracle_mod.delta_rule(q[:, kh:kh + 1], k[:, kh:kh + 1], v[:, h:h + 1],
                                          g[:, h:h + 1], beta[:, h:h + 1], S0=S0[:, h:h + 1])
        np.testing.assert_array_equal(o[:, h], o1[:, 0])
        np.testing.assert_array_equal(S[:, h], S1[:, 0])
    # the other plausible map (h mod H_k) gives a different answer on head 1
    o_wrong, _, _ = oracle_mod.delta_rule(q[:, 1:2], k[:, 1:2], v[:, 1:2], g[:, 1:2],
                                          beta[:, 1:2], S0=S0[:, 1:2])
    assert not np.allclose(o[:, 1], o_wrong[:, 0])


def test_continuation_and_checkpoints(oracle_mod):
    """prefill(T) == prefill(T1) then prefill(T - T1) from the handed-off state
    == prefill(T1) then single-token steps; checkpoint m == the state after
    the first m*N tokens."""
    T, N = 200, 64
    q, k, v, g, beta, S0 = _dr_case(40, T=T, H_k=1, H_v=2, d_k=8, d_v=8)
    o, S, ck = oracle_mod.delta_rule(q, k, v, g, beta, S0=S0, ckpt_every=N)
    assert ck.shape[0] == 3
    for m in range(1, 4):
        _, Sm, _ = oracle_mod.delta_rule(q[:m * N], k[:m * N], v[:m * N], g[:m * N],
                                         beta[:m * N], S0=S0)
        np.testing.assert_array_equal(ck[m - 1], Sm[0])
    T1 = 77
    o1, S1, _ = oracle_mod.delta_rule(q[:T1], k[:T1], v[:T1], g[:T1], beta[:T1], S0=S0)
    o2, S2, _ = oracle_mod.delta_rule(q[T1:], k[T1:], v[T1:], g[T1:], beta[T1:], S0=S1)
    np.testing.assert_array_equal(np.concatenate([o1, o2]), o)
    np.testing.assert_array_equal(S2, S)
    St = S1
    for t in range(T1, T1 + 5):
        ot, St, _ = oracle_mod.delta_rule(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1],
                                          beta[t:t + 1], S0=St)
        np.testing.assert_array_equal(ot[0], o[t])


def test_linear_in_v_from_zero_state(oracle_mod):
    q, k, v, g, beta, _ = _dr_case(50, T=30, d_k=6, d_v=5)
    v2 = _rng(51).standard_normal(v.shape)
    o1, S1, _ = oracle_mod.delta_rule(q, k, v, g, beta)
    o2, S2, _ = oracle_mod.delta_rule(q, k, v2, g, beta)
    o3, S3, _ = oracle_mod.delta_rule(q, k, 2.5 * v + v2, g, beta)
    np.testing.assert_allclose(o3, 2.5 * o1 + o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S3, 2.5 * S1 + S2, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- RMSNormGated
def test_rmsnorm_gated_hand_fixture(oracle_mod):
    rows = [np.array(list(map(float, r.split()))) for r in golden_rows("rmsnorm_gated_hand.txt")]
    o, w, z, want = rows
    out = oracle_mod.rmsnorm_gated(o.reshape(1, 1, 3), z.reshape(1, 3), w)
    np.testing.assert_allclose(out[0], want, rtol=1e-15, atol=1e-300)


def test_rmsnorm_gated_constant_vector_and_zero_gate(oracle_mod):
    d = 16
    w = _rng(60).standard_normal(d)
    z = _rng(61).standard_normal((1, d))
    for c in (3.0, -0.5, 1e-4):
        o = np.full((1, 1, d), c)
        out = oracle_mod.rmsnorm_gated(o, z, w)
        want = math.copysign(math.sqrt(c * c / (c * c + 1e-6)), c) * w * z[0] / (1 + np.exp(-z[0]))
        np.testing.assert_allclose(out[0], want, rtol=1e-13)
    out0 = oracle_mod.rmsnorm_gated(_rng(62).standard_normal((2, 3, d)), np.zeros((2, 3 * d)), w)
    assert np.all(out0 == 0.0)


# --------------------------------------------------------------------------- whole layer
def test_tiny_layer_finite_and_decode_matches_prefill(oracle_mod):
    import workloads as W
    wl = W.WORKLOADS["tiny_f32"]
    s = wl.shape
    d = W.workload_inputs("tiny_f32")
    f = W.to_f64
    r = oracle_mod.layer_prefill(f(d["mixed_qkv"]), f(d["z"]), f(d["a"]), f(d["b"]),
                                 f(d["conv_w"]), f(d["A_log"]), f(d["dt_bias"]), f(d["norm_w"]),
                                 s.H_k, s.H_v, s.d_k, s.d_v)
    for key in ("y", "o", "S", "out", "conv_state"):
        assert np.all(np.isfinite(r[key])), key
    assert r["out"].shape == (64, 64) and r["S"].shape == (1, 4, 16, 16)
    # the first 40 tokens by prefill, then 24 single-token steps == full prefill
    T1 = 40
    x, z, a, b = (f(d[n]) for n in ("mixed_qkv", "z", "a", "b"))
    r1 = oracle_mod.layer_prefill(x[:T1], z[:T1], a[:T1], b[:T1], f(d["conv_w"]), f(d["A_log"]),
                                  f(d["dt_bias"]), f(d["norm_w"]), s.H_k, s.H_v, s.d_k, s.d_v)
    S, cs = r1["S"], r1["conv_state"]
    for t in range(T1, 64):
        out, S, cs, _ = oracle_mod.layer_decode_step(
            x[t:t + 1], z[t:t + 1], a[t:t + 1], b[t:t + 1], f(d["conv_w"]), f(d["A_log"]),
            f(d["dt_bias"]), f(d["norm_w"]), s.H_k, s.H_v, s.d_k, s.d_v, S, cs)
        np.testing.assert_allclose(out[0], r["out"][t], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S, r["S"], rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(cs, r["conv_state"])
