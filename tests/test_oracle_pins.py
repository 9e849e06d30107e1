"""Pins for the fp64 CPU oracle: closed forms, invariants, brute force, special
cases that reduce to textbook formulas or library routines, and a hand-worked
fixture.  None of these calls the CUDA path; none needs a GPU.

Each pin is chosen so that a plausible slip in the oracle (a dropped decay, a
wrong sign in the delta rule, decay on the wrong axis, read-out before the
update, q and k swapped) fails at least one of them; test_oracle_mutations.py
plants those slips in copies of the oracle and checks that they are caught.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, T, H, K, V, unit_k=False, g_zero=False, beta=None):
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, V))
    g = np.zeros((T, H, K)) if g_zero else np.maximum(-5.0, -np.logaddexp(0.0, rng.standard_normal((T, H, K))))
    b = rng.uniform(0.05, 1.0, (T, H)) if beta is None else np.full((T, H), float(beta))
    return q, k, v, g, b


# ---------------------------------------------------------------- closed form
def test_closed_form_single_token():
    """T=1, S0=0: S1 = beta k v^T and o = scale * beta (q.k) v (post-update read-out)."""
    rng = np.random.default_rng(11)
    for K, V in ((5, 3), (64, 64), (128, 128)):
        q, k, v, g, b = _rand(rng, 1, 3, K, V)
        scale = K ** -0.5
        o, s = oracle.kda_forward(q, k, v, g, b, scale=scale)
        for h in range(3):
            qk = float(q[0, h] @ k[0, h])
            np.testing.assert_allclose(o[0, h], scale * b[0, h] * qk * v[0, h], rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(s[0, h], b[0, h] * np.outer(k[0, h], v[0, h]), rtol=1e-13, atol=1e-15)
        assert np.abs(o).max() > 0  # a pre-update read-out would give exactly zero


def test_default_scale_is_inverse_sqrt_head_dim():
    rng = np.random.default_rng(12)
    q, k, v, g, b = _rand(rng, 3, 1, 64, 8)
    o1, _ = oracle.kda_forward(q, k, v, g, b)
    o2, _ = oracle.kda_forward(q, k, v, g, b, scale=0.125)
    np.testing.assert_array_equal(o1, o2)


# ---------------------------------------------------------------- invariants
def test_delta_rule_overwrites_value_under_key():
    """g=0, beta=1, |k|=1: after the step S^T k = v for any prior state."""
    rng = np.random.default_rng(13)
    K, V, H = 16, 7, 2
    for _ in range(5):
        q, k, v, g, b = _rand(rng, 1, H, K, V, unit_k=True, g_zero=True, beta=1.0)
        s0 = rng.standard_normal((1, H, K, V))
        _, s = oracle.kda_forward(q, k, v, g, b, initial_state=s0)
        for h in range(H):
            np.testing.assert_allclose(s[0, h].T @ k[0, h], v[0, h], rtol=1e-12, atol=1e-12)


def test_beta_zero_is_pure_channelwise_decay():
    """beta=0: S_T = Diag(exp(sum_t g_t)) S0 and o_t = scale (Diag(e^{G_t}) S0)^T q_t."""
    rng = np.random.default_rng(14)
    T, H, K, V = 9, 2, 6, 5
    q, k, v, g, b = _rand(rng, T, H, K, V, beta=0.0)
    s0 = rng.standard_normal((1, H, K, V))
    o, s = oracle.kda_forward(q, k, v, g, b, scale=0.3, initial_state=s0)
    G = np.cumsum(g, axis=0)
    for h in range(H):
        np.testing.assert_allclose(s[0, h], np.exp(G[-1, h])[:, None] * s0[0, h], rtol=1e-12)
        for t in range(T):
            want = 0.3 * (np.exp(G[t, h])[:, None] * s0[0, h]).T @ q[t, h]
            np.testing.assert_allclose(o[t, h], want, rtol=1e-11, atol=1e-14)


def _transition(k, g, b):
    K = k.shape[0]
    return (np.eye(K) - b * np.outer(k, k)) @ np.diag(np.exp(g))


def test_brute_force_transition_products():
    """S_t = M_t...M_1 S0 + sum_j (M_t...M_{j+1}) beta_j k_j v_j^T, M_j = (I - beta_j k_j k_j^T) Diag(e^{g_j})."""
    rng = np.random.default_rng(15)
    T, H, K, V = 7, 2, 4, 3
    q, k, v, g, b = _rand(rng, T, H, K, V)
    s0 = rng.standard_normal((1, H, K, V))
    scale = 0.7
    o, s = oracle.kda_forward(q, k, v, g, b, scale=scale, initial_state=s0)
    for h in range(H):
        for t in range(T):
            # S_t by the explicit product formula
            St = np.eye(K)
            for j in range(t + 1):
                St = _transition(k[j, h], g[j, h], b[j, h]) @ St
            St = St @ s0[0, h]
            for j in range(t + 1):
                P = np.eye(K)
                for i in range(j + 1, t + 1):
                    P = _transition(k[i, h], g[i, h], b[i, h]) @ P
                St = St + P @ (b[j, h] * np.outer(k[j, h], v[j, h]))
            np.testing.assert_allclose(o[t, h], scale * St.T @ q[t, h], rtol=1e-11, atol=1e-13)
            if t == T - 1:
                np.testing.assert_allclose(s[0, h], St, rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------- special cases
def test_scalar_decay_is_gated_delta_rule():
    """g equal across channels: the gated delta rule S_t = a_t (I - b k k^T) S_{t-1} + b k v^T."""
    rng = np.random.default_rng(16)
    T, K, V = 12, 8, 5
    q, k, v, _, b = _rand(rng, T, 1, K, V)
    a = rng.uniform(0.2, 1.0, T)
    g = np.repeat(np.log(a)[:, None, None], K, axis=2)
    o, s = oracle.kda_forward(q, k, v, g, b, scale=1.0)
    S = np.zeros((K, V))
    for t in range(T):
        kt = k[t, 0]
        S = a[t] * (np.eye(K) - b[t, 0] * np.outer(kt, kt)) @ S + b[t, 0] * np.outer(kt, v[t, 0])
        np.testing.assert_allclose(o[t, 0], S.T @ q[t, 0], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(s[0, 0], S, rtol=1e-11, atol=1e-13)


def test_plain_delta_rule_and_constant_state():
    rng = np.random.default_rng(17)
    T, K, V = 10, 6, 4
    q, k, v, g, b = _rand(rng, T, 1, K, V, g_zero=True)
    s0 = rng.standard_normal((1, 1, K, V))
    o, s = oracle.kda_forward(q, k, v, g, b, scale=1.0, initial_state=s0)
    S = s0[0, 0].copy()
    for t in range(T):  # Widrow-Hoff / delta rule: S += beta k (v - S^T k)^T
        S = S + b[t, 0] * np.outer(k[t, 0], v[t, 0] - S.T @ k[t, 0])
    np.testing.assert_allclose(s[0, 0], S, rtol=1e-11, atol=1e-12)
    # beta = 0 and g = 0: the state never changes and o_t = S0^T q_t
    o2, s2 = oracle.kda_forward(q, k, v, g, np.zeros_like(b), scale=1.0, initial_state=s0)
    np.testing.assert_array_equal(s2, s0)
    np.testing.assert_allclose(o2[:, 0], q[:, 0] @ s0[0, 0], rtol=1e-13)


def test_joint_linearity_in_values_and_initial_state():
    rng = np.random.default_rng(18)
    T, H, K, V = 8, 2, 5, 4
    q, k, v1, g, b = _rand(rng, T, H, K, V)
    v2 = rng.standard_normal(v1.shape)
    s1 = rng.standard_normal((1, H, K, V))
    s2 = rng.standard_normal((1, H, K, V))
    a1, a2 = 0.7, -1.9
    oa, sa = oracle.kda_forward(q, k, v1, g, b, initial_state=s1)
    ob, sb = oracle.kda_forward(q, k, v2, g, b, initial_state=s2)
    oc, sc = oracle.kda_forward(q, k, a1 * v1 + a2 * v2, g, b, initial_state=a1 * s1 + a2 * s2)
    np.testing.assert_allclose(oc, a1 * oa + a2 * ob, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(sc, a1 * sa + a2 * sb, rtol=1e-10, atol=1e-12)


def test_householder_norm_invariants():
    """beta=2, |k|=1, g=0, v=0: each step is a reflection, so ||S||_F is kept;
    beta in (0,1], g<=0, v=0: ||S||_F never grows."""
    rng = np.random.default_rng(19)
    T, K, V = 20, 6, 3
    q, k, v, g, b = _rand(rng, T, 1, K, V, unit_k=True, g_zero=True, beta=2.0)
    s0 = rng.standard_normal((1, 1, K, V))
    for t in range(1, T + 1):
        _, s = oracle.kda_forward(q[:t], k[:t], 0 * v[:t], g[:t], b[:t], initial_state=s0)
        assert abs(np.linalg.norm(s) - np.linalg.norm(s0)) < 1e-12 * np.linalg.norm(s0)
    q, k, v, g, b = _rand(rng, T, 1, K, V, unit_k=True)
    prev = np.linalg.norm(s0)
    for t in range(1, T + 1):
        _, s = oracle.kda_forward(q[:t], k[:t], 0 * v[:t], g[:t], b[:t], initial_state=s0)
        cur = np.linalg.norm(s)
        assert cur <= prev * (1 + 1e-13)
        prev = cur


def test_padding_tokens_leave_state_unchanged():
    rng = np.random.default_rng(20)
    T, P, H, K, V = 5, 4, 2, 6, 5
    q, k, v, g, b = _rand(rng, T, H, K, V)
    s0 = rng.standard_normal((1, H, K, V))
    o, s = oracle.kda_forward(q, k, v, g, b, initial_state=s0)
    pad = lambda a: np.concatenate([a, np.zeros((P,) + a.shape[1:])], axis=0)  # noqa: E731
    op, sp = oracle.kda_forward(pad(q), pad(k), pad(v), pad(g), pad(b), initial_state=s0)
    np.testing.assert_array_equal(sp, s)
    np.testing.assert_array_equal(op[:T], o)
    assert not op[T:].any()


def test_varlen_equals_separate_sequences():
    rng = np.random.default_rng(21)
    lens = [3, 0, 9, 1, 6]
    H, K, V = 2, 5, 4
    T = sum(lens)
    q, k, v, g, b = _rand(rng, T, H, K, V)
    s0 = rng.standard_normal((len(lens), H, K, V))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, s = oracle.kda_forward(q, k, v, g, b, initial_state=s0, cu_seqlens=cu)
    for n in range(len(lens)):
        a, e = cu[n], cu[n + 1]
        on, sn = oracle.kda_forward(q[a:e], k[a:e], v[a:e], g[a:e], b[a:e], initial_state=s0[n:n + 1])
        np.testing.assert_array_equal(o[a:e], on)
        np.testing.assert_array_equal(s[n], sn[0])
    # an empty sequence returns its initial state
    np.testing.assert_array_equal(s[1], s0[1])


def test_decay_axis_is_key_channel_and_heads_are_independent():
    """Per-channel decay acts on rows (key channels) of S; permuting heads permutes outputs."""
    rng = np.random.default_rng(22)
    T, H, K, V = 6, 3, 8, 5
    q, k, v, _, b = _rand(rng, T, H, K, V)
    A = rng.uniform(-1, 1, K)  # one value per channel, shared by all heads
    g = -np.exp(A)[None, None, :] * rng.uniform(0.1, 1.0, (T, H, 1))
    s0 = rng.standard_normal((1, H, K, V))
    o, s = oracle.kda_forward(q, k, v, g, np.zeros_like(b), initial_state=s0)
    decay = np.exp(g.sum(0))  # [H, K]
    for h in range(H):
        np.testing.assert_allclose(s[0, h], decay[h][:, None] * s0[0, h], rtol=1e-12)
    perm = [2, 0, 1]
    o1, s1 = oracle.kda_forward(q, k, v, g, b, initial_state=s0)
    o2, s2 = oracle.kda_forward(q[:, perm], k[:, perm], v[:, perm], g[:, perm], b[:, perm],
                                initial_state=s0[:, perm])
    np.testing.assert_array_equal(o2, o1[:, perm])
    np.testing.assert_array_equal(s2, s1[:, perm])


# ---------------------------------------------------------------- golden fixture
def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, *nums = line.split()
                vals[key] = np.array([float(x) for x in nums])
    return vals


def test_hand_worked_fixture():
    gv = _read_golden("kda_hand_worked_t2.txt")
    st = lambda a, b: np.stack([gv[a], gv[b]])[:, None, :]  # noqa: E731  [T=2, H=1, D]
    beta = np.array([[gv["beta1"][0]], [gv["beta2"][0]]])
    o, s = oracle.kda_forward(st("q1", "q2"), st("k1", "k2"), st("v1", "v2"), st("g1", "g2"), beta,
                              scale=float(gv["scale"][0]))
    np.testing.assert_allclose(o[0, 0], gv["o1"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(o[1, 0], gv["o2"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(s[0, 0].ravel(), gv["S2"], rtol=0, atol=1e-14)


# ---------------------------------------------------------------- prologue pins
def test_short_conv_matches_numpy_convolve_with_restarts():
    rng = np.random.default_rng(30)
    lens = [5, 1, 8, 3]
    C, W = 7, 4
    x = rng.standard_normal((sum(lens), C))
    w = rng.standard_normal((C, W))
    cu = np.concatenate([[0], np.cumsum(lens)])
    y = oracle.short_conv(x, w, cu_seqlens=cu)
    for n in range(len(lens)):
        a, e = cu[n], cu[n + 1]
        for c in range(C):
            # causal: tap W-1 multiplies the current token, tap 0 the token W-1 steps back
            want = np.convolve(x[a:e, c], w[c, ::-1])[: e - a]
            np.testing.assert_allclose(y[a:e, c], want, rtol=1e-13, atol=1e-14)
    ys = oracle.short_conv(x, w, cu_seqlens=cu, act=1)
    np.testing.assert_allclose(ys, y * (0.5 * (1 + np.tanh(0.5 * y))), rtol=1e-12, atol=1e-14)


def test_short_conv_one_hot_tap_is_identity():
    rng = np.random.default_rng(31)
    x = rng.standard_normal((2, 11, 6))
    w = np.zeros((6, 4))
    w[:, 3] = 1.0
    np.testing.assert_array_equal(oracle.short_conv(x, w), x)
    w = np.zeros((6, 4))
    w[:, 2] = 1.0  # one-token delay, zero at the start of each of the 2 sequences
    y = oracle.short_conv(x, w)
    np.testing.assert_array_equal(y[:, 1:], x[:, :-1])
    assert not y[:, 0].any()


def test_l2norm_matches_linalg_norm():
    rng = np.random.default_rng(32)
    x = rng.standard_normal((5, 3, 128)) * 3.0
    y = oracle.l2norm(x, eps=0.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(y, x / np.linalg.norm(x, axis=-1, keepdims=True), rtol=1e-14)
    y = oracle.l2norm(x, eps=1e-6)
    np.testing.assert_allclose(y, x / np.sqrt(np.linalg.norm(x, axis=-1, keepdims=True) ** 2 + 1e-6),
                               rtol=1e-13)


def test_gate_special_cases():
    rng = np.random.default_rng(33)
    T, H, K = 7, 3, 16
    x = rng.standard_normal((T, H, K)) * 3
    zero_bias = np.zeros(H * K)
    # A_log = 0, dt_bias = 0: g = max(-5, -softplus(x)), softplus from numpy.logaddexp
    g = oracle.gate(x, np.zeros(K), zero_bias)
    np.testing.assert_allclose(g, np.maximum(-5.0, -np.logaddexp(0.0, x)), rtol=1e-14)
    assert g.max() <= 0.0
    # large inputs hit the lower bound exactly
    g = oracle.gate(np.full((1, H, K), 50.0), np.zeros(K), zero_bias)
    assert np.all(g == -5.0)
    # A_log = ln(a_c) per channel, shared across heads: g = max(-5, -a_c softplus(x))
    a = rng.uniform(0.2, 2.0, K)
    g = oracle.gate(x, np.log(a), zero_bias)
    np.testing.assert_allclose(g, np.maximum(-5.0, -a[None, None, :] * np.logaddexp(0.0, x)), rtol=1e-13)
    # dt_bias is indexed [h*K + c]: a bias on head 1 alone changes only head 1
    db = np.zeros(H * K)
    db[K:2 * K] = rng.uniform(-1, 1, K)
    g0 = oracle.gate(x, np.zeros(K), zero_bias)
    g1 = oracle.gate(x, np.zeros(K), db)
    np.testing.assert_array_equal(g1[:, [0, 2]], g0[:, [0, 2]])
    np.testing.assert_allclose(g1[:, 1], np.maximum(-5.0, -np.logaddexp(0.0, x[:, 1] + db[K:2 * K])),
                               rtol=1e-14)


def test_prologue_composition():
    rng = np.random.default_rng(34)
    B, T, H, K, V = 1, 9, 2, 8, 4
    qr, kr, gx = (rng.standard_normal((B, T, H, K)) for _ in range(3))
    vr = rng.standard_normal((B, T, H, V))
    wq, wk = rng.standard_normal((H * K, 4)), rng.standard_normal((H * K, 4))
    wv = rng.standard_normal((H * V, 4))
    A, db = rng.uniform(-1, 1, K), rng.uniform(-1, 1, H * K)
    q, k, v, g = oracle.prologue(qr, kr, vr, gx, (wq, wk, wv), A, db)
    for h in range(H):
        conv = np.stack([np.convolve(qr[0, :, h, c], wq[h * K + c, ::-1])[:T] for c in range(K)], -1)
        want = conv / np.sqrt(np.sum(conv * conv, axis=-1, keepdims=True) + 1e-6)
        np.testing.assert_allclose(q[0, :, h], want, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(np.linalg.norm(q, axis=-1), 1.0, rtol=1e-5)
    np.testing.assert_allclose(np.linalg.norm(k, axis=-1), 1.0, rtol=1e-5)
    np.testing.assert_allclose(v.reshape(T, H * V), oracle.short_conv(vr.reshape(T, H * V), wv), rtol=0)
    np.testing.assert_allclose(g, oracle.gate(gx, A, db), rtol=0)
    assert np.all((g <= 0) & (g >= -5))


@pytest.mark.parametrize("nthreads", [1, 3])
def test_thread_count_does_not_change_results(nthreads):
    rng = np.random.default_rng(40)
    q, k, v, g, b = _rand(rng, 17, 5, 8, 6)
    o1, s1 = oracle.kda_forward(q, k, v, g, b, nthreads=1)
    o2, s2 = oracle.kda_forward(q, k, v, g, b, nthreads=nthreads)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2)


# ---------------------------------------------------------------- output gate
def _og_inputs(rng, rows=7, V=16):
    return rng.standard_normal((rows, V)), rng.standard_normal((rows, V)), rng.uniform(0.5, 1.5, V)


def test_output_gate_homogeneous_of_degree_zero_in_o():
    """eps = 0: scaling a row of o by c > 0 leaves the output unchanged; c < 0 flips it."""
    rng = np.random.default_rng(41)
    o, g, w = _og_inputs(rng)
    base = oracle.output_gate(o, g, w, eps=0.0)
    np.testing.assert_allclose(oracle.output_gate(3.7 * o, g, w, eps=0.0), base, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(oracle.output_gate(-0.2 * o, g, w, eps=0.0), -base, rtol=1e-13, atol=1e-15)


def test_output_gate_sigmoid_reflection():
    """sigmoid(x) + sigmoid(-x) = 1 and sigmoid(x) / sigmoid(-x) = e^x: the outputs for
    gate and -gate add up to the normed, weighted row and their ratio is e^gate."""
    rng = np.random.default_rng(42)
    o, g, w = _og_inputs(rng)
    a = oracle.output_gate(o, g, w, eps=1e-3)
    b = oracle.output_gate(o, -g, w, eps=1e-3)
    full = oracle.output_gate(o, np.full_like(g, 60.0), w, eps=1e-3)  # sigmoid(60) = 1 in fp64
    np.testing.assert_allclose(a + b, full, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(a / b, np.exp(g), rtol=1e-12)


def test_output_gate_rows_have_unit_rms():
    """eps = 0, weight 1, gate open: every output row has root-mean-square 1 (an RMS
    norm over the V channels, not over their sum)."""
    rng = np.random.default_rng(43)
    for V in (16, 64, 128):
        o = rng.standard_normal((5, V)) * rng.uniform(0.01, 100.0, (5, 1))
        out = oracle.output_gate(o, np.full((5, V), 60.0), None, eps=0.0)
        np.testing.assert_allclose(np.sqrt(np.mean(out * out, axis=-1)), 1.0, rtol=1e-13)


def test_output_gate_channel_equivariance_and_weight_linearity():
    """Permuting the channels of o, gate and weight permutes the output; the output is
    linear in the weight; rows are independent of one another."""
    rng = np.random.default_rng(44)
    o, g, w = _og_inputs(rng)
    base = oracle.output_gate(o, g, w)
    perm = rng.permutation(o.shape[1])
    np.testing.assert_allclose(oracle.output_gate(o[:, perm], g[:, perm], w[perm]), base[:, perm], rtol=1e-13)
    np.testing.assert_allclose(oracle.output_gate(o, g, 2.5 * w), 2.5 * base, rtol=1e-13)
    np.testing.assert_allclose(oracle.output_gate(o[::-1], g[::-1], w), base[::-1], rtol=1e-13)


def test_output_gate_constant_row_closed_form():
    """o = c (all V channels), gate 0, weight 1: out = c / sqrt(c^2 + eps) / 2."""
    for c, eps in ((0.5, 0.25), (-2.0, 1e-6), (1e-3, 1e-6)):
        out = oracle.output_gate(np.full((1, 8), c), np.zeros((1, 8)), None, eps=eps)
        np.testing.assert_allclose(out, c / np.sqrt(c * c + eps) / 2.0, rtol=1e-14)


# ---------------------------------------------------------------- segments (context parallelism)
def test_segment_composition_equals_the_whole_sequence():
    """Split a sequence into segments: the final state of the whole is reached by
    S_in(r+1) = M_r S_in(r) + S_zero_r, with M_r the product of the per-token
    factors and S_zero_r the segment's final state from a zero start; and the
    segment's final state from S_in is exactly M_r S_in + S_zero_r."""
    rng = np.random.default_rng(51)
    T, H, K, V = 23, 2, 6, 4
    q, k, v, g, b = _rand(rng, T, H, K, V)
    s0 = rng.standard_normal((1, H, K, V))
    _, s_all = oracle.kda_forward(q, k, v, g, b, initial_state=s0)
    s_in = s0[0]
    for a, e in ((0, 7), (7, 8), (8, 23)):
        sl = slice(a, e)
        _, s_zero = oracle.kda_forward(q[sl], k[sl], v[sl], g[sl], b[sl])
        M = oracle.segment_transition(k[sl], g[sl], b[sl])
        _, s_from = oracle.kda_forward(q[sl], k[sl], v[sl], g[sl], b[sl], initial_state=s_in[None])
        s_next = oracle.state_compose(M, s_in, s_zero[0])
        np.testing.assert_allclose(s_next, s_from[0], rtol=1e-12, atol=1e-12)
        s_in = s_next
    np.testing.assert_allclose(s_in, s_all[0], rtol=1e-12, atol=1e-12)


def test_segment_transition_special_cases():
    """beta = 0: M = Diag(exp(sum of g)); g = 0, beta = 1, one unit k: M = I - k k^T
    (a projector: M M = M); an empty segment: M = I."""
    rng = np.random.default_rng(52)
    T, H, K = 5, 2, 4
    _, k, _, g, _ = _rand(rng, T, H, K, 1)
    M = oracle.segment_transition(k, g, np.zeros((T, H)))
    for h in range(H):
        np.testing.assert_allclose(M[h], np.diag(np.exp(g[:, h].sum(axis=0))), rtol=1e-13, atol=1e-15)
    ku = k[:1] / np.linalg.norm(k[:1], axis=-1, keepdims=True)
    P = oracle.segment_transition(ku, np.zeros_like(ku), np.ones((1, H)))
    for h in range(H):
        np.testing.assert_allclose(P[h], np.eye(K) - np.outer(ku[0, h], ku[0, h]), atol=1e-15)
        np.testing.assert_allclose(P[h] @ P[h], P[h], atol=1e-14)
    np.testing.assert_allclose(oracle.segment_transition(k[:0], g[:0], np.zeros((0, H))),
                               np.broadcast_to(np.eye(K), (H, K, K)), atol=0)


# ---------------------------------------------------------------- backward
def _loss(q, k, v, g, b, s0, dO, dST, scale):
    o, sT = oracle.kda_forward(q, k, v, g, b, scale=scale, initial_state=s0)
    return float(np.sum(dO * o) + np.sum(dST * sT))


def test_backward_matches_central_differences():
    """Every gradient entry against a central difference of <dO, o> + <dS_T, S_T>
    (step 1e-6 in fp64), on a tiny chain crossing a 64-token checkpoint block."""
    rng = np.random.default_rng(91)
    for T, K, V in ((5, 3, 2), (70, 2, 2)):
        H = 1
        q, k, v, g, b = _rand(rng, T, H, K, V)
        s0 = rng.standard_normal((1, H, K, V))
        dO = rng.standard_normal((T, H, V))
        dST = rng.standard_normal((1, H, K, V))
        scale = 0.7
        gr = oracle.kda_backward(q, k, v, g, b, dO, dS_T=dST, scale=scale, initial_state=s0)
        args = {"q": q, "k": k, "v": v, "g": g, "beta": b, "s0": s0}
        names = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "s0": "dS0"}
        step = 1e-6
        for name, arr in args.items():
            flat = arr.reshape(-1)
            idx = range(flat.size) if flat.size <= 12 else rng.choice(flat.size, 12, replace=False)
            for i in idx:
                old = flat[i]
                flat[i] = old + step
                lp = _loss(q, k, v, g, b, s0, dO, dST, scale)
                flat[i] = old - step
                lm = _loss(q, k, v, g, b, s0, dO, dST, scale)
                flat[i] = old
                fd = (lp - lm) / (2 * step)
                an = gr[names[name]].reshape(-1)[i]
                assert abs(fd - an) <= 1e-6 * (1.0 + abs(fd)), (name, i, fd, an)


def test_backward_single_token_closed_forms():
    """T=1, S0=0, dS_T=0: o = scale beta (q.k) v, so dq = scale beta (v.dO) k,
    dk = scale beta (v.dO) q, dv = scale beta (q.k) dO, dbeta = scale (q.k)(v.dO),
    and dg = 0 (the decay acts on the zero state)."""
    rng = np.random.default_rng(92)
    K, V, scale = 4, 3, 0.5
    q, k, v, g, b = _rand(rng, 1, 1, K, V)
    dO = rng.standard_normal((1, 1, V))
    gr = oracle.kda_backward(q, k, v, g, b, dO, scale=scale)
    qk, vd, bt = float(q[0, 0] @ k[0, 0]), float(v[0, 0] @ dO[0, 0]), float(b[0, 0])
    np.testing.assert_allclose(gr["dq"][0, 0], scale * bt * vd * k[0, 0], rtol=1e-13)
    np.testing.assert_allclose(gr["dk"][0, 0], scale * bt * vd * q[0, 0], rtol=1e-13)
    np.testing.assert_allclose(gr["dv"][0, 0], scale * bt * qk * dO[0, 0], rtol=1e-13)
    np.testing.assert_allclose(gr["dbeta"][0, 0], scale * qk * vd, rtol=1e-13)
    np.testing.assert_allclose(gr["dg"][0, 0], 0.0, atol=1e-15)


def test_backward_adjoint_identity():
    """(o, S_T) is linear in (v, S0) for fixed q, k, g, beta, so for any (dO, dS_T)
    <dO, o> + <dS_T, S_T> = <dv, v> + <dS0, S0>."""
    rng = np.random.default_rng(93)
    T, H, K, V = 40, 2, 5, 4
    q, k, v, g, b = _rand(rng, T, H, K, V)
    s0 = rng.standard_normal((1, H, K, V))
    dO = rng.standard_normal((T, H, V))
    dST = rng.standard_normal((1, H, K, V))
    lhs = _loss(q, k, v, g, b, s0, dO, dST, K ** -0.5)
    gr = oracle.kda_backward(q, k, v, g, b, dO, dS_T=dST, initial_state=s0)
    rhs = float(np.sum(gr["dv"] * v) + np.sum(gr["dS0"] * s0))
    assert abs(lhs - rhs) <= 1e-10 * (1.0 + abs(lhs))


def test_backward_packed_equals_separate():
    """Packed sequences: each sequence's gradients are those of its own chain."""
    rng = np.random.default_rng(94)
    lens = [3, 0, 9, 5]
    T, H, K, V = sum(lens), 2, 3, 2
    q, k, v, g, b = _rand(rng, T, H, K, V)
    dO = rng.standard_normal((T, H, V))
    s0 = rng.standard_normal((len(lens), H, K, V))
    cu = np.concatenate([[0], np.cumsum(lens)])
    gr = oracle.kda_backward(q, k, v, g, b, dO, initial_state=s0, cu_seqlens=cu)
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        one = oracle.kda_backward(q[sl], k[sl], v[sl], g[sl], b[sl], dO[sl], initial_state=s0[n:n + 1])
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            np.testing.assert_allclose(gr[key][sl], one[key], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(gr["dS0"][n], one["dS0"][0], rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- gate projections
def _proj_inputs(rng, D, R, HK, NH, rows):
    return (rng.standard_normal((rows, D)), rng.standard_normal((R, D)), rng.standard_normal((HK, R)),
            rng.standard_normal((NH, D)))


def test_gate_proj_rank_one_is_an_outer_product():
    # f_a = a^T (one row), f_b = b (one column): gate_x_t = (a . x_t) b
    rng = np.random.default_rng(31)
    x, a, b, bp = _proj_inputs(rng, 7, 1, 6, 3, 4)
    gx, _ = oracle.gate_proj(x, a, b, bp)
    for t in range(4):
        s = 0.0
        for d in range(7):
            s += a[0, d] * x[t, d]
        for j in range(6):
            assert abs(gx[t, j] - s * b[j, 0]) <= 1e-12 * (1.0 + abs(s * b[j, 0]))


def test_gate_proj_brute_force_loops():
    rng = np.random.default_rng(32)
    D, R, HK, NH, rows = 5, 3, 4, 2, 3
    x, fa, fb, bp = _proj_inputs(rng, D, R, HK, NH, rows)
    gx, beta = oracle.gate_proj(x, fa, fb, bp)
    for t in range(rows):
        y = [sum(fa[i, d] * x[t, d] for d in range(D)) for i in range(R)]
        for j in range(HK):
            ref = sum(fb[j, i] * y[i] for i in range(R))
            assert abs(gx[t, j] - ref) <= 1e-12 * (1.0 + abs(ref))
        for h in range(NH):
            z = sum(bp[h, d] * x[t, d] for d in range(D))
            ref = np.exp(z) / (np.exp(z) + 1.0)   # the other form of the logistic function
            assert abs(beta[t, h] - ref) <= 1e-14


def test_gate_proj_beta_special_cases():
    rng = np.random.default_rng(33)
    x, fa, fb, bp = _proj_inputs(rng, 6, 2, 4, 3, 5)
    _, half = oracle.gate_proj(x, fa, fb, np.zeros_like(bp))
    assert np.all(half == 0.5)
    _, b1 = oracle.gate_proj(x, fa, fb, bp)
    _, b2 = oracle.gate_proj(x, fa, fb, -bp)
    np.testing.assert_allclose(b1 + b2, 1.0, rtol=0, atol=1e-15)   # sigmoid(-z) = 1 - sigmoid(z)
    assert np.all((b1 > 0.0) & (b1 < 1.0))


def test_gate_proj_is_linear_in_x_and_row_local():
    rng = np.random.default_rng(34)
    x1, fa, fb, bp = _proj_inputs(rng, 6, 3, 5, 2, 4)
    x2 = rng.standard_normal(x1.shape)
    g1, _ = oracle.gate_proj(x1, fa, fb, bp)
    g2, _ = oracle.gate_proj(x2, fa, fb, bp)
    g12, _ = oracle.gate_proj(x1 + 2.5 * x2, fa, fb, bp)
    np.testing.assert_allclose(g12, g1 + 2.5 * g2, rtol=1e-12, atol=1e-12)
    perm = np.array([2, 0, 3, 1])
    gp, bperm = oracle.gate_proj(x1[perm], fa, fb, bp)
    _, b1 = oracle.gate_proj(x1, fa, fb, bp)
    np.testing.assert_array_equal(gp, g1[perm])
    np.testing.assert_array_equal(bperm, b1[perm])
    # leading dimensions are rows: [B, T, D] -> [B, T, HK] and [B, T, NH]
    g3, b3 = oracle.gate_proj(x1.reshape(2, 2, 6), fa, fb, bp)
    assert g3.shape == (2, 2, 5) and b3.shape == (2, 2, 2)
    np.testing.assert_array_equal(g3.reshape(4, 5), g1)
