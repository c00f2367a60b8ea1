"""Pins of the fp64 recurrent oracle against facts fixed by the gated delta rule itself
(the FlashQLA pages print no tensors, so every pin comes from the definition, a closed form,
an invariant, an independent formulation or finite differences).

The rule (FlashQLA pages, "GDN chunked prefill optimisation"): S_t = exp(g_t) S_{t-1}
(I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = scale S_t q_t, with h = S^T stored
[K, V]."""
import json
import os

import numpy as np
import pytest

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(seed, T=11, Hqk=1, Hv=2, K=8, V=12, B=1, unit_k=True, h0=True, beta01=True):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, T, Hqk, K))
    k = r.standard_normal((B, T, Hqk, K))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = r.standard_normal((B, T, Hv, V))
    g = -np.log1p(np.exp(r.standard_normal((B, T, Hv))))
    beta = 1 / (1 + np.exp(-r.standard_normal((B, T, Hv)))) if beta01 else r.uniform(0, 1, (B, T, Hv))
    h0a = 0.3 * r.standard_normal((B, Hv, K, V)) if h0 else None
    return q, k, v, g, beta, h0a


def test_hand_worked_fixture():
    f = json.load(open(os.path.join(GOLDEN, "tiny_hand_worked.json")))
    sh = lambda x, d: np.array(x, np.float64).reshape(d)
    q = sh(f["q"], (1, 2, 1, 2)); k = sh(f["k"], (1, 2, 1, 2)); v = sh(f["v"], (1, 2, 1, 2))
    g = sh(f["g"], (1, 2, 1)); beta = sh(f["beta"], (1, 2, 1)); h0 = sh(f["h0"], (1, 1, 2, 2))
    o, ht = orc.fwd(q, k, v, g, beta, f["scale"], h0=h0)
    np.testing.assert_allclose(o.reshape(2, 2), np.array(f["o"]), atol=1e-14)
    np.testing.assert_allclose(ht.reshape(2, 2), np.array(f["ht"]), atol=1e-14)


def test_single_token_matrix_form():
    """T=1 in the S-space matrix form of the definition (catches a transposed state or a
    swapped decay/erase order)."""
    q, k, v, g, beta, h0 = rnd(1, T=1, K=5, V=7)
    o, ht = orc.fwd(q, k, v, g, beta, 0.7, h0=h0)
    for j in range(2):
        S0 = h0[0, j].T
        kk, vv, qq = k[0, 0, 0], v[0, 0, j], q[0, 0, 0]
        a, b = np.exp(g[0, 0, j]), beta[0, 0, j]
        S1 = a * S0 @ (np.eye(5) - b * np.outer(kk, kk)) + b * np.outer(vv, kk)
        np.testing.assert_allclose(ht[0, j], S1.T, atol=1e-13)
        np.testing.assert_allclose(o[0, 0, j], 0.7 * S1 @ qq, atol=1e-13)


def test_beta_zero_pure_decay():
    q, k, v, g, beta, h0 = rnd(2, T=13)
    beta[:] = 0.0
    o, ht = orc.fwd(q, k, v, g, beta, 0.5, h0=h0)
    gam = np.cumsum(g[0], axis=0)  # [T, Hv]
    for j in range(2):
        for t in range(13):
            ref = 0.5 * np.exp(gam[t, j]) * h0[0, j].T @ q[0, t, 0]
            np.testing.assert_allclose(o[0, t, j], ref, atol=1e-13)
        np.testing.assert_allclose(ht[0, j], np.exp(gam[-1, j]) * h0[0, j], atol=1e-13)


@pytest.mark.parametrize("gated", [True, False])
def test_no_erase_equals_quadratic_linear_attention(gated):
    """Without the erase term the layer is gated causal linear attention; its quadratic
    form is an independent formulation.  With g = 0 it is plain causal linear attention."""
    q, k, v, g, beta, h0 = rnd(3, T=15, Hqk=2, Hv=4, unit_k=False)
    if not gated:
        g[:] = 0.0
    o, ht = orc.fwd(q, k, v, g, beta, 0.3, h0=h0, flags=orc.NO_ERASE)
    gam = np.cumsum(g[0], axis=0)
    T = 15
    for j in range(4):
        qh = j // 2
        for t in range(T):
            acc = np.exp(gam[t, j]) * h0[0, j].T @ q[0, t, qh]
            for s in range(t + 1):
                acc = acc + np.exp(gam[t, j] - gam[s, j]) * beta[0, s, j] * v[0, s, j] * (k[0, s, qh] @ q[0, t, qh])
            np.testing.assert_allclose(o[0, t, j], 0.3 * acc, rtol=1e-12, atol=1e-12)
        H = np.exp(gam[-1, j]) * h0[0, j]
        for s in range(T):
            H = H + np.exp(gam[-1, j] - gam[s, j]) * beta[0, s, j] * np.outer(k[0, s, qh], v[0, s, j])
        np.testing.assert_allclose(ht[0, j], H, rtol=1e-12, atol=1e-12)


def test_delta_rule_stores_value_exactly():
    """beta = 1 and |k| = 1: after each write the memory returns v_t for k_t, whatever the
    history, so with q = k and scale = 1 the output equals v."""
    q, k, v, g, beta, h0 = rnd(4, T=20, K=6, V=9)
    beta[:] = 1.0
    o, _ = orc.fwd(k, k, v, g, beta, 1.0, h0=h0)
    np.testing.assert_allclose(o, v, atol=1e-12)


def test_orthonormal_keys_projection():
    """g = 0, beta = 1, orthonormal keys (T <= K): h_T = (I - sum k k^T) h0 + sum k v^T."""
    r = np.random.default_rng(5)
    K, V, T = 10, 4, 6
    Qm, _ = np.linalg.qr(r.standard_normal((K, K)))
    k = Qm[:, :T].T.reshape(1, T, 1, K)
    q = r.standard_normal((1, T, 1, K))
    v = r.standard_normal((1, T, 1, V))
    g = np.zeros((1, T, 1)); beta = np.ones((1, T, 1))
    h0 = r.standard_normal((1, 1, K, V))
    _, ht = orc.fwd(q, k, v, g, beta, 1.0, h0=h0)
    kk = k[0, :, 0]
    ref = (np.eye(K) - kk.T @ kk) @ h0[0, 0] + kk.T @ v[0, :, 0]
    np.testing.assert_allclose(ht[0, 0], ref, atol=1e-12)


def test_linearity_in_values_and_initial_state():
    q, k, v, g, beta, h0 = rnd(6)
    _, _, v2, _, _, h02 = rnd(7)
    a, b = 0.7, -1.9
    o1, t1 = orc.fwd(q, k, v, g, beta, 1.0, h0=h0)
    o2, t2 = orc.fwd(q, k, v2, g, beta, 1.0, h0=h02)
    o3, t3 = orc.fwd(q, k, a * v + b * v2, g, beta, 1.0, h0=a * h0 + b * h02)
    np.testing.assert_allclose(o3, a * o1 + b * o2, atol=1e-12)
    np.testing.assert_allclose(t3, a * t1 + b * t2, atol=1e-12)


def test_contraction_bound():
    """beta in [0,1], |k| <= 1: two initial states move apart by at most exp(sum g) in the
    spectral norm (each step multiplies the difference by exp(g) (I - beta k k^T))."""
    q, k, v, g, beta, h0 = rnd(8, T=30)
    h0b = h0 + np.random.default_rng(9).standard_normal(h0.shape)
    _, ta = orc.fwd(q, k, v, g, beta, 1.0, h0=h0)
    _, tb = orc.fwd(q, k, v, g, beta, 1.0, h0=h0b)
    for j in range(2):
        lhs = np.linalg.norm(ta[0, j] - tb[0, j], 2)
        rhs = np.exp(g[0, :, j].sum()) * np.linalg.norm(h0[0, j] - h0b[0, j], 2)
        assert lhs <= rhs * (1 + 1e-9)
        assert lhs > 0


def test_gqa_blocked_head_mapping():
    """v-head j reads q/k head j // (Hv / Hqk)."""
    q, k, v, g, beta, h0 = rnd(10, Hqk=2, Hv=6)
    o, ht = orc.fwd(q, k, v, g, beta, 0.9, h0=h0)
    for j in range(6):
        sl = slice(j, j + 1)
        o1, t1 = orc.fwd(q[:, :, j // 3:j // 3 + 1], k[:, :, j // 3:j // 3 + 1], v[:, :, sl],
                         g[:, :, sl], beta[:, :, sl], 0.9, h0=h0[:, sl])
        np.testing.assert_array_equal(o[:, :, sl], o1)
        np.testing.assert_array_equal(ht[:, sl], t1)


def test_varlen_equals_separate_runs():
    lens = [5, 0, 17, 1, 9]
    T = sum(lens)
    q, k, v, g, beta, _ = rnd(11, T=T, Hqk=1, Hv=2)
    h0 = np.random.default_rng(12).standard_normal((len(lens), 2, 8, 12))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, ht = orc.fwd(q, k, v, g, beta, 0.8, h0=h0, cu_seqlens=cu)
    for s, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        o1, t1 = orc.fwd(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b], 0.8,
                         h0=h0[s:s + 1])
        np.testing.assert_array_equal(o[:, a:b], o1)
        np.testing.assert_array_equal(ht[s], t1[0])
    assert np.array_equal(ht[1], h0[1])  # empty sequence keeps its initial state


def test_batch_equals_varlen():
    q, k, v, g, beta, h0 = rnd(13, B=3, T=7)
    o, ht = orc.fwd(q, k, v, g, beta, 0.8, h0=h0)
    f = lambda x: x.reshape((1, 21) + x.shape[2:])
    o2, t2 = orc.fwd(f(q), f(k), f(v), f(g), f(beta), 0.8, h0=h0, cu_seqlens=[0, 7, 14, 21])
    np.testing.assert_array_equal(o.reshape(o2.shape), o2)
    np.testing.assert_array_equal(ht, t2)


def test_prefill_split_invariance():
    q, k, v, g, beta, h0 = rnd(14, T=40)
    o, ht = orc.fwd(q, k, v, g, beta, 0.6, h0=h0)
    s = slice(0, 23), slice(23, 40)
    oa, ta = orc.fwd(*(x[:, s[0]] for x in (q, k, v, g, beta)), 0.6, h0=h0)
    ob, tb = orc.fwd(*(x[:, s[1]] for x in (q, k, v, g, beta)), 0.6, h0=ta)
    np.testing.assert_allclose(np.concatenate([oa, ob], 1), o, atol=1e-12)
    np.testing.assert_allclose(tb, ht, atol=1e-12)


# ---------------------------------------------------------------- backward


def _loss(q, k, v, g, beta, h0, dO, dht, scale, cu, flags=0):
    o, ht = orc.fwd(q, k, v, g, beta, scale, h0=h0, cu_seqlens=cu, flags=flags)
    return float(np.sum(o * dO) + np.sum(ht * dht))


@pytest.mark.parametrize("flags", [0, orc.NO_ERASE])
def test_backward_matches_central_differences_everywhere(flags):
    """Every coordinate of every input, tiny sizes, two packed sequences and G = 2."""
    lens = [17, 9]
    T = sum(lens)
    cu = np.array([0] + list(np.cumsum(lens)))
    q, k, v, g, beta, _ = rnd(15, T=T, Hqk=1, Hv=2, K=8, V=12)
    r = np.random.default_rng(16)
    h0 = 0.3 * r.standard_normal((2, 2, 8, 12))
    dO = r.standard_normal(v.shape)
    dht = r.standard_normal(h0.shape)
    scale = 0.77
    dq, dk, dv, dg, db, dh0 = orc.bwd(q, k, v, g, beta, scale, dO, h0=h0, dht=dht,
                                     cu_seqlens=cu, flags=flags)
    args = dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0)
    grads = dict(q=dq, k=dk, v=dv, g=dg, beta=db, h0=dh0)
    eps = 1e-6
    for name, x in args.items():
        num = np.zeros_like(x)
        flat = x.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + eps
            lp = _loss(**args, dO=dO, dht=dht, scale=scale, cu=cu, flags=flags)
            flat[i] = old - eps
            lm = _loss(**args, dO=dO, dht=dht, scale=scale, cu=cu, flags=flags)
            flat[i] = old
            num.reshape(-1)[i] = (lp - lm) / (2 * eps)
        err = np.abs(num - grads[name]).max() / max(np.abs(num).max(), 1e-30)
        assert err < 1e-7, (name, err)


def test_backward_random_direction_medium():
    """Directional derivative along a random direction of all inputs at once (T = 200,
    K = 16, V = 24, G = 3)."""
    q, k, v, g, beta, h0 = rnd(17, T=200, Hqk=1, Hv=3, K=16, V=24)
    r = np.random.default_rng(18)
    dO = r.standard_normal(v.shape)
    dht = r.standard_normal(h0.shape)
    grads = orc.bwd(q, k, v, g, beta, 0.5, dO, h0=h0, dht=dht)
    xs = [q, k, v, g, beta, h0]
    dirs = [r.standard_normal(x.shape) for x in xs]
    eps = 1e-6
    plus = [x + eps * d for x, d in zip(xs, dirs)]
    minus = [x - eps * d for x, d in zip(xs, dirs)]
    lp = _loss(*plus, dO, dht, 0.5, None)
    lm = _loss(*minus, dO, dht, 0.5, None)
    num = (lp - lm) / (2 * eps)
    ana = sum(float(np.sum(gr * d)) for gr, d in zip(grads, dirs))
    assert abs(num - ana) <= 1e-7 * max(abs(ana), 1.0)
