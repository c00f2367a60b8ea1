"""Pins of the prologue oracle (oracle/prologue.py): closed forms of the three activations
and central finite differences of its hand-written reverse mode."""
import numpy as np

from oracle import prologue as pro


def rnd(seed, T=5, Hqk=2, Hv=4, K=6):
    r = np.random.default_rng(seed)
    return (r.standard_normal((1, T, Hqk, K)), r.standard_normal((1, T, Hqk, K)),
            r.standard_normal((1, T, Hv)), r.standard_normal((1, T, Hv)),
            0.5 * r.standard_normal(Hv), r.standard_normal(Hv))


def test_l2norm_direction_and_length():
    q_raw, k_raw, a, b, A_log, dt = rnd(1)
    q, k, _, _ = pro.fwd(q_raw, k_raw, a, b, A_log, dt)
    for x, y in ((q_raw, q), (k_raw, k)):
        s = (x * x).sum(-1)
        np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.sqrt(s / (s + 1e-6)), rtol=1e-13)
        cos = (x * y).sum(-1) / (np.linalg.norm(x, axis=-1) * np.linalg.norm(y, axis=-1))
        np.testing.assert_allclose(cos, 1.0, rtol=1e-13)
    # a zero row stays zero (eps keeps the division finite)
    z = np.zeros((1, 1, 1, 4))
    assert np.all(pro.l2norm(z) == 0)


def test_gate_closed_forms():
    A_log = np.array([0.0, np.log(2.0), -1.0])
    dt = np.array([0.0, 1.0, -2.0])
    a = -dt[None, None, :].copy()                     # a + dt_bias = 0: softplus = ln 2
    b = np.array([[[0.0, 3.0, -3.0]]])
    _, _, g, beta = pro.fwd(np.ones((1, 1, 1, 2)), np.ones((1, 1, 1, 2)), a, b, A_log, dt)
    np.testing.assert_allclose(g[0, 0], -np.exp(A_log) * np.log(2.0), rtol=1e-15)
    np.testing.assert_allclose(beta[0, 0], [0.5, 1 / (1 + np.exp(-3.0)), 1 / (1 + np.exp(3.0))],
                               rtol=1e-15)
    np.testing.assert_allclose(beta[0, 0, 1] + beta[0, 0, 2], 1.0, rtol=1e-15)
    # large pre-activations: softplus(u) -> u, so g -> -exp(A_log) u
    g2 = pro.fwd(np.ones((1, 1, 1, 2)), np.ones((1, 1, 1, 2)), np.full((1, 1, 3), 40.0),
                 b, A_log, np.zeros(3))[2]
    np.testing.assert_allclose(g2[0, 0], -np.exp(A_log) * 40.0, rtol=1e-15)


def test_reverse_mode_by_central_differences():
    q_raw, k_raw, a, b, A_log, dt = rnd(2)
    r = np.random.default_rng(3)
    dq, dk = r.standard_normal(q_raw.shape), r.standard_normal(k_raw.shape)
    dg, dbeta = r.standard_normal(a.shape), r.standard_normal(b.shape)

    def loss(qr, kr, aa, bb, al, dd):
        q, k, g, beta = pro.fwd(qr, kr, aa, bb, al, dd)
        return (q * dq).sum() + (k * dk).sum() + (g * dg).sum() + (beta * dbeta).sum()

    args = [q_raw, k_raw, a, b, A_log, dt]
    grads = pro.bwd(q_raw, k_raw, a, b, A_log, dt, dq, dk, dg, dbeta)
    h = 1e-6
    for i, (x, gx) in enumerate(zip(args, grads)):
        assert gx.shape == x.shape
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            ap, am = list(args), list(args)
            ap[i], am[i] = xp, xm
            fd[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        np.testing.assert_allclose(gx, fd, rtol=1e-6, atol=1e-8)
