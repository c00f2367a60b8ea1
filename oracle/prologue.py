"""fp64 numpy oracle of the fused prologue and its reverse mode.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg of the
benchmark may import this module; the product path never does.  It shares no code with the
kernels.

The FlashQLA pages take q, k, g and beta as the method's inputs (agentlenshq "GDN chunked
prefill optimisation": g a log-decay, beta a write strength, q and k the unit keys of the
delta rule) and say nothing of how a layer forms them.  The reading implemented here:

    q = q_raw / sqrt(|q_raw|^2 + eps)      k likewise        (over the last axis, eps = 1e-6)
    g = -exp(A_log[j]) * softplus(a + dt_bias[j])           softplus(x) = log(1 + e^x)
    beta = 1 / (1 + exp(-b))

Shapes: q_raw, k_raw [..., K]; a, b [..., Hv]; A_log, dt_bias [Hv].
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def softplus(x):
    return np.logaddexp(0.0, x)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def l2norm(x, eps=EPS):
    x = _f64(x)
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps)


def fwd(q_raw, k_raw, a, b, A_log, dt_bias, eps=EPS):
    """Returns (q, k, g, beta) in fp64."""
    a, b, A_log, dt_bias = (_f64(x) for x in (a, b, A_log, dt_bias))
    g = -np.exp(A_log) * softplus(a + dt_bias)
    return l2norm(q_raw, eps), l2norm(k_raw, eps), g, sigmoid(b)


def bwd(q_raw, k_raw, a, b, A_log, dt_bias, dq, dk, dg, dbeta, eps=EPS):
    """Reverse mode of :func:`fwd` for the loss <q, dq> + <k, dk> + <g, dg> + <beta, dbeta>.

    For y = x / n with n = sqrt(|x|^2 + eps): dy/dx = (I - y y^T) / n, so
    dx = (dy - y <y, dy>) / n.  d softplus(u)/du = sigmoid(u), d sigmoid(b)/db =
    sigmoid(b)(1 - sigmoid(b)), dg/dA_log = g.  A_log and dt_bias are shared by every
    token, so their gradients sum over all leading axes.
    Returns (dq_raw, dk_raw, da, db, dA_log, ddt_bias)."""
    a, b, A_log, dt_bias, dg, dbeta = (_f64(x) for x in (a, b, A_log, dt_bias, dg, dbeta))

    def norm_bwd(x, dy):
        x, dy = _f64(x), _f64(dy)
        n = np.sqrt((x * x).sum(-1, keepdims=True) + eps)
        y = x / n
        return (dy - y * (y * dy).sum(-1, keepdims=True)) / n

    u = a + dt_bias
    g = -np.exp(A_log) * softplus(u)
    da = dg * (-np.exp(A_log)) * sigmoid(u)
    bt = sigmoid(b)
    lead = tuple(range(a.ndim - 1))
    return (norm_bwd(q_raw, dq), norm_bwd(k_raw, dk), da, dbeta * bt * (1.0 - bt),
            (dg * g).sum(axis=lead), da.sum(axis=lead))
