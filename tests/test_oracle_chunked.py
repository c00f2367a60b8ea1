"""The chunk-form algebra the kernels follow (oracle/chunked.py), pinned against the per-token
oracle: chunked forward for several chunk sizes, context parallelism over chunk ranges (exact
fix-up and warm-up), and the chunk-form backward."""
import numpy as np
import pytest

from oracle import chunked, oracle as orc


def rnd(seed, T, Hqk, Hv, K=8, V=12, nseq=1, h0=True):
    r = np.random.default_rng(seed)
    nrm = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    q = nrm(r.standard_normal((1, T, Hqk, K)))
    k = nrm(r.standard_normal((1, T, Hqk, K)))
    v = r.standard_normal((1, T, Hv, V))
    g = -np.log1p(np.exp(r.standard_normal((1, T, Hv))))
    beta = 1 / (1 + np.exp(-r.standard_normal((1, T, Hv))))
    h0a = 0.3 * r.standard_normal((nseq, Hv, K, V)) if h0 else None
    return q, k, v, g, beta, h0a


@pytest.mark.parametrize("chunk", [1, 3, 16, 64, 70])
@pytest.mark.parametrize("G", [1, 2, 3])
def test_chunked_equals_recurrent(chunk, G):
    T = 70
    q, k, v, g, beta, h0 = rnd(100 + chunk + G, T, 1, G)
    o, ht = orc.fwd(q, k, v, g, beta, 0.6, h0=h0)
    oc, htc = chunked.fwd(q, k, v, g, beta, 0.6, h0=h0, chunk=chunk)
    np.testing.assert_allclose(oc, o, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(htc, ht, rtol=1e-11, atol=1e-11)


def test_chunked_varlen_with_partial_and_empty_sequences():
    lens = [37, 0, 5, 64, 129]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, g, beta, h0 = rnd(7, T, 2, 4, nseq=len(lens))
    o, ht = orc.fwd(q, k, v, g, beta, 0.6, h0=h0, cu_seqlens=cu)
    oc, htc = chunked.fwd(q, k, v, g, beta, 0.6, h0=h0, cu_seqlens=cu, chunk=16)
    np.testing.assert_allclose(oc, o, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(htc, ht, rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("seg", [1, 2, 3, 7])
def test_context_parallel_exact_equals_serial(seg):
    lens = [150, 33, 0, 96]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, g, beta, h0 = rnd(30 + seg, T, 1, 2, nseq=len(lens))
    o, ht = orc.fwd(q, k, v, g, beta, 0.6, h0=h0, cu_seqlens=cu)
    oc, htc = chunked.fwd_cp(q, k, v, g, beta, 0.6, h0=h0, cu_seqlens=cu, chunk=8,
                             seg_chunks=seg)
    np.testing.assert_allclose(oc, o, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(htc, ht, rtol=1e-10, atol=1e-10)


def test_context_parallel_warmup_error_within_contraction_bound():
    """Warm-up starts segment j's scan w chunks early from zero.  Its entering-state error
    is the true state at the window start carried through the window, so it is at most
    exp(sum of g over the window) times that state's spectral norm."""
    T, C, seg, w = 256, 8, 8, 2
    q, k, v, g, beta, h0 = rnd(41, T, 1, 1)
    g *= 0.05  # mild decay, so the warm-up error is far above rounding
    o, ht = orc.fwd(q, k, v, g, beta, 1.0, h0=h0)
    ow, htw = chunked.fwd_cp(q, k, v, g, beta, 1.0, h0=h0, chunk=C, seg_chunks=seg, warmup=w)
    # the first segment is exact
    np.testing.assert_allclose(ow[:, :seg * C], o[:, :seg * C], atol=1e-11)
    # bound the final-state error through the last segment's warm-up window
    start = (T // C // seg - 1) * seg * C
    w0 = start - w * C
    _, h_at_w0 = orc.fwd(q[:, :w0], k[:, :w0], v[:, :w0], g[:, :w0], beta[:, :w0], 1.0, h0=h0)
    bound = np.exp(g[0, w0:, 0].sum()) * np.linalg.norm(h_at_w0[0, 0], 2)
    err = np.linalg.norm(htw[0, 0] - ht[0, 0], 2)
    assert 1e-8 < err <= bound * (1 + 1e-9)
    # and warm-up with a window that reaches the sequence start is exact
    oe, hte = chunked.fwd_cp(q, k, v, g, beta, 1.0, h0=h0, chunk=C, seg_chunks=seg,
                             warmup=T // C)
    np.testing.assert_allclose(oe, o, atol=1e-10)


@pytest.mark.parametrize("chunk", [1, 5, 16])
def test_chunked_backward_equals_recurrent_backward(chunk):
    lens = [23, 0, 40, 9]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, g, beta, h0 = rnd(50 + chunk, T, 2, 4, nseq=len(lens))
    r = np.random.default_rng(51)
    dO = r.standard_normal(v.shape)
    dht = r.standard_normal(h0.shape)
    ref = orc.bwd(q, k, v, g, beta, 0.7, dO, h0=h0, dht=dht, cu_seqlens=cu)
    got = chunked.bwd(q, k, v, g, beta, 0.7, dO, h0=h0, dht=dht, cu_seqlens=cu, chunk=chunk)
    for name, a, b in zip(["dq", "dk", "dv", "dg", "dbeta", "dh0"], got, ref):
        np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-9, err_msg=name)


# ---- the low-level forward's intermediates (gamma, T per token, state entering every chunk)

def test_lowlevel_states_are_prefix_recurrences():
    """h of chunk n of a sequence is the per-token recurrence's final state after the
    sequence's first n*chunk tokens (h0 for n = 0); o and ht are the recurrence's."""
    lens = [37, 0, 5, 64, 129]
    C = 16
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, g, beta, h0 = rnd(8, sum(lens), 2, 4, nseq=len(lens))
    gam, A, o, hs, ht = chunked.fwd_lowlevel(q, k, v, g, beta, 0.6, h0=h0, cu_seqlens=cu, chunk=C)
    ro, rht = orc.fwd(q, k, v, g, beta, 0.6, h0=h0, cu_seqlens=cu)
    np.testing.assert_allclose(o, ro, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(ht, rht, rtol=1e-11, atol=1e-11)
    n_all = 0
    for s, L in enumerate(lens):
        for n in range(-(-L // C)):
            t0, t1 = cu[s], cu[s] + n * C
            sl = lambda x: x[:, t0:t1]
            _, pre = orc.fwd(sl(q), sl(k), sl(v), sl(g), sl(beta), 0.6, h0=h0[s:s + 1])
            np.testing.assert_allclose(hs[n_all], pre[0], rtol=1e-11, atol=1e-11)
            n_all += 1
    assert hs.shape[0] == n_all


def test_lowlevel_gamma_restarts_at_chunk_and_sequence_starts():
    lens = [3, 20, 0, 9]
    C = 8
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, _, beta, _ = rnd(9, sum(lens), 1, 2, h0=False)
    g = np.full(beta.shape, -0.1)
    gam = chunked.fwd_lowlevel(q, k, v, g, beta, 1.0, cu_seqlens=cu, chunk=C)[0]
    for s in range(len(lens)):
        for t in range(cu[s], cu[s + 1]):
            pos = (t - cu[s]) % C
            np.testing.assert_allclose(gam[t], -0.1 * (pos + 1), rtol=1e-14)


def test_lowlevel_T_closed_forms():
    """Rows of T = (I + L)^-1 with L_ij = beta_i exp(g_{j+1} + ... + g_i) <k_i, k_j> (i > j):
    for three tokens T_10 = -L_10, T_21 = -L_21, T_20 = -L_20 + L_21 L_10 (Neumann series
    of a nilpotent L); the diagonal is 1 and everything past it 0."""
    q, k, v, g, beta, _ = rnd(10, 3, 1, 1, h0=False)
    A = chunked.fwd_lowlevel(q, k, v, g, beta, 1.0, chunk=64)[1][:, 0]
    kk = lambda i, j: float(np.dot(k[0, i, 0], k[0, j, 0]))
    Lm = lambda i, j: beta[0, i, 0] * np.exp(g[0, j + 1:i + 1, 0].sum()) * kk(i, j)
    want = np.zeros((3, 64))
    want[0, 0] = want[1, 1] = want[2, 2] = 1.0
    want[1, 0] = -Lm(1, 0)
    want[2, 1] = -Lm(2, 1)
    want[2, 0] = -Lm(2, 0) + Lm(2, 1) * Lm(1, 0)
    np.testing.assert_allclose(A, want, rtol=1e-12, atol=1e-14)


def test_lowlevel_T_inverts_the_chunk_matrix_by_loops():
    """(I + L) T = I on every chunk of a ragged sequence, L built entry by entry."""
    T_len, C = 45, 16
    q, k, v, g, beta, _ = rnd(11, T_len, 1, 2, h0=False)
    A = chunked.fwd_lowlevel(q, k, v, g, beta, 1.0, chunk=C)[1]
    for j in range(2):
        for c0 in range(0, T_len, C):
            c = min(C, T_len - c0)
            Lc = np.eye(c)
            for i in range(c):
                for jj in range(i):
                    dec = np.exp(sum(g[0, c0 + m, j] for m in range(jj + 1, i + 1)))
                    Lc[i, jj] = beta[0, c0 + i, j] * dec * np.dot(k[0, c0 + i, 0], k[0, c0 + jj, 0])
            Tc = A[c0:c0 + c, j, :c]
            np.testing.assert_allclose(Lc @ Tc, np.eye(c), atol=1e-12)
            assert np.all(A[c0:c0 + c, j, c:] == 0)


def test_transition_norm_bound_used_by_the_exact_mode():
    """The decay-bounded exact mode drops a segment's transition when the product of the
    per-token bounds exp(g_t) max(1, |1 - beta_t |k_t|^2|) falls below 2^-126.  That product
    bounds the 2-norm of the token transitions' product X -> (I - beta k k^T) exp(g) X in any
    order of factors: checked on random chains, with keys of length up to 1.8 (so that some
    factors expand) and with the factors composed in the recurrence's order."""
    rng = np.random.default_rng(7)
    for trial in range(40):
        n = int(rng.integers(1, 40))
        d = 8
        k = rng.standard_normal((n, d))
        k *= (rng.uniform(0.2, 1.8, n) / np.linalg.norm(k, axis=1))[:, None]
        beta = rng.uniform(0.0, 1.0, n)
        g = -rng.exponential(0.3, n) * (trial % 3)  # some chains without decay
        phi = np.eye(d)
        log_bound = 0.0
        for t in range(n):
            step = np.exp(g[t]) * (np.eye(d) - beta[t] * np.outer(k[t], k[t]))
            phi = step @ phi
            log_bound += g[t] + np.log(max(1.0, abs(1.0 - beta[t] * k[t] @ k[t])))
        assert np.linalg.norm(phi, 2) <= np.exp(log_bound) * (1 + 1e-12)
