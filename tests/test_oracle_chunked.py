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
