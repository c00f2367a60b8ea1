"""Chunk-form restatement of the gated delta rule in fp64 numpy: the algebra the CUDA
kernels follow, checked here against the per-token oracle before any kernel uses it.

TEST INFRASTRUCTURE ONLY (tests and nothing else import it).  It shares no code with the
kernels.

Everything is written per (sequence, v-head) over chunks of C tokens (FlashQLA pages, "GDN
chunked prefill optimisation": the chunked prefill keeps per-chunk intermediates W, U and
the state S).  For one chunk of c <= C rows, with gamma the in-chunk inclusive cumsum of g,
e = exp(gamma), eC = e[c-1], D_ij = exp(gamma_i - gamma_j) for i >= j (0 above), Dm its
strictly-lower part and h the state entering the chunk (h = S^T, K x V):

    A  = diag(beta) (K K^T * Dm)            T = (I + A)^-1   (unit lower triangular)
    W  = T diag(beta e) K                   U = T diag(beta) V
    V' = U - W h                            (the corrected values, "V'")
    O  = scale (diag(e) Q h + (Q K^T * D) V')
    h' = eC h + Khat^T V',   Khat = diag(eC / e) K

Context parallelism over chunk ranges (FlashQLA pages, "AutoCP" and "warm-up"): the chunk
map h -> h' is affine, h' = (eC I - Khat^T W) h + Khat^T U, so a segment of chunks maps
its entering state by h_out = M h_in + S.  The exact mode computes (M_j, S_j) per segment,
composes them serially (the fix-up) and reruns each segment from its true entering state.
The warm-up mode instead starts segment j's scan w chunks early from a zero state.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def _cu(cu_seqlens, B, T):
    if cu_seqlens is None:
        return np.arange(B + 1, dtype=np.int64) * T
    return np.asarray(cu_seqlens, dtype=np.int64)


class _Chunk:
    """Per-chunk intermediates of one (sequence, v-head) chunk."""

    def __init__(self, Kc, Qc, Vc, gc, bc):
        c = len(gc)
        self.K, self.Q, self.V, self.beta = Kc, Qc, Vc, bc
        self.gam = np.cumsum(gc)
        self.e = np.exp(self.gam)
        self.eC = self.e[-1]
        diff = self.gam[:, None] - self.gam[None, :]
        lower = np.tril(np.ones((c, c), dtype=bool))
        self.D = np.where(lower, np.exp(np.where(lower, diff, 0.0)), 0.0)
        self.Dm = np.tril(self.D, -1)
        self.Bm = Kc @ Kc.T
        self.A = bc[:, None] * self.Bm * self.Dm
        self.T = solve_triangular(np.eye(c) + self.A, np.eye(c), lower=True,
                                  unit_diagonal=True)
        self.YW = (bc * self.e)[:, None] * Kc
        self.YU = bc[:, None] * Vc
        self.W = self.T @ self.YW
        self.U = self.T @ self.YU
        self.P = (Qc @ Kc.T) * self.D
        self.kd = np.exp(self.gam[-1] - self.gam)  # eC / e
        self.Khat = self.kd[:, None] * Kc

    def vprime(self, h):
        return self.U - self.W @ h

    def out(self, h, vp, scale):
        return scale * (self.e[:, None] * (self.Q @ h) + self.P @ vp)

    def next_state(self, h, vp):
        return self.eC * h + self.Khat.T @ vp

    def transition(self, X):
        """Linear part of the chunk map applied to X: eC X - Khat^T (W X)."""
        return self.eC * X - self.Khat.T @ (self.W @ X)


def _chunks_of(q, k, v, g, beta, t0, t1, qh, j, C):
    for c0 in range(t0, t1, C):
        c1 = min(c0 + C, t1)
        yield c0, c1, _Chunk(k[c0:c1, qh], q[c0:c1, qh], v[c0:c1, j], g[c0:c1, j],
                             beta[c0:c1, j])


def _packed(q, k, v, g, beta, dO=None):
    B, T = q.shape[:2]
    f = lambda x: None if x is None else np.asarray(x, np.float64).reshape((B * T,) + x.shape[2:])
    return B, T, f(q), f(k), f(v), f(g), f(beta), f(dO)


def fwd(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, chunk=64):
    """Chunked forward.  Shapes as the oracle: q/k [B,T,Hqk,K], v [B,T,Hv,V], g/beta
    [B,T,Hv].  Returns (o, ht)."""
    B, T, q, k, v, g, beta, _ = _packed(q, k, v, g, beta)
    Hqk, K = q.shape[1:]
    Hv, V = v.shape[1:]
    G = Hv // Hqk
    cu = _cu(cu_seqlens, B, T)
    N = len(cu) - 1
    o = np.zeros((B * T, Hv, V))
    ht = np.zeros((N, Hv, K, V))
    for s in range(N):
        for j in range(Hv):
            h = np.zeros((K, V)) if h0 is None else np.array(h0[s, j], np.float64)
            for c0, c1, ch in _chunks_of(q, k, v, g, beta, cu[s], cu[s + 1], j // G, j, chunk):
                vp = ch.vprime(h)
                o[c0:c1, j] = ch.out(h, vp, scale)
                h = ch.next_state(h, vp)
            ht[s, j] = h
    return o.reshape(B, T, Hv, V), ht


def fwd_lowlevel(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, chunk=64):
    """Chunked forward that also returns the low-level intermediates of the pages' low-level
    forward (FlashQLA pages, aisparkup "usage" section: g, A, o, h, final state), read as

        gam [TT, Hv]        gamma, the in-chunk inclusive cumsum of g
        A   [TT, Hv, chunk] each token's row of its chunk's T = (I + A)^-1, zero past the
                            token's own column (and for the missing rows of a short chunk)
        h   [NC, Hv, K, V]  the state entering every chunk, chunks of all sequences in order

    with TT = B*T packed tokens.  Returns (gam, A, o, h, ht); o is [B, T, Hv, V]."""
    B, T, q, k, v, g, beta, _ = _packed(q, k, v, g, beta)
    Hqk, K = q.shape[1:]
    Hv, V = v.shape[1:]
    G = Hv // Hqk
    cu = _cu(cu_seqlens, B, T)
    N = len(cu) - 1
    nchunks = [-(-int(cu[s + 1] - cu[s]) // chunk) for s in range(N)]
    first = np.concatenate([[0], np.cumsum(nchunks)]).astype(np.int64)
    o = np.zeros((B * T, Hv, V))
    ht = np.zeros((N, Hv, K, V))
    gam = np.zeros((B * T, Hv))
    A = np.zeros((B * T, Hv, chunk))
    hs = np.zeros((int(first[-1]), Hv, K, V))
    for s in range(N):
        for j in range(Hv):
            h = np.zeros((K, V)) if h0 is None else np.array(h0[s, j], np.float64)
            for n, (c0, c1, ch) in enumerate(_chunks_of(q, k, v, g, beta, cu[s], cu[s + 1],
                                                        j // G, j, chunk)):
                hs[first[s] + n, j] = h
                gam[c0:c1, j] = ch.gam
                A[c0:c1, j, :c1 - c0] = ch.T
                vp = ch.vprime(h)
                o[c0:c1, j] = ch.out(h, vp, scale)
                h = ch.next_state(h, vp)
            ht[s, j] = h
    return gam, A.reshape(B * T, Hv, chunk), o.reshape(B, T, Hv, V), hs, ht


def fwd_cp(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, chunk=64, seg_chunks=4,
           warmup=None):
    """Chunked forward with context parallelism over chunk ranges of ``seg_chunks`` chunks.

    warmup=None: exact mode (segment transitions (M_j, S_j), serial fix-up, rerun).
    warmup=w:    each segment j > 0 starts w chunks early from a zero state (or from h0 when
                 the window reaches the sequence start) and discards the warm-up outputs.
    """
    B, T, q, k, v, g, beta, _ = _packed(q, k, v, g, beta)
    Hqk, K = q.shape[1:]
    Hv, V = v.shape[1:]
    G = Hv // Hqk
    cu = _cu(cu_seqlens, B, T)
    N = len(cu) - 1
    o = np.zeros((B * T, Hv, V))
    ht = np.zeros((N, Hv, K, V))
    for s in range(N):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        nch = -(-(t1 - t0) // chunk)
        segs = [(a, min(a + seg_chunks, nch)) for a in range(0, nch, seg_chunks)]
        for j in range(Hv):
            qh = j // G
            hs = np.zeros((K, V)) if h0 is None else np.array(h0[s, j], np.float64)
            chunks = list(_chunks_of(q, k, v, g, beta, t0, t1, qh, j, chunk))
            if warmup is None:
                # phase A: segment transitions; fix-up: serial composition
                h_in = [hs]
                for a, b in segs[:-1]:
                    Sj = np.zeros((K, V)) if a > 0 else hs.copy()
                    Mj = np.eye(K)
                    for _, _, ch in chunks[a:b]:
                        Sj = ch.next_state(Sj, ch.vprime(Sj))
                        Mj = ch.transition(Mj)
                    h_in.append(Sj if a == 0 else Mj @ h_in[-1] + Sj)
            else:
                h_in = [hs]
                for a, _ in segs[1:]:
                    w0 = a - warmup
                    h = hs.copy() if w0 <= 0 else np.zeros((K, V))
                    for _, _, ch in chunks[max(w0, 0):a]:
                        h = ch.next_state(h, ch.vprime(h))
                    h_in.append(h)
            # phase C: every segment from its entering state
            for (a, b), h in zip(segs, h_in):
                for c0, c1, ch in chunks[a:b]:
                    vp = ch.vprime(h)
                    o[c0:c1, j] = ch.out(h, vp, scale)
                    h = ch.next_state(h, vp)
                if b == nch:
                    ht[s, j] = h
            if nch == 0:
                ht[s, j] = hs
    return o.reshape(B, T, Hv, V), ht


def bwd(q, k, v, g, beta, scale, dO, h0=None, dht=None, cu_seqlens=None, chunk=64):
    """Chunk-form reverse mode.  Returns dq, dk, dv, dg, dbeta, dh0.

    For each chunk, going backwards, with dh the gradient w.r.t. the state leaving the
    chunk and dOs = scale dO:
        dV'  = P^T dOs + Khat dh                 dP   = (dOs V'^T) on i >= j
        dQ   = diag(e) dOs h^T + (dP * D) K      dK   = (dP * D)^T Q + diag(eC/e) (V' dh^T)
        dW   = -dV' h^T   dU = dV'               dT   = dW YW^T + dU YU^T
        dYW  = T^T dW     dYU = T^T dU           dA   = strictly-lower(-T^T dT T^T)
        dK  += (dB + dB^T) K + diag(beta e) dYW,  dB = diag(beta) (dA * Dm)
        dV   = diag(beta) dYU
        dbeta_i = sum_j dA_ij (Bm * Dm)_ij + e_i <dYW_i, K_i> + <dYU_i, V_i>
        dgamma  = rowsum - colsum of (dP * P) and of (dA * A)
                  + e_i <dOs_i, (Q h)_i> + beta_i e_i <dYW_i, K_i> - r_i,
                  r_i = <(V' dh^T)_i, Khat_i>;  dgamma_{c-1} += sum_i r_i + eC <dh, h>
        dg_t = sum_{i >= t} dgamma_i             (reverse in-chunk cumsum)
        dh_in = eC dh + Q^T diag(e) dOs - W^T dV'
    """
    B, T, q, k, v, g, beta, dO = _packed(q, k, v, g, beta, dO)
    Hqk, K = q.shape[1:]
    Hv, V = v.shape[1:]
    G = Hv // Hqk
    cu = _cu(cu_seqlens, B, T)
    N = len(cu) - 1
    TT = B * T
    dqp = np.zeros((TT, Hv, K))
    dkp = np.zeros((TT, Hv, K))
    dv = np.zeros((TT, Hv, V))
    dg = np.zeros((TT, Hv))
    db = np.zeros((TT, Hv))
    dh0 = np.zeros((N, Hv, K, V))
    for s in range(N):
        for j in range(Hv):
            qh = j // G
            h = np.zeros((K, V)) if h0 is None else np.array(h0[s, j], np.float64)
            chunks = []
            for c0, c1, ch in _chunks_of(q, k, v, g, beta, cu[s], cu[s + 1], qh, j, chunk):
                chunks.append((c0, c1, ch, h))
                h = ch.next_state(h, ch.vprime(h))
            dh = np.zeros((K, V)) if dht is None else np.array(dht[s, j], np.float64)
            for c0, c1, ch, h in reversed(chunks):
                dOs = scale * dO[c0:c1, j]
                vp = ch.vprime(h)
                c = c1 - c0
                lower = np.tril(np.ones((c, c)))
                dVp = ch.P.T @ dOs + ch.Khat @ dh
                dP = (dOs @ vp.T) * lower
                dQk = dP * ch.D
                dQ = ch.e[:, None] * (dOs @ h.T) + dQk @ ch.K
                dKhat = vp @ dh.T
                dK = dQk.T @ ch.Q + ch.kd[:, None] * dKhat
                dW = -dVp @ h.T
                dU = dVp
                dT = dW @ ch.YW.T + dU @ ch.YU.T
                dYW = ch.T.T @ dW
                dYU = ch.T.T @ dU
                dA = np.tril(-ch.T.T @ dT @ ch.T.T, -1)
                dBm = ch.beta[:, None] * dA * ch.Dm
                dK += (dBm + dBm.T) @ ch.K + (ch.beta * ch.e)[:, None] * dYW
                dV = ch.beta[:, None] * dYU
                tW = np.sum(dYW * ch.K, axis=1)
                dbeta = np.sum(dA * ch.Bm * ch.Dm, axis=1) + ch.e * tW + np.sum(dYU * ch.V, axis=1)
                PP = dP * ch.P
                AA = dA * ch.A
                r = np.sum(dKhat * ch.Khat, axis=1)
                dgam = (PP.sum(1) - PP.sum(0) + AA.sum(1) - AA.sum(0)
                        + ch.e * np.sum(dOs * (ch.Q @ h), axis=1) + ch.beta * ch.e * tW - r)
                dgam[-1] += r.sum() + ch.eC * np.sum(dh * h)
                dg[c0:c1, j] = np.cumsum(dgam[::-1])[::-1]
                db[c0:c1, j] = dbeta
                dqp[c0:c1, j] = dQ
                dkp[c0:c1, j] = dK
                dv[c0:c1, j] = dV
                dh = ch.eC * dh + ch.Q.T @ (ch.e[:, None] * dOs) - ch.W.T @ dVp
            dh0[s, j] = dh
    dq = dqp.reshape(TT, Hqk, G, K).sum(2)
    dk = dkp.reshape(TT, Hqk, G, K).sum(2)
    return (dq.reshape(B, T, Hqk, K), dk.reshape(B, T, Hqk, K), dv.reshape(B, T, Hv, V),
            dg.reshape(B, T, Hv), db.reshape(B, T, Hv), dh0)
