/*
 * Gated delta rule: plain per-token recurrent oracle in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this file;
 * only the tests, the smoke check and the CPU-baseline leg of the benchmark use it.  It
 * shares no code with the CUDA kernels.
 *
 * What it computes (FlashQLA pages, "GDN chunked prefill optimisation" section: the layer
 * is a Gated Delta Network whose state S is updated token by token; the chunked kernels
 * reach the same result faster).  Per sequence and per v-head j, with the q/k head
 * qh = j / G (G = Hv / Hqk, blocked grouping) and the state h = S^T (K x V, h[k][v]):
 *
 *     h  <- exp(g_t) * h                      (gate decay first)
 *     u  <- h^T k_t                           (what the memory already returns for k_t)
 *     d  <- beta_t * (v_t - u)                (delta-rule correction)
 *     h  <- h + k_t d^T                       (rank-one write)
 *     o_t = scale * h^T q_t
 *
 * which is S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 * o_t = scale * S_t q_t, written with h = S^T.  The final state is h after the last
 * token; the initial state is h0 (zero when absent).
 *
 * Backward: hand-written reverse mode of exactly those five lines, with forward
 * checkpoints every OR_BLOCK tokens and a forward recompute inside each block.
 *
 * Layout (all host fp64, tokens packed by cu_seqlens; B sequences of length T are the
 * special case cu = {0, T, 2T, ...}):
 *     q, k     [TT, Hqk, K]        v, o, dO   [TT, Hv, V]
 *     g, beta  [TT, Hv]            h0, ht     [N, Hv, K, V]   (h[k][v])
 *
 * flags bit 0 (OR_NO_ERASE) drops the erase term (u = 0): a test hook that turns the
 * layer into plain gated linear attention with write strength beta, so the result can be
 * pinned against the quadratic attention form.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_NO_ERASE 1
#define OR_BLOCK 64

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int check_args(int N, const int64_t* cu, int Hqk, int Hv, int K, int V) {
    if (N < 0 || !cu || Hqk <= 0 || Hv <= 0 || K <= 0 || V <= 0) return 1;
    if (Hv % Hqk != 0) return 1;
    if (cu[0] != 0) return 1;
    for (int s = 0; s < N; ++s)
        if (cu[s + 1] < cu[s]) return 1;
    return 0;
}

/* One token of the forward recurrence on state h (K x V), in place.
 * Writes u (V) and d (V) for the caller; returns nothing else. */
static void token_step(double* h, int K, int V, const double* kt, const double* vt,
                       double gt, double bt, int flags, double* u, double* d) {
    const double a = exp(gt);
    for (int i = 0; i < K * V; ++i) h[i] *= a;
    for (int c = 0; c < V; ++c) u[c] = 0.0;
    if (!(flags & OR_NO_ERASE)) {
        for (int r = 0; r < K; ++r) {
            const double kr = kt[r];
            const double* hr = h + (size_t)r * V;
            for (int c = 0; c < V; ++c) u[c] += hr[c] * kr;
        }
    }
    for (int c = 0; c < V; ++c) d[c] = bt * (vt[c] - u[c]);
    for (int r = 0; r < K; ++r) {
        const double kr = kt[r];
        double* hr = h + (size_t)r * V;
        for (int c = 0; c < V; ++c) hr[c] += kr * d[c];
    }
}

int oracle_fwd(int N, const int64_t* cu, int Hqk, int Hv, int K, int V,
               const double* q, const double* k, const double* v, const double* g,
               const double* beta, double scale, const double* h0, double* o, double* ht,
               int flags, int nthreads) {
    if (check_args(N, cu, Hqk, Hv, K, V)) return 1;
    const int G = Hv / Hqk;
    const int units = N * Hv;
    int err = 0;
    if (nthreads <= 0) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : err)
    for (int unit = 0; unit < units; ++unit) {
        const int s = unit / Hv, j = unit % Hv, qh = j / G;
        double* h = (double*)malloc(sizeof(double) * ((size_t)K * V + 2 * (size_t)V));
        if (!h) { err |= 1; continue; }
        double* u = h + (size_t)K * V;
        double* d = u + V;
        if (h0) memcpy(h, h0 + ((size_t)s * Hv + j) * K * V, sizeof(double) * K * V);
        else memset(h, 0, sizeof(double) * K * V);
        for (int64_t t = cu[s]; t < cu[s + 1]; ++t) {
            const double* kt = k + ((size_t)t * Hqk + qh) * K;
            const double* qt = q + ((size_t)t * Hqk + qh) * K;
            const double* vt = v + ((size_t)t * Hv + j) * V;
            token_step(h, K, V, kt, vt, g[t * Hv + j], beta[t * Hv + j], flags, u, d);
            double* ot = o + ((size_t)t * Hv + j) * V;
            for (int c = 0; c < V; ++c) ot[c] = 0.0;
            for (int r = 0; r < K; ++r) {
                const double qr = qt[r];
                const double* hr = h + (size_t)r * V;
                for (int c = 0; c < V; ++c) ot[c] += hr[c] * qr;
            }
            for (int c = 0; c < V; ++c) ot[c] *= scale;
        }
        if (ht) memcpy(ht + ((size_t)s * Hv + j) * K * V, h, sizeof(double) * K * V);
        free(h);
    }
    return err;
}

/*
 * Reverse mode of oracle_fwd.  dO [TT, Hv, V]; dht [N, Hv, K, V] or NULL (zero).
 * Outputs dq, dk [TT, Hqk, K] (summed over the G v-heads of each q/k head in ascending
 * head order), dv [TT, Hv, V], dg, dbeta [TT, Hv], dh0 [N, Hv, K, V] (may be NULL).
 *
 * Per token t, going backwards, with hb = exp(g_t) h_{t-1} and u, d, h_t from the forward
 * lines above, and dh the gradient with respect to h_t:
 *     dh   += scale q_t dO_t^T          dq_t  = scale h_t dO_t
 *     dk_t  = dh d                      dd    = dh^T k_t
 *     dbeta = dd . (v_t - u)            dv_t  = beta dd        du = -beta dd
 *     dhb   = dh + k_t du^T             dk_t += hb du
 *     dg_t  = <dhb, hb>                 dh    = exp(g_t) dhb    (gradient w.r.t. h_{t-1})
 */
int oracle_bwd(int N, const int64_t* cu, int Hqk, int Hv, int K, int V,
               const double* q, const double* k, const double* v, const double* g,
               const double* beta, double scale, const double* h0, const double* dO,
               const double* dht, double* dq, double* dk, double* dv, double* dg,
               double* dbeta, double* dh0, int flags, int nthreads) {
    if (check_args(N, cu, Hqk, Hv, K, V)) return 1;
    const int G = Hv / Hqk;
    const int64_t TT = cu[N];
    const int units = N * Hv;
    const size_t KV = (size_t)K * V;
    /* per-v-head partial dq, dk, reduced over the group afterwards in a fixed order */
    double* dqp = (double*)calloc((size_t)TT * Hv * K + 1, sizeof(double));
    double* dkp = (double*)calloc((size_t)TT * Hv * K + 1, sizeof(double));
    if (!dqp || !dkp) { free(dqp); free(dkp); return 2; }
    int err = 0;
    if (nthreads <= 0) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : err)
    for (int unit = 0; unit < units; ++unit) {
        const int s = unit / Hv, j = unit % Hv, qh = j / G;
        const int64_t t0 = cu[s], t1 = cu[s + 1], L = t1 - t0;
        const int64_t nblk = (L + OR_BLOCK - 1) / OR_BLOCK;
        /* ckpt[b] = state before the first token of block b; blk[i] = state before token i of a block */
        double* ckpt = (double*)malloc(sizeof(double) * KV * (size_t)(nblk > 0 ? nblk : 1));
        double* blk = (double*)malloc(sizeof(double) * KV * OR_BLOCK);
        double* work = (double*)malloc(sizeof(double) * (3 * KV + 8 * (size_t)V + 2 * (size_t)K));
        if (!ckpt || !blk || !work) { free(ckpt); free(blk); free(work); err |= 2; continue; }
        double* h = work;
        double* dh = h + KV;
        double* hb = dh + KV;
        double* u = hb + KV;
        double* d = u + V;
        double* dd = d + V;
        double* du = dd + V;
        double* dkt = du + V;   /* K */
        double* dqt = dkt + K;  /* K */

        if (h0) memcpy(h, h0 + ((size_t)s * Hv + j) * KV, sizeof(double) * KV);
        else memset(h, 0, sizeof(double) * KV);
        for (int64_t b = 0; b < nblk; ++b) {
            memcpy(ckpt + (size_t)b * KV, h, sizeof(double) * KV);
            const int64_t e = (b + 1) * OR_BLOCK < L ? (b + 1) * OR_BLOCK : L;
            for (int64_t i = b * OR_BLOCK; i < e; ++i) {
                const int64_t t = t0 + i;
                token_step(h, K, V, k + ((size_t)t * Hqk + qh) * K, v + ((size_t)t * Hv + j) * V,
                           g[t * Hv + j], beta[t * Hv + j], flags, u, d);
            }
        }
        if (dht) memcpy(dh, dht + ((size_t)s * Hv + j) * KV, sizeof(double) * KV);
        else memset(dh, 0, sizeof(double) * KV);

        for (int64_t b = nblk - 1; b >= 0; --b) {
            const int64_t ib = b * OR_BLOCK;
            const int64_t e = (b + 1) * OR_BLOCK < L ? (b + 1) * OR_BLOCK : L;
            memcpy(h, ckpt + (size_t)b * KV, sizeof(double) * KV);
            for (int64_t i = ib; i < e; ++i) {
                const int64_t t = t0 + i;
                memcpy(blk + (size_t)(i - ib) * KV, h, sizeof(double) * KV);
                token_step(h, K, V, k + ((size_t)t * Hqk + qh) * K, v + ((size_t)t * Hv + j) * V,
                           g[t * Hv + j], beta[t * Hv + j], flags, u, d);
            }
            for (int64_t i = e - 1; i >= ib; --i) {
                const int64_t t = t0 + i;
                const double* kt = k + ((size_t)t * Hqk + qh) * K;
                const double* qt = q + ((size_t)t * Hqk + qh) * K;
                const double* vt = v + ((size_t)t * Hv + j) * V;
                const double* dot = dO + ((size_t)t * Hv + j) * V;
                const double gt = g[t * Hv + j], bt = beta[t * Hv + j];
                const double a = exp(gt);
                /* rebuild hb, u, d and h_t from h_{t-1} */
                const double* hp = blk + (size_t)(i - ib) * KV;
                for (size_t x = 0; x < KV; ++x) hb[x] = a * hp[x];
                for (int c = 0; c < V; ++c) u[c] = 0.0;
                if (!(flags & OR_NO_ERASE)) {
                    for (int r = 0; r < K; ++r)
                        for (int c = 0; c < V; ++c) u[c] += hb[(size_t)r * V + c] * kt[r];
                }
                for (int c = 0; c < V; ++c) d[c] = bt * (vt[c] - u[c]);
                /* h (reused as h_t) */
                for (int r = 0; r < K; ++r)
                    for (int c = 0; c < V; ++c) h[(size_t)r * V + c] = hb[(size_t)r * V + c] + kt[r] * d[c];
                /* output line */
                for (int r = 0; r < K; ++r) {
                    double acc = 0.0;
                    for (int c = 0; c < V; ++c) {
                        dh[(size_t)r * V + c] += scale * qt[r] * dot[c];
                        acc += h[(size_t)r * V + c] * dot[c];
                    }
                    dqt[r] = scale * acc;
                }
                /* write line */
                for (int c = 0; c < V; ++c) dd[c] = 0.0;
                for (int r = 0; r < K; ++r) {
                    double acc = 0.0;
                    for (int c = 0; c < V; ++c) {
                        acc += dh[(size_t)r * V + c] * d[c];
                        dd[c] += dh[(size_t)r * V + c] * kt[r];
                    }
                    dkt[r] = acc;
                }
                double db = 0.0;
                for (int c = 0; c < V; ++c) {
                    db += dd[c] * (vt[c] - u[c]);
                    dv[((size_t)t * Hv + j) * V + c] = bt * dd[c];
                    du[c] = (flags & OR_NO_ERASE) ? 0.0 : -bt * dd[c];
                }
                dbeta[t * Hv + j] = db;
                /* read line (u = hb^T k) and decay line */
                double dgt = 0.0;
                for (int r = 0; r < K; ++r) {
                    double acc = 0.0;
                    for (int c = 0; c < V; ++c) {
                        const size_t x = (size_t)r * V + c;
                        acc += hb[x] * du[c];
                        const double dhb = dh[x] + kt[r] * du[c];
                        dgt += dhb * hb[x];
                        dh[x] = a * dhb;
                    }
                    dkt[r] += acc;
                }
                dg[t * Hv + j] = dgt;
                memcpy(dqp + ((size_t)t * Hv + j) * K, dqt, sizeof(double) * K);
                memcpy(dkp + ((size_t)t * Hv + j) * K, dkt, sizeof(double) * K);
            }
        }
        if (dh0) memcpy(dh0 + ((size_t)s * Hv + j) * KV, dh, sizeof(double) * KV);
        free(ckpt); free(blk); free(work);
    }
    if (!err) {
        for (int64_t t = 0; t < TT; ++t)
            for (int qh = 0; qh < Hqk; ++qh) {
                double* dqo = dq + ((size_t)t * Hqk + qh) * K;
                double* dko = dk + ((size_t)t * Hqk + qh) * K;
                for (int r = 0; r < K; ++r) { dqo[r] = 0.0; dko[r] = 0.0; }
                for (int jj = qh * G; jj < (qh + 1) * G; ++jj) {
                    const double* a = dqp + ((size_t)t * Hv + jj) * K;
                    const double* b = dkp + ((size_t)t * Hv + jj) * K;
                    for (int r = 0; r < K; ++r) { dqo[r] += a[r]; dko[r] += b[r]; }
                }
            }
    }
    free(dqp); free(dkp);
    return err;
}
