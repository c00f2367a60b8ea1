// C ABI of the GDN library: argument validation, the host-side planner (segment length for
// intra-GPU context parallelism), workspace layout and kernel launches.  Nothing here
// allocates, frees or synchronises.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <set>
#include <tuple>
#include <vector>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace gdn {
cudaError_t smem_attr_once(const void* kern, int bytes) {
    static std::mutex mu;
    static std::set<std::tuple<const void*, int, int>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const auto key = std::make_tuple(kern, dev, bytes);
    std::lock_guard<std::mutex> lock(mu);
    if (done.count(key)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert(key);
    return e;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    return n > 0 ? n : 148;
}
}  // namespace gdn

namespace {

thread_local char g_err[512] = "";

gdn_status fail(gdn_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

using gdn::sm_count;

// Host plan of one call.
struct HostPlan {
    int N = 0;              // sequences
    int C = 64;             // chunk size
    int L = 1;              // chunks per segment
    int warmup = 0;
    int cp = gdn::CP_NONE;
    int total_segs = 0;
    int total_chunks = 0;
    int max_nseg = 0;
    int64_t total_tokens = 0;
    int64_t prep_stride = 0;  // bytes per (chunk, v-head) preparation record
    // workspace layout (bytes)
    size_t off_err = 0, off_seg = 0, off_segoff = 0, off_chunkoff = 0, off_hin = 0,
           off_mbuf = 0, off_mbuf_t = 0, off_logb = 0, off_dec = 0, off_rerun = 0, off_prep = 0,
           off_end = 0;
    bool full_cp = false;   // every transition computed and every segment rerun
    // backward only
    size_t off_hist = 0, off_dhist = 0, off_dhb = 0, off_rrerun = 0, off_dqp = 0, off_dkp = 0;
};

constexpr size_t KVB = size_t(128) * 128 * 4;

gdn_status validate_problem(const gdn_problem* p) {
    if (!p) return fail(GDN_ERR_INVALID_ARG, "problem is NULL");
    if (p->K <= 0 || p->V <= 0) return fail(GDN_ERR_INVALID_ARG, "K and V must be positive");
    if (p->K != 128 || p->V != 128)
        return fail(GDN_ERR_UNSUPPORTED, "only K = V = 128 is implemented (got K=%d V=%d)", p->K,
                    p->V);
    if (p->Hqk <= 0 || p->Hv <= 0) return fail(GDN_ERR_INVALID_ARG, "Hqk and Hv must be positive");
    if (p->Hv % p->Hqk != 0)
        return fail(GDN_ERR_INVALID_ARG, "Hv (%d) must be a multiple of Hqk (%d)", p->Hv, p->Hqk);
    if (p->dtype != GDN_BF16 && p->dtype != GDN_FP32)
        return fail(GDN_ERR_INVALID_ARG, "dtype must be GDN_BF16 or GDN_FP32");
    if (!isfinite(p->scale) || !(p->scale > 0.f))
        return fail(GDN_ERR_INVALID_ARG, "scale must be finite and > 0 (got %g)", double(p->scale));
    if (p->T < 0 || p->B < 0) return fail(GDN_ERR_INVALID_ARG, "B and T must be >= 0");
    if (p->cp_mode < GDN_CP_AUTO || p->cp_mode > GDN_CP_EXACT_FULL)
        return fail(GDN_ERR_INVALID_ARG, "unknown cp_mode %d", p->cp_mode);
    if (p->cp_segment_chunks < 0 || p->warmup_chunks < 0 || !(p->cp_lambda >= 0.f))
        return fail(GDN_ERR_INVALID_ARG, "cp_segment_chunks, warmup_chunks, cp_lambda must be >= 0");
    if ((p->cu_seqlens == nullptr) != (p->cu_seqlens_host == nullptr))
        return fail(GDN_ERR_INVALID_ARG, "cu_seqlens and cu_seqlens_host go together");
    if (p->cu_seqlens) {
        if (p->B != 1) return fail(GDN_ERR_INVALID_ARG, "varlen needs B == 1 (got %d)", p->B);
        if (p->num_seqs < 1) return fail(GDN_ERR_INVALID_ARG, "num_seqs must be >= 1");
        if (!aligned16(p->cu_seqlens) && (reinterpret_cast<uintptr_t>(p->cu_seqlens) & 3u))
            return fail(GDN_ERR_INVALID_ARG, "cu_seqlens must be 4-byte aligned");
        const int32_t* cu = p->cu_seqlens_host;
        if (cu[0] != 0) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens[0] must be 0");
        for (int s = 0; s < p->num_seqs; ++s)
            if (cu[s + 1] < cu[s])
                return fail(GDN_ERR_INVALID_ARG, "cu_seqlens must be non-decreasing (at %d)", s);
        if (cu[p->num_seqs] != p->T)
            return fail(GDN_ERR_INVALID_ARG, "cu_seqlens[num_seqs] (%d) must equal T (%d)",
                        cu[p->num_seqs], p->T);
    }
    return GDN_OK;
}

// Estimated time of a segmentation with L chunks per segment, in units of one chunk step
// of the output stage: the waves of the two chunk-scan launches (one CTA per SM; the first
// phase runs a segment's state and transition in one CTA) times the chunks a CTA scans, plus
// the serial fix-up steps.  The step costs are measured ratios on GB300 (a first-phase chunk
// step ~1.0 of an output chunk step; a fix-up step as below).
double cp_cost(int L, const int* nts, int N, int Hv, int sms, bool exact, int warmup, bool bounded) {
    constexpr double tC = 1.0, tA = 1.0;
    if (bounded) {
        // exact mode with decay bounds, costed for decaying gates: one pass of L chunks plus
        // the ~2 chunks each segment scans into the next, and the three extra launches
        // (transitions, fix-up, correction: ~3 us each, returning at once) when segmented.
        // Each wave of a scan launch also pays its start (set-up, the first chunks' tiles in
        // flight) and its end (the last state out, the spread of its CTAs' ends): ~5 chunk
        // steps, fitted to the forward at 32768 tokens x 8 / 24 heads, where one wave of
        // 88-chunk scans ran 0.351 ms, two of 45 chunks 0.366 ms, three of 29 chunks 0.378 ms.
        constexpr double tW = 5.0;
        long segs = 0;
        int maxn = 0;
        for (int s = 0; s < N; ++s) {
            const int ns = std::max(1, (nts[s] + L - 1) / L);
            segs += ns;
            maxn = std::max(maxn, ns);
        }
        const long cw = (segs * Hv + sms - 1) / sms;
        const int Lc = std::min(L, *std::max_element(nts, nts + N));
        return maxn > 1 ? double(cw) * (Lc + 2 + tW) * tC + 4.0 : double(cw) * (Lc + tW) * tC;
    }
    long segs = 0, actas = 0;
    int maxn = 0;
    for (int s = 0; s < N; ++s) {
        const int ns = std::max(1, (nts[s] + L - 1) / L);
        segs += ns;
        maxn = std::max(maxn, ns);
        if (ns > 1) actas += ns - 1;
    }
    const long cw = (segs * Hv + sms - 1) / sms;
    const long aw = (actas * Hv + sms - 1) / sms;
    const int Lc = std::min(L, *std::max_element(nts, nts + N));
    double cost = double(cw) * Lc * tC;
    if (maxn > 1) {
        cost += double(aw) * (exact ? Lc : std::min(warmup, Lc)) * tA;
        if (exact) {
            // fix-up step: ~0.43 us fixed + ~0.53 us per column group of its CTAs, against
            // ~1.84 us per chunk step; more chains than one wave holds repeat it
            const int cg = gdn::fixup_groups(N * Hv);
            const long fw = (long(N) * Hv * (128 / (8 * cg)) + sms - 1) / sms;
            const double tF = (0.43 + 0.53 * cg) / 1.84;
            cost += double(fw) * std::max(0, maxn - 2) * tF;
        }
    }
    return cost;
}

// Segment length.  FlashQLA's AutoCP picks the chunks per CP rank as L = lambda * sqrt(N)
// (N = chunks of a sequence); an explicit cp_lambda keeps that rule.  By default the planner
// instead minimises cp_cost over L, which accounts for the wave quantisation of the launches
// on this GPU's SM count.
void plan(const gdn_problem* p, HostPlan& h, bool backward = false, int sms_override = 0) {
    h.C = gdn::fwd_chunk_size(p->dtype);
    h.N = p->cu_seqlens ? p->num_seqs : p->B;
    int nt_max = 0;
    int64_t total_chunks = 0;
    for (int s = 0; s < h.N; ++s) {
        const int len = p->cu_seqlens ? p->cu_seqlens_host[s + 1] - p->cu_seqlens_host[s] : p->T;
        const int nt = (len + h.C - 1) / h.C;
        nt_max = std::max(nt_max, nt);
        total_chunks += nt;
    }
    h.total_tokens = p->cu_seqlens ? p->T : int64_t(p->B) * p->T;
    int L = std::max(nt_max, 1);
    h.cp = gdn::CP_NONE;
    const int warm = p->warmup_chunks > 0 ? p->warmup_chunks : 8;
    int autoL = L;
    if (p->cp_mode != GDN_CP_OFF && nt_max > 1) {
        if (p->cp_lambda > 0.f) {
            autoL = std::max(1, int(ceilf(p->cp_lambda * sqrtf(float(nt_max)))));
        } else {
            std::vector<int> nts(h.N);
            for (int s = 0; s < h.N; ++s) {
                const int len = p->cu_seqlens ? p->cu_seqlens_host[s + 1] - p->cu_seqlens_host[s] : p->T;
                nts[s] = (len + h.C - 1) / h.C;
            }
            const int sms = sms_override > 0 ? sms_override : sm_count();
            const bool exact = p->cp_mode != GDN_CP_WARMUP;
            const bool bounded_cost = exact && p->cp_mode != GDN_CP_EXACT_FULL && p->dtype == GDN_BF16;
            double best = 1e300;
            for (int cand = nt_max; cand >= 1; --cand) {  // ties go to longer segments
                const double c = cp_cost(cand, nts.data(), h.N, p->Hv, sms, exact, warm, bounded_cost);
                if (c < best - 1e-9) {
                    best = c;
                    autoL = cand;
                }
            }
        }
    }
    switch (p->cp_mode) {
        case GDN_CP_OFF:
            break;
        case GDN_CP_AUTO:
            L = autoL;
            break;
        case GDN_CP_EXACT:
        case GDN_CP_EXACT_FULL:
        case GDN_CP_WARMUP:
            L = p->cp_segment_chunks > 0 ? p->cp_segment_chunks : autoL;
            break;
    }
    L = std::max(1, std::min(L, std::max(nt_max, 1)));
    int total_segs = 0, max_nseg = 0;
    for (int s = 0; s < h.N; ++s) {
        const int len = p->cu_seqlens ? p->cu_seqlens_host[s + 1] - p->cu_seqlens_host[s] : p->T;
        const int nt = (len + h.C - 1) / h.C;
        const int ns = std::max(1, (nt + L - 1) / L);
        total_segs += ns;
        max_nseg = std::max(max_nseg, ns);
    }
    h.L = L;
    h.total_segs = total_segs;
    h.total_chunks = int(total_chunks);
    h.max_nseg = max_nseg;
    if (max_nseg > 1)
        h.cp = (p->cp_mode == GDN_CP_WARMUP && !backward) ? gdn::CP_WARMUP : gdn::CP_EXACT;
    h.warmup = p->warmup_chunks > 0 ? p->warmup_chunks : 8;
    // exact mode with decay bounds on the bf16 path; every transition and rerun otherwise
    h.full_cp = p->cp_mode == GDN_CP_EXACT_FULL || p->dtype != GDN_BF16;
    const bool bounded = h.cp == gdn::CP_EXACT && !h.full_cp;

    size_t off = 0;
    h.off_err = off;
    off = align_up(off + sizeof(int), 256);
    h.off_seg = off;
    off = align_up(off + sizeof(int2) * size_t(total_segs), 256);
    h.off_segoff = off;
    off = align_up(off + sizeof(int) * size_t(h.N + 1), 256);
    h.off_chunkoff = off;
    off = align_up(off + sizeof(int) * size_t(h.N + 1), 256);
    h.off_hin = off;
    if (h.cp != gdn::CP_NONE) off += KVB * size_t(total_segs) * p->Hv;
    h.off_mbuf = off;
    if (h.cp == gdn::CP_EXACT) off += KVB * size_t(total_segs) * p->Hv;
    h.off_mbuf_t = off;  // the backward's reverse fix-up reads the transitions untransposed
    if (h.cp == gdn::CP_EXACT && backward && p->dtype == GDN_BF16) off += KVB * size_t(total_segs) * p->Hv;
    off = align_up(off, 256);
    h.off_logb = off;  // per (chunk, v-head) transition log-bound, per (segment, v-head) decision
    if (bounded) off = align_up(off + sizeof(float) * size_t(h.total_chunks) * p->Hv, 256);
    h.off_dec = off;
    if (bounded) off = align_up(off + sizeof(int) * size_t(total_segs) * p->Hv, 256);
    h.off_rerun = off;
    if (bounded) off = align_up(off + sizeof(int) * size_t(total_segs) * p->Hv, 256);
    h.off_prep = off;  // W', TU, P (and T) tiles of every (chunk, v-head): tensor-core path only
    h.prep_stride = backward ? gdn::PREP_BWD_BYTES : gdn::PREP_FWD_BYTES;
    if (p->dtype == GDN_BF16) off = align_up(off + size_t(h.prep_stride) * h.total_chunks * p->Hv, 256);
    if (backward) {
        const size_t elem = p->dtype == GDN_BF16 ? 2 : 4;
        const size_t per_chunk = size_t(128) * 128 * elem * p->Hv;
        h.off_hist = off;
        off = align_up(off + per_chunk * size_t(h.total_chunks), 256);
        h.off_dhist = off;
        off = align_up(off + per_chunk * size_t(h.total_chunks), 256);
        h.off_dhb = off;
        if (h.cp != gdn::CP_NONE) off = align_up(off + KVB * size_t(total_segs) * p->Hv, 256);
        h.off_rrerun = off;
        if (bounded) off = align_up(off + sizeof(int) * size_t(total_segs) * p->Hv, 256);
        h.off_dqp = off;
        if (p->Hv != p->Hqk) {
            const size_t part = size_t(h.total_tokens) * p->Hv * 128 * 4;
            off = align_up(off + part, 256);
            h.off_dkp = off;
            off = align_up(off + part, 256);
        } else {
            h.off_dkp = off;
        }
    }
    h.off_end = align_up(off, 256);
}

void fill_problem(const gdn_problem* p, const HostPlan& h, char* ws, gdn::Problem& P) {
    P.err = reinterpret_cast<int*>(ws + h.off_err);
    P.plan.seg = reinterpret_cast<int2*>(ws + h.off_seg);
    P.plan.seg_off = reinterpret_cast<int*>(ws + h.off_segoff);
    P.plan.chunk_off = reinterpret_cast<int*>(ws + h.off_chunkoff);
    if (!p->cu_seqlens) {  // equal lengths: the decomposition in closed form
        const int nt = (p->T + h.C - 1) / h.C;
        P.plan.uni_nt = nt;
        P.plan.uni_ns = std::max(1, (nt + h.L - 1) / h.L);
        P.plan.uni_n = h.N;
    } else {
        P.plan.uni_nt = P.plan.uni_ns = P.plan.uni_n = 0;
    }
    P.hin = h.cp != gdn::CP_NONE ? reinterpret_cast<float*>(ws + h.off_hin) : nullptr;
    P.mbuf = h.cp == gdn::CP_EXACT ? reinterpret_cast<float*>(ws + h.off_mbuf) : nullptr;
    P.mbuf_t = (h.cp == gdn::CP_EXACT && h.prep_stride == gdn::PREP_BWD_BYTES && p->dtype == GDN_BF16)
                   ? reinterpret_cast<float*>(ws + h.off_mbuf_t)
                   : nullptr;
    P.prep = p->dtype == GDN_BF16 ? ws + h.off_prep : nullptr;
    P.prep_stride = h.prep_stride;
    P.cu = p->cu_seqlens;
    P.N = h.N;
    P.T = p->T;
    P.Hqk = p->Hqk;
    P.Hv = p->Hv;
    P.total_segs = h.total_segs;
    P.total_chunks = h.total_chunks;
    P.L = h.L;
    P.warmup = h.warmup;
    P.cp = h.cp;
    P.full_cp = h.full_cp ? 1 : 0;
    const bool bounded = h.cp == gdn::CP_EXACT && !h.full_cp;
    P.logb = bounded ? reinterpret_cast<float*>(ws + h.off_logb) : nullptr;
    P.dec = bounded ? reinterpret_cast<int*>(ws + h.off_dec) : nullptr;
    P.rerun = bounded ? reinterpret_cast<int*>(ws + h.off_rerun) : nullptr;
    P.scale = p->scale;
}

// bf16 runs on the tcgen05 kernels; the fp32 test mode on the CUDA-core kernels.
bool use_tensor_cores(int dtype) { return dtype == GDN_BF16; }

gdn_status check_ptrs(std::initializer_list<const void*> required,
                      std::initializer_list<const void*> optional) {
    for (const void* x : required) {
        if (!x) return fail(GDN_ERR_INVALID_ARG, "a required tensor pointer is NULL");
        if (!aligned16(x)) return fail(GDN_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    }
    for (const void* x : optional)
        if (x && !aligned16(x))
            return fail(GDN_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    return GDN_OK;
}

}  // namespace

namespace gdn {
// Message for gdn_last_error() from entry points defined in other files.
void set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }
}  // namespace gdn

extern "C" {

const char* gdn_last_error(void) { return g_err; }

gdn_status gdn_device_status(const void* workspace, void* stream) {
    if (!workspace || !aligned16(workspace)) return fail(GDN_ERR_INVALID_ARG, "workspace missing or not 16-byte aligned");
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "reading the error word: %s", cudaGetErrorString(e));
    if (word & int(0x80000000u))  // ERR_BOUNDS: set by checked builds only
        return fail(GDN_ERR_BOUNDS, "a checked build skipped an out-of-range store (error word 0x%08x)",
                    unsigned(word));
    if (word != 0)
        return fail(GDN_ERR_TIMEOUT, "a device-side wait gave up (error word 0x%08x)", unsigned(word));
    return GDN_OK;
}

gdn_status gdn_debug_plan(const gdn_problem* p, int32_t sms, int32_t* chunks_per_segment,
                          int32_t* segments) {
    gdn_status st = validate_problem(p);
    if (st != GDN_OK) return st;
    if (!chunks_per_segment || !segments) return fail(GDN_ERR_INVALID_ARG, "output pointer is NULL");
    if (sms <= 0) return fail(GDN_ERR_INVALID_ARG, "sms must be positive (got %d)", sms);
    HostPlan h;
    plan(p, h, false, sms);
    *chunks_per_segment = h.L;
    *segments = h.total_segs;
    g_err[0] = 0;
    return GDN_OK;
}

gdn_status gdn_debug_wait_timeout(void* workspace, int32_t limit_us, void* stream) {
    if (!workspace || !aligned16(workspace)) return fail(GDN_ERR_INVALID_ARG, "workspace missing or not 16-byte aligned");
    if (limit_us < 1 || limit_us > 1000000) return fail(GDN_ERR_INVALID_ARG, "limit_us must be in [1, 1000000]");
    const cudaError_t e = gdn::launch_debug_wait(static_cast<int*>(workspace), limit_us,
                                                 static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "debug wait launch: %s", cudaGetErrorString(e));
    return GDN_OK;
}

gdn_status gdn_chunk_fwd_workspace_size(const gdn_problem* p, size_t* bytes) {
    gdn_status st = validate_problem(p);
    if (st != GDN_OK) return st;
    if (!bytes) return fail(GDN_ERR_INVALID_ARG, "bytes is NULL");
    HostPlan h;
    plan(p, h);
    *bytes = h.off_end;
    g_err[0] = 0;
    return GDN_OK;
}

gdn_status gdn_chunk_fwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* h0, void* o,
                         float* ht, void* workspace, size_t workspace_bytes, void* stream) {
    gdn_status st = validate_problem(p);
    if (st != GDN_OK) return st;
    HostPlan h;
    plan(p, h);
    if (h.total_tokens > 0) {
        st = check_ptrs({q, k, v, g, beta, o}, {h0, ht});
    } else {
        st = check_ptrs({}, {q, k, v, g, beta, o, h0, ht});
    }
    if (st != GDN_OK) return st;
    if (h.N == 0) {
        g_err[0] = 0;
        return GDN_OK;
    }
    if (!workspace || workspace_bytes < h.off_end)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", h.off_end,
                    workspace ? workspace_bytes : size_t(0));
    if (!aligned16(workspace)) return fail(GDN_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    gdn::Problem P{};
    P.q = q;
    P.k = k;
    P.v = v;
    P.g = g;
    P.beta = beta;
    P.h0 = h0;
    P.o = o;
    P.ht = ht;
    fill_problem(p, h, static_cast<char*>(workspace), P);
    cudaError_t e = use_tensor_cores(p->dtype)
                        ? gdn::launch_fwd_tc(P, false, h.total_tokens, static_cast<cudaStream_t>(stream))
                        : gdn::launch_fwd(P, p->dtype, false, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "CUDA error: %s", cudaGetErrorString(e));
    g_err[0] = 0;
    return GDN_OK;
}

gdn_status gdn_chunk_bwd_workspace_size(const gdn_problem* p, size_t* bytes) {
    gdn_status st = validate_problem(p);
    if (st != GDN_OK) return st;
    if (!bytes) return fail(GDN_ERR_INVALID_ARG, "bytes is NULL");
    HostPlan h;
    plan(p, h, true);
    *bytes = h.off_end;
    g_err[0] = 0;
    return GDN_OK;
}

gdn_status gdn_chunk_bwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* h0, const void* dO,
                         const float* dht, void* dq, void* dk, void* dv, float* dg,
                         float* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                         void* stream) {
    gdn_status st = validate_problem(p);
    if (st != GDN_OK) return st;
    HostPlan h;
    plan(p, h, true);
    if (h.total_tokens > 0)
        st = check_ptrs({q, k, v, g, beta, dO, dq, dk, dv, dg, dbeta}, {h0, dht, dh0});
    else
        st = check_ptrs({}, {q, k, v, g, beta, dO, dq, dk, dv, dg, dbeta, h0, dht, dh0});
    if (st != GDN_OK) return st;
    if (h.N == 0) {
        g_err[0] = 0;
        return GDN_OK;
    }
    if (!workspace || workspace_bytes < h.off_end)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", h.off_end,
                    workspace ? workspace_bytes : size_t(0));
    if (!aligned16(workspace)) return fail(GDN_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    char* ws = static_cast<char*>(workspace);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    gdn::BwdProblem B{};
    gdn::Problem& P = B.f;
    P.q = q;
    P.k = k;
    P.v = v;
    P.g = g;
    P.beta = beta;
    P.h0 = h0;
    P.o = nullptr;
    P.ht = nullptr;
    fill_problem(p, h, ws, P);
    P.hist = ws + h.off_hist;
    B.dO = dO;
    B.dht = dht;
    B.dh0 = dh0;
    B.dq = dq;
    B.dk = dk;
    B.dv = dv;
    B.dg = dg;
    B.dbeta = dbeta;
    B.dhist = ws + h.off_dhist;
    B.dhb = h.cp != gdn::CP_NONE ? reinterpret_cast<float*>(ws + h.off_dhb) : nullptr;
    B.rrerun = P.dec ? reinterpret_cast<int*>(ws + h.off_rrerun) : nullptr;
    B.dqp = p->Hv != p->Hqk ? reinterpret_cast<float*>(ws + h.off_dqp) : nullptr;
    B.dkp = p->Hv != p->Hqk ? reinterpret_cast<float*>(ws + h.off_dkp) : nullptr;
    // recompute the state entering every chunk, then the reverse scan and local gradients
    // (bf16 always on the tensor-core forward: the reverse scan reads its chunk records)
    cudaError_t e = p->dtype == GDN_BF16 ? gdn::launch_fwd_tc(P, true, h.total_tokens, cs)
                                         : gdn::launch_fwd(P, p->dtype, true, cs);
    if (e == cudaSuccess) e = gdn::launch_bwd(B, p->dtype, cs);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "CUDA error: %s", cudaGetErrorString(e));
    g_err[0] = 0;
    return GDN_OK;
}

gdn_status gdn_chunk_layout(const gdn_problem* p, int32_t* chunk_size, int64_t* total_chunks) {
    gdn_status st = validate_problem(p);
    if (st != GDN_OK) return st;
    if (!chunk_size || !total_chunks) return fail(GDN_ERR_INVALID_ARG, "output pointer is NULL");
    HostPlan h;
    plan(p, h, true);
    *chunk_size = h.C;
    *total_chunks = h.total_chunks;
    g_err[0] = 0;
    return GDN_OK;
}

gdn_status gdn_chunk_fwd_saved(const gdn_problem* p, const void* q, const void* k, const void* v,
                               const float* g, const float* beta, const float* h0, void* o,
                               float* ht, float* g_cum, void* A, void* h_chunks, void* workspace,
                               size_t workspace_bytes, void* stream) {
    gdn_status st = validate_problem(p);
    if (st != GDN_OK) return st;
    HostPlan h;
    plan(p, h, true);  // the backward's plan: exact CP, chunk records with T, M untransposed
    if (h.total_chunks > 0)
        st = check_ptrs({q, k, v, g, beta, o, h_chunks}, {h0, ht, g_cum, A});
    else
        st = check_ptrs({}, {q, k, v, g, beta, o, h0, ht, g_cum, A, h_chunks});
    if (st != GDN_OK) return st;
    if (h.N == 0) {
        g_err[0] = 0;
        return GDN_OK;
    }
    if (!workspace || workspace_bytes < h.off_end)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", h.off_end,
                    workspace ? workspace_bytes : size_t(0));
    if (!aligned16(workspace)) return fail(GDN_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    gdn::Problem P{};
    P.q = q;
    P.k = k;
    P.v = v;
    P.g = g;
    P.beta = beta;
    P.h0 = h0;
    P.o = o;
    P.ht = ht;
    fill_problem(p, h, static_cast<char*>(workspace), P);
    P.hist = h_chunks;
    P.gam_out = g_cum;
    P.a_out = A;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = p->dtype == GDN_BF16 ? gdn::launch_fwd_tc(P, false, h.total_tokens, cs)
                                         : gdn::launch_fwd(P, p->dtype, false, cs);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "CUDA error: %s", cudaGetErrorString(e));
    g_err[0] = 0;
    return GDN_OK;
}

gdn_status gdn_chunk_bwd_saved(const gdn_problem* p, const void* q, const void* k, const void* v,
                               const float* g, const float* beta, const void* h_chunks,
                               const void* dO, const float* dht, void* dq, void* dk, void* dv,
                               float* dg, float* dbeta, float* dh0, void* workspace,
                               size_t workspace_bytes, void* stream) {
    gdn_status st = validate_problem(p);
    if (st != GDN_OK) return st;
    HostPlan h;
    plan(p, h, true);
    if (h.total_chunks > 0)
        st = check_ptrs({q, k, v, g, beta, h_chunks, dO, dq, dk, dv, dg, dbeta}, {dht, dh0});
    else
        st = check_ptrs({}, {q, k, v, g, beta, h_chunks, dO, dq, dk, dv, dg, dbeta, dht, dh0});
    if (st != GDN_OK) return st;
    if (h.N == 0) {
        g_err[0] = 0;
        return GDN_OK;
    }
    if (!workspace || workspace_bytes < h.off_end)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", h.off_end,
                    workspace ? workspace_bytes : size_t(0));
    if (!aligned16(workspace)) return fail(GDN_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    char* ws = static_cast<char*>(workspace);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    gdn::BwdProblem B{};
    gdn::Problem& P = B.f;
    P.q = q;
    P.k = k;
    P.v = v;
    P.g = g;
    P.beta = beta;
    fill_problem(p, h, ws, P);
    P.hist = const_cast<void*>(h_chunks);
    B.dO = dO;
    B.dht = dht;
    B.dh0 = dh0;
    B.dq = dq;
    B.dk = dk;
    B.dv = dv;
    B.dg = dg;
    B.dbeta = dbeta;
    B.dhist = ws + h.off_dhist;
    B.dhb = h.cp != gdn::CP_NONE ? reinterpret_cast<float*>(ws + h.off_dhb) : nullptr;
    B.rrerun = P.dec ? reinterpret_cast<int*>(ws + h.off_rrerun) : nullptr;
    B.dqp = p->Hv != p->Hqk ? reinterpret_cast<float*>(ws + h.off_dqp) : nullptr;
    B.dkp = p->Hv != p->Hqk ? reinterpret_cast<float*>(ws + h.off_dkp) : nullptr;
    // the states, chunk records and segment transitions come from gdn_chunk_fwd_saved: only
    // the work decomposition is rebuilt before the reverse scan and the local gradients
    gdn::launch_plan(P, h.C, cs);
    cudaError_t e = gdn::launch_bwd(B, p->dtype, cs);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "CUDA error: %s", cudaGetErrorString(e));
    g_err[0] = 0;
    return GDN_OK;
}

namespace {
gdn_status prologue_common(const gdn_problem* p, gdn::PrologueArgs& A) {
    gdn_status st = validate_problem(p);
    if (st != GDN_OK) return st;
    const int64_t T_total = p->cu_seqlens ? int64_t(p->T) : int64_t(p->B) * p->T;
    A.dtype = p->dtype;
    A.rows = T_total * p->Hqk;
    A.gates = T_total * p->Hv;
    A.Hv = p->Hv;
    return GDN_OK;
}
}  // namespace

gdn_status gdn_prologue_fwd(const gdn_problem* p, const void* q_raw, const void* k_raw,
                            const float* a, const float* b, const float* A_log,
                            const float* dt_bias, void* q, void* k, float* g, float* beta,
                            void* stream) {
    gdn::PrologueArgs A{};
    gdn_status st = prologue_common(p, A);
    if (st != GDN_OK) return st;
    st = A.rows > 0 ? check_ptrs({q_raw, k_raw, a, b, A_log, dt_bias, q, k, g, beta}, {})
                    : check_ptrs({A_log, dt_bias}, {q_raw, k_raw, a, b, q, k, g, beta});
    if (st != GDN_OK) return st;
    if (A.rows == 0) {
        g_err[0] = 0;
        return GDN_OK;
    }
    A.q_raw = q_raw;
    A.k_raw = k_raw;
    A.a = a;
    A.b = b;
    A.A_log = A_log;
    A.dt_bias = dt_bias;
    A.q = q;
    A.k = k;
    A.g = g;
    A.beta = beta;
    cudaError_t e = gdn::launch_prologue_fwd(A, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "CUDA error: %s", cudaGetErrorString(e));
    g_err[0] = 0;
    return GDN_OK;
}

gdn_status gdn_prologue_bwd_workspace_size(const gdn_problem* p, size_t* bytes) {
    gdn_status st = validate_problem(p);
    if (st != GDN_OK) return st;
    if (!bytes) return fail(GDN_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = gdn::prologue_bwd_workspace(p->Hv);
    g_err[0] = 0;
    return GDN_OK;
}

gdn_status gdn_prologue_bwd(const gdn_problem* p, const void* q_raw, const void* k_raw,
                            const float* a, const float* b, const float* A_log,
                            const float* dt_bias, const void* dq, const void* dk,
                            const float* dg, const float* dbeta, void* dq_raw, void* dk_raw,
                            float* da, float* db, float* dA_log, float* ddt_bias,
                            void* workspace, size_t workspace_bytes, void* stream) {
    gdn::PrologueArgs A{};
    gdn_status st = prologue_common(p, A);
    if (st != GDN_OK) return st;
    st = A.rows > 0 ? check_ptrs({q_raw, k_raw, a, b, A_log, dt_bias, dq, dk, dg, dbeta, dq_raw,
                                  dk_raw, da, db, dA_log, ddt_bias}, {})
                    : check_ptrs({A_log, dt_bias, dA_log, ddt_bias},
                                 {q_raw, k_raw, a, b, dq, dk, dg, dbeta, dq_raw, dk_raw, da, db});
    if (st != GDN_OK) return st;
    const size_t need = gdn::prologue_bwd_workspace(p->Hv);
    if (!workspace || workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : size_t(0));
    if (!aligned16(workspace)) return fail(GDN_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    A.q_raw = q_raw;
    A.k_raw = k_raw;
    A.a = a;
    A.b = b;
    A.A_log = A_log;
    A.dt_bias = dt_bias;
    A.dq = dq;
    A.dk = dk;
    A.dg = dg;
    A.dbeta = dbeta;
    A.dq_raw = dq_raw;
    A.dk_raw = dk_raw;
    A.da = da;
    A.db = db;
    A.dA_log = dA_log;
    A.ddt_bias = ddt_bias;
    A.part = static_cast<float*>(workspace);
    cudaError_t e = gdn::launch_prologue_bwd(A, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "CUDA error: %s", cudaGetErrorString(e));
    g_err[0] = 0;
    return GDN_OK;
}

}  // extern "C"
