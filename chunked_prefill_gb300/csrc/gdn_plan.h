// Host/device shared description of one call's work decomposition.
//
// Each sequence s has NT_s = ceil(len_s / C) chunks, split into nseg_s = max(1,
// ceil(NT_s / L)) segments of L chunks (FlashQLA pages, "AutoCP": CP ranks of L chunks
// each).  Segments of all sequences are numbered globally; seg_off[s] is the first global
// segment of sequence s and chunk_off[s] its first global chunk.
#pragma once
#include <stdint.h>

namespace gdn {

enum CpKind { CP_NONE = 0, CP_EXACT = 1, CP_WARMUP = 2 };

// A transition whose 2-norm is bounded by exp(LOG_NEGLIGIBLE) = 2^-126 (the smallest normal
// fp32 number) contributes less than 2^-126 ||h|| to any state it maps h into: it is dropped.
constexpr float LOG_NEGLIGIBLE = -87.33654475f;

// Work decomposition: the segments of the sequences and the first chunk of each sequence.  A
// batch of equal-length sequences (no cu_seqlens) has it in closed form (uni_ns > 0: every
// sequence has uni_ns segments and uni_nt chunks) and no kernel writes or reads the arrays;
// packed sequences read the arrays the planner kernel writes from the device cu_seqlens.
struct PlanDev {
    int2* seg;          // [total_segs] (sequence, local segment index)
    int* seg_off;       // [N+1]
    int* chunk_off;     // [N+1]
    int uni_ns;         // > 0: segments per sequence of an equal-length batch
    int uni_nt;         //      chunks per sequence
    int uni_n;          //      sequences
};
// (sequence, local segment) of global segment g, or (-1, -1) past the last
__device__ __forceinline__ int2 plan_seg(const PlanDev& p, int g) {
    if (p.uni_ns > 0)
        return g < p.uni_n * p.uni_ns ? make_int2(g / p.uni_ns, g % p.uni_ns) : make_int2(-1, -1);
    return p.seg[g];
}
// first global segment of sequence s (s = N: the number of segments)
__device__ __forceinline__ int plan_seg_off(const PlanDev& p, int s) {
    return p.uni_ns > 0 ? s * p.uni_ns : p.seg_off[s];
}
// first global chunk of sequence s (s = N: the number of chunks)
__device__ __forceinline__ int plan_chunk_off(const PlanDev& p, int s) {
    return p.uni_ns > 0 ? s * p.uni_nt : p.chunk_off[s];
}

struct Problem {
    // tensors
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    const float* h0;    // [N, Hv, K, V] or null
    void* o;
    float* ht;          // [N, Hv, K, V] or null
    // workspace
    float* hin;         // [total_segs, Hv, K, V]  entering state of each segment
    float* mbuf;        // [total_segs, Hv, K, K]  segment transitions, stored transposed (exact CP)
    float* mbuf_t;      // the same transitions untransposed (bf16 backward only), or null
    void* hist;         // [total_chunks, Hv, K, V] entering state of every chunk (bwd); in the
                        // output stage non-null asks for the same store next to the outputs
    float* gam_out;     // [T, Hv] in-chunk cumulative gate gamma, or null (not returned)
    void* a_out;        // [T, Hv, C] row of the chunk's T = (I + A)^-1 for every token, or null
    void* prep;         // [total_chunks, Hv] records of prep_stride bytes (tensor-core path)
    int64_t prep_stride;  // 32 KB (W', TU, P), or 40 KB with T as well (the backward needs it)
    PlanDev plan;
    const int* cu;      // device cu_seqlens or null
    int N, T, Hqk, Hv;
    int total_segs, total_chunks;
    int L;              // chunks per segment
    int warmup;         // warm-up chunks (CP_WARMUP)
    int cp;             // CpKind
    // Exact context parallelism with decay bounds (bf16 path, CP_EXACT unless full_cp):
    // logb[chunk][v-head] = log of a bound on the 2-norm of the chunk's state transition
    // (written by the preparation), dec[segment][v-head] = -1 when the segment's transition is
    // not negligible, else 0 (written by the first output pass; read by the transition, fix-up
    // and correction launches)
    float* logb;        // [total_chunks, Hv] or null
    int* dec;           // [total_segs, Hv] or null
    int* rerun;         // [total_segs, Hv] or null: some result of the segment is left to the
                        // correction pass
    int full_cp;        // 1: every transition computed and every segment rerun (no bound)
    int prep_heads;     // v-heads per preparation CTA (set by the preparation's launcher)
    float scale;
    int* err;           // device error word (bounded waits that timed out), or null
};

// Backward: the forward fields (recompute of the per-chunk states uses them) plus the
// gradient tensors and the backward's own workspace.
struct BwdProblem {
    Problem f;
    const void* dO;     // [T, Hv, V]
    const float* dht;   // [N, Hv, K, V] or null (zero)
    float* dh0;         // [N, Hv, K, V] or null (not returned)
    void* dq;           // [T, Hqk, K]
    void* dk;           // [T, Hqk, K]
    void* dv;           // [T, Hv, V]
    float* dg;          // [T, Hv]
    float* dbeta;       // [T, Hv]
    void* dhist;        // [total_chunks, Hv, K, V] gradient w.r.t. the state leaving each chunk
    float* dhb;         // [total_segs, Hv, K, V] gradient entering each segment from the right
    int* rrerun;        // [total_segs, Hv] decay-bounded reverse scan: some gradient of the
                        // segment is left to the correction pass (or null)
    float* dqp;         // [T, Hv, K] per-v-head partial dq (G > 1) or null
    float* dkp;         // [T, Hv, K] per-v-head partial dk (G > 1) or null
};

}  // namespace gdn
