"""GPU parity of the forward (gdn_chunk_fwd through the C ABI) against the fp64 oracle.

Tolerances: max|err| <= 1e-2 max|ref| per output tensor for bf16 inputs with fp32
accumulation, <= 1e-4 max|ref| in the fp32 test mode."""
import numpy as np
import pytest
import torch

from chunked_prefill_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from oracle import chunked
from tests.gpu_util import BF16_TOL, FP32_TOL, as_packed, gpu_fwd, oracle_fwd, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_prefill_gb300 import build
    build.build()


def check(inp, tol, **kw):
    o, ht = gpu_fwd(inp, **kw)
    ro, rht = oracle_fwd(inp)
    eo, eh = rel_err(o, ro), rel_err(ht, rht)
    assert eo <= tol, f"o rel err {eo}"
    assert eh <= tol, f"ht rel err {eh}"
    return eo, eh


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, BF16_TOL), (torch.float32, FP32_TOL)])
def test_small_workload(dtype, tol):
    """B=1, T=256, 2 q/k heads shared by 4 v heads, h0 = 0: the small workload."""
    check(workload_inputs("fwd_t256_hqk2_hv4", dtype=dtype), tol)


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, BF16_TOL), (torch.float32, FP32_TOL)])
@pytest.mark.parametrize("B,T,Hqk,Hv,h0", [
    (1, 1, 1, 1, True), (1, 63, 1, 3, False), (2, 64, 2, 2, True), (1, 65, 1, 2, True),
    (3, 200, 1, 4, True), (1, 129, 3, 6, False),
    (1, 300, 1, 12, True),  # a q/k group of 12 v-heads: the preparation splits it in two slices
])
def test_odd_shapes(dtype, tol, B, T, Hqk, Hv, h0):
    inp = make_inputs(B, T, Hqk, Hv, seed=T * 7 + Hv, dtype=dtype, h0_std=0.1 if h0 else 0.0)
    check(inp, tol, cp_mode=1)
    check(inp, tol)  # planner's choice


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("cp_kw", [dict(cp_mode=2, cp_segment_chunks=3), dict(cp_mode=1), {}])
def test_equal_length_batch_matches_packed(dtype, cp_kw):
    """An equal-length batch (3 x 593 tokens: 10 chunks, the last cut) takes its segmentation
    in closed form and launches no planner; packed along one row with cu_seqlens it reads the
    planner's arrays.  Same kernels, same segments: bitwise-equal results."""
    inp = make_inputs(3, 64 * 9 + 17, 2, 4, seed=71, dtype=dtype, h0_std=0.1)
    o1, h1 = gpu_fwd(inp, **cp_kw)
    o2, h2 = gpu_fwd(as_packed(inp), **cp_kw)
    assert np.array_equal(o1.reshape(o2.shape), o2)
    assert np.array_equal(h1, h2)
    ro, rh = oracle_fwd(inp)
    tol = BF16_TOL if dtype == torch.bfloat16 else FP32_TOL
    assert rel_err(o1, ro) <= tol and rel_err(h1, rh) <= tol


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, BF16_TOL), (torch.float32, FP32_TOL)])
def test_varlen_with_empty_and_partial_sequences(dtype, tol):
    lens = [0, 1, 63, 64, 65, 130, 0, 7, 300]
    inp = make_inputs(1, sum(lens), 2, 4, seed=5, dtype=dtype, h0_std=0.1, lengths=lens)
    check(inp, tol, cp_mode=1)
    check(inp, tol, cp_mode=2, cp_segment_chunks=1)
    check(inp, tol, cp_mode=2, cp_segment_chunks=2)


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, BF16_TOL), (torch.float32, FP32_TOL)])
@pytest.mark.parametrize("seg", [1, 2, 3, 5, 64])
def test_context_parallel_exact(dtype, tol, seg):
    """Exact intra-GPU context parallelism: any segment length gives the serial result."""
    inp = make_inputs(1, 64 * 13 + 17, 1, 2, seed=11, dtype=dtype, h0_std=0.1)
    check(inp, tol, cp_mode=2, cp_segment_chunks=seg)


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, BF16_TOL), (torch.float32, FP32_TOL)])
@pytest.mark.parametrize("Hqk,Hv", [(2, 12), (4, 24), (4, 48)])
def test_context_parallel_many_heads(dtype, tol, Hqk, Hv):
    """Enough (sequence, v-head) chains that the fix-up runs 2, 4 or 8 column groups per CTA."""
    inp = make_inputs(1, 64 * 12 + 5, Hqk, Hv, seed=12 + Hv, dtype=dtype, h0_std=0.1)
    check(inp, tol, cp_mode=2, cp_segment_chunks=2)


def test_warmup_mode_matches_its_own_definition_fp32():
    """The opt-in warm-up mode is not exact; in the fp32 test mode it must equal the fp64
    chunk-form warm-up (same chunk size, segment length and window) to 1e-4."""
    inp = make_inputs(1, 32 * 24, 1, 2, seed=12, dtype=torch.float32, h0_std=0.1)
    inp.g.mul_(0.05)  # mild decay: the warm-up error is far above rounding
    o, ht = gpu_fwd(inp, cp_mode=3, cp_segment_chunks=4, warmup_chunks=2)
    cu = None
    ro, rht = chunked.fwd_cp(inp.q.double().numpy(), inp.k.double().numpy(),
                             inp.v.double().numpy(), inp.g.double().numpy(),
                             inp.beta.double().numpy(), inp.scale, h0=inp.h0.double().numpy(),
                             cu_seqlens=cu, chunk=32, seg_chunks=4, warmup=2)
    assert rel_err(o, ro) <= FP32_TOL
    assert rel_err(ht, rht) <= FP32_TOL
    # and it differs measurably from the exact result
    eo, _ = oracle_fwd(inp)
    assert rel_err(o, eo) > 1e-3


def _mixed_decay(inp, lo, hi):
    """No decay (g = 0) on tokens [lo, hi) of v-head 0, mild decay elsewhere on it, the
    default gates on the other v-heads: segments inside [lo, hi) keep their entering state
    (their transitions are computed and composed), the others forget it."""
    inp.g[:, :, 0].mul_(0.05)
    inp.g[:, lo:hi, 0] = 0.0
    return inp


@pytest.mark.parametrize("seg", [1, 2, 3, 4, 7])
def test_context_parallel_decay_bounded_mixed(seg):
    """Exact mode with decay bounds against the oracle and against the mode that computes
    every transition and reruns every segment (GDN_CP_EXACT_FULL), on gates that make some
    segments' transitions negligible and others not."""
    inp = _mixed_decay(make_inputs(1, 64 * 40 + 17, 1, 3, seed=31, h0_std=0.1), 64 * 9, 64 * 27)
    ro, rht = oracle_fwd(inp)
    o_b, ht_b = gpu_fwd(inp, cp_mode=2, cp_segment_chunks=seg)
    o_f, ht_f = gpu_fwd(inp, cp_mode=4, cp_segment_chunks=seg)
    for o, ht in ((o_b, ht_b), (o_f, ht_f)):
        assert rel_err(o, ro) <= BF16_TOL and rel_err(ht, rht) <= BF16_TOL
    # both are the exact result: they differ by rounding only
    assert rel_err(o_b, o_f) <= BF16_TOL and rel_err(ht_b, ht_f) <= BF16_TOL


def test_context_parallel_decay_bounded_large_keys():
    """Keys longer than 1 (beta |k|^2 up to ~2.9): some tokens' transitions expand, the
    chunks' log-bounds turn positive and the running sum is no longer monotone."""
    inp = make_inputs(1, 64 * 30 + 9, 2, 4, seed=32, h0_std=0.1)
    inp.k = (inp.k.float() * 1.7).to(inp.k.dtype)
    inp.g.mul_(0.3)
    for seg in (2, 5):
        check(inp, BF16_TOL, cp_mode=2, cp_segment_chunks=seg)


def test_context_parallel_decay_bounded_varlen_and_backward():
    """Varlen with empty, one-chunk and long sequences, mixed decay, through the forward and
    the backward (whose recompute and reverse fix-up use the same decisions)."""
    from tests.gpu_util import gpu_bwd, oracle_bwd
    lens = [0, 700, 64, 1500, 3, 900]
    inp = make_inputs(1, sum(lens), 1, 2, seed=33, h0_std=0.1, lengths=lens, backward=True)
    inp = _mixed_decay(inp, 800, 2000)
    check(inp, BF16_TOL, cp_mode=2, cp_segment_chunks=3)
    got = gpu_bwd(inp, cp_mode=2, cp_segment_chunks=3)
    ref = oracle_bwd(inp)
    for name, a, r in zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), got, ref):
        assert rel_err(a.reshape(r.shape), r) <= BF16_TOL, name


def _warmup_bounds(inp, chunk, seg_chunks, warmup):
    """Contraction bound of the warm-up mode's error (one sequence, every v-head): segment
    j >= 1 starts its scan `warmup` chunks early from zero, so its state at the segment start
    misses Phi h(s_j - w chunks), with ||Phi||_2 <= exp(sum of g over the window) when every
    beta ||k||^2 lies in [0, 2]; later in the segment the miss only contracts further.  Returns
    (bound on max |o error|, bound on max |ht error|), h(.) taken from the oracle on the
    prefix."""
    from oracle import oracle as orc
    T = inp.q.shape[1]
    g = inp.g[0].double().numpy()                 # [T, Hv]
    kn = (inp.k[0].double() ** 2).sum(-1).numpy()  # [T, Hqk]
    G = inp.v.shape[2] // inp.q.shape[2]
    assert (inp.beta[0].double().numpy() * np.repeat(kn, G, axis=1)).max() <= 2.0
    qn = float((inp.q[0].double() ** 2).sum(-1).sqrt().max())
    seg_tokens = seg_chunks * chunk
    bo, bh = 0.0, 0.0
    for s0 in range(seg_tokens, T, seg_tokens):
        w0 = max(0, s0 - warmup * chunk)
        if w0 == 0:
            continue  # the window reaches the sequence start: that segment is exact
        _, h_w = orc.fwd(inp.q[:, :w0], inp.k[:, :w0], inp.v[:, :w0], inp.g[:, :w0],
                         inp.beta[:, :w0], inp.scale, h0=inp.h0)
        for j in range(g.shape[1]):
            miss = np.exp(g[w0:s0, j].sum()) * np.linalg.norm(h_w[0, j], 2)
            bo = max(bo, inp.scale * qn * miss)
            if s0 + seg_tokens >= T:  # the last segment's miss reaches the final state
                bh = max(bh, np.exp(g[w0:T, j].sum()) * np.linalg.norm(h_w[0, j], 2))
    return bo, bh


@pytest.mark.parametrize("dtype,chunk,tol", [(torch.float32, 32, FP32_TOL), (torch.bfloat16, 64, BF16_TOL)])
def test_warmup_mode_error_within_contraction_bound(dtype, chunk, tol):
    """The opt-in warm-up mode's measured error stays within the contraction bound that the
    gates fix (plus the dtype's parity tolerance for rounding), with decay mild enough that
    the bound is far above rounding."""
    inp = make_inputs(1, chunk * 24, 1, 2, seed=13, dtype=dtype, h0_std=0.1)
    inp.g.mul_(0.05)
    o, ht = gpu_fwd(inp, cp_mode=3, cp_segment_chunks=4, warmup_chunks=2)
    ro, rht = oracle_fwd(inp)
    bo, bh = _warmup_bounds(inp, chunk, 4, 2)
    eo = float(np.abs(o - ro).max())
    eh = float(np.abs(ht - rht).max())
    assert eo <= 1.001 * bo + tol * np.abs(ro).max(), (eo, bo)
    assert eh <= 1.001 * bh + tol * np.abs(rht).max(), (eh, bh)
    if dtype == torch.float32:  # the bound, not the rounding allowance, is what is tested
        assert bo > 10 * tol * np.abs(ro).max()


def test_no_final_state_and_determinism():
    inp = make_inputs(1, 777, 2, 4, seed=14, h0_std=0.1)
    o1, ht = gpu_fwd(inp, output_final_state=False)
    assert ht is None
    o2, _ = gpu_fwd(inp, output_final_state=False)
    assert np.array_equal(o1, o2)


def test_extreme_decay_and_zero_beta():
    """Strong decay (gamma over a chunk far below -80) and beta = 0 rows."""
    inp = make_inputs(1, 300, 1, 2, seed=15, h0_std=0.1, gate_scale=8.0)
    inp.beta[:, ::3] = 0.0
    check(inp, BF16_TOL)


@pytest.mark.parametrize("name", ["fwd_t32k_hqk2_hv8", "fwd_t32k_hqk8_hv24",
                                  "fwd_varlen16_64k_hqk4_hv16"])
def test_full_size_workloads(name):
    """The full-size forward workloads in the benchmark's launch configuration (AUTO)."""
    check(workload_inputs(name), BF16_TOL)
