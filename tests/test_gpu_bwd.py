"""GPU parity of the backward (gdn_chunk_bwd through the C ABI) against the fp64 oracle's
hand-written reverse mode, on L = <o, dO> + <ht, dht>.

Tolerances as for the forward: max|err| <= 1e-2 max|ref| per gradient tensor for bf16 inputs,
<= 1e-4 max|ref| in the fp32 test mode."""
import numpy as np
import pytest
import torch

from chunked_prefill_gb300.inputs import make_inputs, workload_inputs
from tests.gpu_util import BF16_TOL, FP32_TOL, as_packed, gpu_bwd, oracle_bwd, rel_err

pytestmark = pytest.mark.gpu
NAMES = ["dq", "dk", "dv", "dg", "dbeta", "dh0"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_prefill_gb300 import build
    build.build()


def check(inp, tol, **kw):
    got = gpu_bwd(inp, **kw)
    ref = oracle_bwd(inp)
    errs = {}
    for name, a, b in zip(NAMES, got, ref):
        if a is None:
            continue
        errs[name] = rel_err(a.reshape(b.shape), b)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"relative errors above {tol}: {bad} (all: {errs})"
    return errs


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, BF16_TOL), (torch.float32, FP32_TOL)])
def test_small_training_step(dtype, tol):
    inp = make_inputs(1, 256, 2, 4, seed=40, dtype=dtype, h0_std=0.1, backward=True)
    check(inp, tol)


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, BF16_TOL), (torch.float32, FP32_TOL)])
@pytest.mark.parametrize("B,T,Hqk,Hv,h0", [
    (1, 1, 1, 1, True), (1, 63, 1, 3, False), (2, 64, 2, 2, True), (1, 65, 1, 2, True),
    (3, 200, 1, 3, True), (1, 129, 2, 2, False), (1, 200, 1, 10, True),
])
def test_odd_shapes(dtype, tol, B, T, Hqk, Hv, h0):
    inp = make_inputs(B, T, Hqk, Hv, seed=T * 3 + Hv, dtype=dtype, h0_std=0.1 if h0 else 0.0,
                      backward=True)
    check(inp, tol, cp_mode=1)
    check(inp, tol)


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, BF16_TOL), (torch.float32, FP32_TOL)])
def test_varlen_with_empty_sequences(dtype, tol):
    lens = [0, 5, 64, 130, 0, 77]
    inp = make_inputs(1, sum(lens), 2, 4, seed=41, dtype=dtype, h0_std=0.1, lengths=lens,
                      backward=True)
    check(inp, tol, cp_mode=1)
    check(inp, tol, cp_mode=2, cp_segment_chunks=1)


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, BF16_TOL), (torch.float32, FP32_TOL)])
@pytest.mark.parametrize("seg", [1, 2, 3, 5])
def test_context_parallel_exact(dtype, tol, seg):
    inp = make_inputs(1, 64 * 11 + 9, 1, 2, seed=42, dtype=dtype, h0_std=0.1, backward=True)
    check(inp, tol, cp_mode=2, cp_segment_chunks=seg)


def test_without_final_state_gradient_or_initial_state():
    inp = make_inputs(1, 300, 1, 2, seed=43, backward=True)
    inp.dht = None
    check(inp, BF16_TOL)


def test_determinism():
    inp = make_inputs(1, 500, 2, 4, seed=44, h0_std=0.1, backward=True)
    a = gpu_bwd(inp)
    b = gpu_bwd(inp)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_autograd_wrapper_matches_oracle():
    from chunked_prefill_gb300 import gdn
    inp = make_inputs(1, 200, 1, 2, seed=45, h0_std=0.1, backward=True)
    xs = {n: getattr(inp, n).cuda().requires_grad_(True) for n in ("q", "k", "v", "g", "beta", "h0")}
    o, ht = gdn.chunk_gated_delta_rule(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"],
                                       scale=inp.scale, initial_state=xs["h0"],
                                       output_final_state=True)
    loss = (o.float() * inp.dO.cuda().float()).sum() + (ht * inp.dht.cuda()).sum()
    loss.backward()
    ref = oracle_bwd(inp)
    for name, key, r in zip(NAMES, ["q", "k", "v", "g", "beta", "h0"], ref):
        got = xs[key].grad.float().cpu().numpy()
        assert rel_err(got.reshape(r.shape), r) <= BF16_TOL, name


def test_full_size_training_step_sampled_heads():
    """The 32K-token, 16/16-head training step in the benchmark's launch configuration; the
    oracle checks a sample of heads (heads are independent when each q/k head has one v
    head)."""
    inp = workload_inputs("fwdbwd_t32k_hqk16_hv16")
    got = gpu_bwd(inp)
    heads = [0, 5, 10, 15]
    sub = make_inputs(1, 16, 1, 1, backward=True)  # container; fields replaced below
    sub.q, sub.k = inp.q[:, :, heads], inp.k[:, :, heads]
    sub.v, sub.dO = inp.v[:, :, heads], inp.dO[:, :, heads]
    sub.g, sub.beta = inp.g[:, :, heads], inp.beta[:, :, heads]
    sub.h0, sub.dht = inp.h0[:, heads], inp.dht[:, heads]
    sub.scale, sub.cu_seqlens = inp.scale, None
    ref = oracle_bwd(sub)
    idx = {"dq": 2, "dk": 2, "dv": 2, "dg": 2, "dbeta": 2, "dh0": 1}
    for name, a, r in zip(NAMES, got, ref):
        a = np.take(a, heads, axis=idx[name])
        assert rel_err(a, r) <= BF16_TOL, name


@pytest.mark.parametrize("Hqk,Hv", [(2, 2), (2, 4)])
@pytest.mark.parametrize("cp_kw", [dict(cp_mode=2, cp_segment_chunks=3), {}])
def test_equal_length_batch_matches_packed(Hqk, Hv, cp_kw):
    """The training step of an equal-length batch (closed-form segmentation, no planner kernel
    in its forward recompute) against the same data packed with cu_seqlens (the planner's
    arrays): bitwise-equal gradients.  With one v-head per q/k head the local-gradient kernel
    writes full chunks' dq, dk, dv as tile stores and the cut last chunk by scalar stores."""
    inp = make_inputs(3, 64 * 9 + 17, Hqk, Hv, seed=72 + Hv, h0_std=0.1, backward=True)
    g1 = gpu_bwd(inp, **cp_kw)
    g2 = gpu_bwd(as_packed(inp), **cp_kw)
    for a, b in zip(g1, g2):
        if a is not None:
            assert np.array_equal(a.reshape(b.shape), b)
    ref = oracle_bwd(inp)
    for got, r in zip(g1, ref):
        if got is not None and r is not None:
            assert rel_err(got.reshape(r.shape), r) <= BF16_TOL


@pytest.mark.parametrize("Hqk,Hv", [(2, 12), (4, 24), (4, 48)])
def test_context_parallel_many_heads(Hqk, Hv):
    """Enough (sequence, v-head) chains that the fix-up runs 2, 4 or 8 column groups per CTA."""
    inp = make_inputs(1, 64 * 12 + 5, Hqk, Hv, seed=46 + Hv, h0_std=0.1, backward=True)
    check(inp, BF16_TOL, cp_mode=2, cp_segment_chunks=2)


@pytest.mark.parametrize("cp_mode", [None, 1])
def test_extreme_decay(cp_mode):
    """Chunk decays past exp(-80): the local-gradient kernel forms exp(gamma_i - gamma_j)
    directly instead of as exp(gamma_i) exp(-gamma_j)."""
    inp = make_inputs(1, 300, 1, 2, seed=47, h0_std=0.1, gate_scale=8.0, backward=True)
    kw = {} if cp_mode is None else {"cp_mode": cp_mode}
    check(inp, BF16_TOL, **kw)


def test_varlen_many_short_sequences():
    """Forty sequences of 1-199 tokens, q/k heads shared by two v-heads: several (chunk,
    v-head) items per CTA of the persistent local-gradient kernel, many of them cut by a
    sequence end (the next item's tiles and first products are requested and issued during
    the current one, except for a cut chunk, whose rows past the end are zeroed first)."""
    lens = [int(x) for x in np.random.RandomState(48).randint(1, 200, size=40)]
    inp = make_inputs(1, sum(lens), 4, 8, seed=48, h0_std=0.1, lengths=lens, backward=True)
    check(inp, BF16_TOL)
    check(inp, BF16_TOL, cp_mode=2, cp_segment_chunks=1)
