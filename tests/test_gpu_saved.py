"""GPU parity of the low-level forward / backward pair with saved intermediates
(gdn_chunk_fwd_saved, gdn_chunk_bwd_saved through the C ABI).

The forward's gamma, per-token rows of T = (I + A)^-1 and per-chunk entering states are
checked against the fp64 chunk-form oracle (itself pinned to the per-token recurrence), its
o and ht against gdn_chunk_fwd (bitwise: same kernels, same decomposition); the backward
from the saved states against gdn_chunk_bwd (bitwise) and the fp64 reverse-mode oracle."""
import numpy as np
import pytest
import torch

from chunked_prefill_gb300.inputs import make_inputs
from oracle import chunked
from tests.gpu_util import BF16_TOL, FP32_TOL, gpu_bwd, gpu_fwd, oracle_bwd, rel_err, to_dev

pytestmark = pytest.mark.gpu
NAMES = ["dq", "dk", "dv", "dg", "dbeta", "dh0"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_prefill_gb300 import build
    build.build()


def saved_fwd(inp, **kw):
    from chunked_prefill_gb300 import gdn
    d = to_dev(inp)
    out = gdn.gdn_chunk_fwd_saved(d["q"], d["k"], d["v"], d["g"], d["beta"], inp.scale,
                                  h0=d["h0"], cu_seqlens=d["cu"],
                                  cu_seqlens_host=inp.cu_seqlens, **kw)
    torch.cuda.synchronize()
    return d, out


def check_forward(inp, tol, **kw):
    from chunked_prefill_gb300 import gdn
    d, (g_cum, A, o, h, ht, ws) = saved_fwd(inp, **kw)
    C = A.shape[-1]
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy()
    rg, rA, ro, rh, rht = chunked.fwd_lowlevel(inp.q.double().numpy(), inp.k.double().numpy(),
                                               inp.v.double().numpy(), inp.g.numpy(),
                                               inp.beta.numpy(), inp.scale,
                                               h0=None if inp.h0 is None else inp.h0.numpy(),
                                               cu_seqlens=cu, chunk=C)
    errs = {
        "g_cum": rel_err(g_cum.cpu().numpy().reshape(rg.shape), rg),
        "A": rel_err(A.float().cpu().numpy().reshape(rA.shape), rA),
        "h": rel_err(h.float().cpu().numpy(), rh),
        "o": rel_err(o.float().cpu().numpy(), ro),
        "ht": rel_err(ht.cpu().numpy(), rht),
    }
    assert errs["g_cum"] <= 1e-5, errs
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"relative errors above {tol}: {bad}"
    # o and ht: the same kernels over the same decomposition as the plain forward
    o2, ht2 = gpu_fwd(inp, **kw)
    assert np.array_equal(o.float().cpu().numpy(), o2)
    assert np.array_equal(ht.cpu().numpy(), ht2)
    return d, h, ws


def check_backward(inp, tol, **kw):
    from chunked_prefill_gb300 import gdn
    d, h, ws = check_forward(inp, tol, **kw)
    got = gdn.gdn_chunk_bwd_saved(d["q"], d["k"], d["v"], d["g"], d["beta"], inp.scale, h, ws,
                                  d["dO"], dht=d["dht"], cu_seqlens=d["cu"],
                                  cu_seqlens_host=inp.cu_seqlens, want_dh0=True, **kw)
    torch.cuda.synchronize()
    got = [x.float().cpu().numpy() for x in got]
    plain = gpu_bwd(inp, **kw)
    for name, a, b in zip(NAMES, got, plain):
        assert np.array_equal(a.reshape(b.shape), b), name
    ref = oracle_bwd(inp)
    errs = {n: rel_err(a.reshape(r.shape), r) for n, a, r in zip(NAMES, got, ref)}
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"relative errors above {tol}: {bad}"


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, BF16_TOL), (torch.float32, FP32_TOL)])
def test_saved_pair_small(dtype, tol):
    inp = make_inputs(1, 256 + 37, 2, 4, seed=60, dtype=dtype, h0_std=0.1, backward=True)
    check_backward(inp, tol)


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, BF16_TOL), (torch.float32, FP32_TOL)])
def test_saved_pair_varlen_with_empty_sequences(dtype, tol):
    lens = [0, 5, 64, 130, 0, 77]
    inp = make_inputs(1, sum(lens), 2, 4, seed=61, dtype=dtype, h0_std=0.1, lengths=lens,
                      backward=True)
    check_backward(inp, tol, cp_mode=2, cp_segment_chunks=1)


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, BF16_TOL), (torch.float32, FP32_TOL)])
@pytest.mark.parametrize("seg", [2, 5])
def test_saved_pair_context_parallel(dtype, tol, seg):
    inp = make_inputs(1, 64 * 11 + 9, 1, 2, seed=62, dtype=dtype, h0_std=0.1, backward=True)
    check_backward(inp, tol, cp_mode=2, cp_segment_chunks=seg)


def test_saved_pair_many_heads_no_initial_state():
    inp = make_inputs(2, 64 * 6 + 3, 4, 24, seed=63, backward=True)
    check_backward(inp, BF16_TOL)


def test_autograd_with_saved_states_matches_recompute():
    from chunked_prefill_gb300 import gdn
    inp = make_inputs(1, 300, 1, 2, seed=64, h0_std=0.1, backward=True)
    grads = []
    for save in (False, True):
        xs = {n: getattr(inp, n).cuda().requires_grad_(True)
              for n in ("q", "k", "v", "g", "beta", "h0")}
        o, ht = gdn.chunk_gated_delta_rule(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"],
                                           scale=inp.scale, initial_state=xs["h0"],
                                           output_final_state=True, save_states=save)
        loss = (o.float() * inp.dO.cuda().float()).sum() + (ht * inp.dht.cuda()).sum()
        loss.backward()
        grads.append([xs[n].grad.float().cpu().numpy() for n in ("q", "k", "v", "g", "beta", "h0")])
    for a, b in zip(*grads):
        assert np.array_equal(a, b)


def test_low_level_names_match_the_saved_pair():
    """chunk_gated_delta_rule_fwd / _bwd (the usage page's low-level names, varlen form) give
    the saved pair's results bit for bit, and those are checked against the oracle above."""
    from chunked_prefill_gb300 import gdn
    lens = [70, 0, 129]
    inp = make_inputs(1, sum(lens), 2, 4, seed=65, h0_std=0.1, lengths=lens, backward=True)
    d, (g_cum, A, o, h, ht, ws) = saved_fwd(inp)
    ref_b = gdn.gdn_chunk_bwd_saved(d["q"], d["k"], d["v"], d["g"], d["beta"], inp.scale, h, ws,
                                    d["dO"], dht=d["dht"], cu_seqlens=d["cu"])
    got_f = gdn.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                           scale=inp.scale, initial_state=d["h0"],
                                           output_final_state=True, cu_seqlens=d["cu"])
    got_b = gdn.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], got_f[3],
                                           d["dO"], dht=d["dht"], scale=inp.scale,
                                           cu_seqlens=d["cu"])
    torch.cuda.synchronize()
    for a, b in zip(got_f, (g_cum, A, o, h, ht)):
        assert torch.equal(a, b)
    for name, a, b in zip(NAMES, got_b, ref_b):
        assert torch.equal(a, b), name
    with pytest.raises(ValueError):
        gdn.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h.clone(),
                                       d["dO"], scale=inp.scale, cu_seqlens=d["cu"])
