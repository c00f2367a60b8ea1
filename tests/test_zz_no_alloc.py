"""gdn_chunk_fwd_noalloc, the allocation-free forward for callers that cannot allocate
device memory (a runtime that owns all device memory through its own pool, a
latency-critical loop where cudaMalloc may synchronise the device, a plug-in interface that
passes only inputs and outputs).  Its scratch is a fixed array inside the library.

Checked through the C ABI against gdn_chunk_fwd (which takes a caller-allocated
workspace), on two calls in a row so that the array's leftover contents from the first call
cannot leak into the second.  This file sorts last so that a run stopping at the first
failure has already run every other test; it also passes on its own in a fresh process."""
import ctypes

import pytest
import torch

from chunked_prefill_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

TOL = 1e-2  # the bf16 parity tolerance used by every forward test


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_prefill_gb300 import build, gdn as g
    build.build()
    L = g.lib()
    L.gdn_chunk_fwd_noalloc.argtypes = [ctypes.POINTER(g.GdnProblem)] + [ctypes.c_void_p] * 9
    L.gdn_chunk_fwd_noalloc.restype = ctypes.c_int
    return g


def _noalloc(g, inp, d, **kw):
    prob = g.Problem(d["q"], d["v"], inp.scale, **kw)
    o = torch.empty_like(d["v"])
    ht = torch.empty(prob.num_seqs, d["v"].shape[2], 128, 128, device="cuda")
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = g.lib().gdn_chunk_fwd_noalloc(prob.ref(), p(d["q"]), p(d["k"]), p(d["v"]), p(d["g"]),
                                       p(d["beta"]), p(d["h0"]), p(o), p(ht),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, o, ht


def _rel(a, b):
    a, b = a.float(), b.float()
    return float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))


def test_noalloc_matches_allocating_forward_twice_in_a_row(gdn):
    cases = [dict(T=64 * 40 + 17, Hqk=1, Hv=2, seed=21, kw=dict(cp_mode=2, cp_segment_chunks=4)),
             dict(T=64 * 25 + 5, Hqk=2, Hv=4, seed=22, kw=dict(cp_mode=2, cp_segment_chunks=3))]
    for c in cases:
        inp = make_inputs(1, c["T"], c["Hqk"], c["Hv"], seed=c["seed"], h0_std=0.1)
        d = {n: getattr(inp, n).cuda() for n in ("q", "k", "v", "g", "beta", "h0")}
        o_ref, ht_ref = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], inp.scale,
                                          h0=d["h0"], **c["kw"])
        rc, o, ht = _noalloc(gdn, inp, d, **c["kw"])
        torch.cuda.synchronize()
        assert rc == 0, gdn.lib().gdn_last_error().decode()
        assert _rel(o, o_ref) <= TOL
        assert _rel(ht, ht_ref) <= TOL


def test_noalloc_rejects_problems_beyond_its_scratch(gdn):
    # one segment per chunk on 32768 tokens x 16 heads needs far more than the fixed array
    inp = make_inputs(1, 32768, 1, 16, seed=23)
    d = {n: getattr(inp, n).cuda() for n in ("q", "k", "v", "g", "beta")}
    d["h0"] = None
    kw = dict(cp_mode=2, cp_segment_chunks=1)
    prob = gdn.Problem(d["q"], d["v"], inp.scale, **kw)
    assert gdn.gdn_chunk_fwd_workspace_size(prob) > (32 << 20)
    rc, _, _ = _noalloc(gdn, inp, d, **kw)
    assert rc == gdn.GDN_ERR_WORKSPACE
    assert "fixed" in gdn.lib().gdn_last_error().decode()
