"""gdn_chunk_fwd_noalloc, the allocation-free forward for callers that cannot allocate
device memory (a runtime that owns all device memory through its own pool, a
latency-critical loop where cudaMalloc may synchronise the device, a plug-in interface that
passes only inputs and outputs).  Its scratch is a fixed array inside the library.

Checked through the C ABI against gdn_chunk_fwd (which takes a caller-allocated
workspace): both run the same kernels with the same plan on the same inputs and the path is
deterministic, so the outputs must be bitwise equal -- a partial leak of the array's leftover
contents from an earlier call would show as a difference.  Each problem is called twice in a
row, after a different problem has left its contents in the array; one comparison with the
fp64 oracle at the bf16 tolerance of every forward test anchors the pair.  The array's error
word is read through gdn_noalloc_device_status, and a wait that runs out on that word is
reported there.  This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process."""
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
    L.gdn_noalloc_device_status.argtypes = [ctypes.c_void_p]
    L.gdn_noalloc_device_status.restype = ctypes.c_int
    L.gdn_noalloc_debug_wait_timeout.argtypes = [ctypes.c_int32, ctypes.c_void_p]
    L.gdn_noalloc_debug_wait_timeout.restype = ctypes.c_int
    return g


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(g, inp, d, **kw):
    prob = g.Problem(d["q"], d["v"], inp.scale, **kw)
    o = torch.empty_like(d["v"])
    ht = torch.empty(prob.num_seqs, d["v"].shape[2], 128, 128, device="cuda")
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = g.lib().gdn_chunk_fwd_noalloc(prob.ref(), p(d["q"]), p(d["k"]), p(d["v"]), p(d["g"]),
                                       p(d["beta"]), p(d["h0"]), p(o), p(ht), _stream())
    return rc, o, ht


def _rel(a, b):
    a, b = a.float(), b.float()
    return float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))


CASES = [dict(T=64 * 40 + 17, Hqk=1, Hv=2, seed=21, kw=dict(cp_mode=2, cp_segment_chunks=4)),
         dict(T=64 * 25 + 5, Hqk=2, Hv=4, seed=22, kw=dict(cp_mode=2, cp_segment_chunks=3))]


def test_noalloc_matches_allocating_forward_twice_in_a_row(gdn):
    from oracle import oracle as orc
    prepared = []
    for c in CASES:
        inp = make_inputs(1, c["T"], c["Hqk"], c["Hv"], seed=c["seed"], h0_std=0.1)
        d = {n: getattr(inp, n).cuda() for n in ("q", "k", "v", "g", "beta", "h0")}
        o_ref, ht_ref = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], inp.scale,
                                          h0=d["h0"], **c["kw"])
        prepared.append((c, inp, d, o_ref, ht_ref))
    # case 0, case 1, then case 0 and case 1 again: every call after the first finds the
    # array holding another call's contents
    for rep in range(2):
        for c, inp, d, o_ref, ht_ref in prepared:
            rc, o, ht = _noalloc(gdn, inp, d, **c["kw"])
            assert rc == 0, gdn.lib().gdn_last_error().decode()
            assert gdn.lib().gdn_noalloc_device_status(_stream()) == gdn.GDN_OK
            assert torch.equal(o, o_ref), f"o differs (call {rep + 1}, seed {c['seed']})"
            assert torch.equal(ht, ht_ref), f"ht differs (call {rep + 1}, seed {c['seed']})"
    c, inp, d, o_ref, ht_ref = prepared[0]
    ro, rht = orc.fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, h0=inp.h0)
    assert _rel(o_ref.cpu(), torch.from_numpy(ro)) <= TOL
    assert _rel(ht_ref.cpu(), torch.from_numpy(rht)) <= TOL


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


def test_noalloc_failure_report_reaches_the_caller(gdn):
    """A bounded wait that runs out on the array's error word is reported by
    gdn_noalloc_device_status; the next no-alloc forward clears the word and is correct."""
    L = gdn.lib()
    assert L.gdn_noalloc_debug_wait_timeout(2000, _stream()) == gdn.GDN_OK
    assert L.gdn_noalloc_device_status(_stream()) == gdn.GDN_ERR_TIMEOUT
    c = CASES[1]
    inp = make_inputs(1, c["T"], c["Hqk"], c["Hv"], seed=c["seed"], h0_std=0.1)
    d = {n: getattr(inp, n).cuda() for n in ("q", "k", "v", "g", "beta", "h0")}
    o_ref, ht_ref = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], inp.scale,
                                      h0=d["h0"], **c["kw"])
    rc, o, ht = _noalloc(gdn, inp, d, **c["kw"])
    assert rc == 0, L.gdn_last_error().decode()
    assert L.gdn_noalloc_device_status(_stream()) == gdn.GDN_OK
    assert torch.equal(o, o_ref) and torch.equal(ht, ht_ref)
