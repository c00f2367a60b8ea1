"""GPU parity of the fused prologue (gdn_prologue_fwd / gdn_prologue_bwd through the C ABI)
against its fp64 oracle, and of the prologue feeding the chunked forward and backward."""
import numpy as np
import pytest
import torch

from chunked_prefill_gb300.inputs import make_inputs, make_prologue_inputs
from oracle import oracle as orc
from oracle import prologue as pro
from tests.gpu_util import BF16_TOL, FP32_TOL, rel_err

pytestmark = pytest.mark.gpu
GATE_TOL = 1e-5  # fp32 activations against fp64


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_prefill_gb300 import build
    build.build()


def np64(t):
    return t.double().cpu().numpy()


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, BF16_TOL), (torch.float32, FP32_TOL)])
@pytest.mark.parametrize("B,T,Hqk,Hv", [(1, 1, 1, 1), (2, 333, 2, 6), (1, 4099, 4, 16)])
def test_prologue_forward_and_reverse(dtype, tol, B, T, Hqk, Hv):
    from chunked_prefill_gb300 import gdn
    d = make_prologue_inputs(B, T, Hqk, Hv, seed=T + Hv, dtype=dtype, backward=True)
    x = {n: t.cuda() for n, t in d.items()}
    names = ("q_raw", "k_raw", "a", "b", "A_log", "dt_bias")
    q, k, g, beta = gdn.gdn_prologue_fwd(*(x[n] for n in names))
    rq, rk, rg, rb = pro.fwd(*(np64(d[n]) for n in names))
    assert rel_err(np64(q), rq) <= tol
    assert rel_err(np64(k), rk) <= tol
    assert rel_err(np64(g), rg) <= GATE_TOL
    assert rel_err(np64(beta), rb) <= GATE_TOL
    got = gdn.gdn_prologue_bwd(*(x[n] for n in names), x["dq"], x["dk"], x["dg"], x["dbeta"])
    ref = pro.bwd(*(np64(d[n]) for n in names), np64(d["dq"]), np64(d["dk"]), np64(d["dg"]),
                  np64(d["dbeta"]))
    for name, a, r, t in zip(["dq_raw", "dk_raw", "da", "db", "dA_log", "ddt_bias"], got, ref,
                             [tol, tol, GATE_TOL, GATE_TOL, 1e-4, 1e-4]):
        assert rel_err(np64(a), r) <= t, name


def test_prologue_in_place_matches_out_of_place():
    from chunked_prefill_gb300 import gdn
    d = make_prologue_inputs(1, 700, 2, 4, seed=5)
    x = {n: t.cuda() for n, t in d.items()}
    names = ("q_raw", "k_raw", "a", "b", "A_log", "dt_bias")
    want = gdn.gdn_prologue_fwd(*(x[n] for n in names))
    L = gdn.lib()
    p = gdn._prologue_problem(x["q_raw"], x["a"])
    import ctypes
    gdn._check(L.gdn_prologue_fwd(ctypes.byref(p), *(gdn._ptr(x[n]) for n in names),
                                  gdn._ptr(x["q_raw"]), gdn._ptr(x["k_raw"]), gdn._ptr(x["a"]),
                                  gdn._ptr(x["b"]), gdn._stream(None)))
    torch.cuda.synchronize()
    for a, b in zip(want, (x["q_raw"], x["k_raw"], x["a"], x["b"])):
        assert torch.equal(a, b)


def test_prologue_then_chunked_path_against_composed_oracle():
    """Raw projections -> prologue -> chunk_gated_delta_rule, forward and backward through
    autograd, against the composed fp64 oracles (prologue, per-token recurrence and their
    reverse modes)."""
    from chunked_prefill_gb300 import gdn
    B, T, Hqk, Hv = 1, 300, 2, 4
    d = make_prologue_inputs(B, T, Hqk, Hv, seed=7)
    side = make_inputs(B, T, Hqk, Hv, seed=8, h0_std=0.1, backward=True)
    names = ("q_raw", "k_raw", "a", "b", "A_log", "dt_bias")
    x = {n: d[n].cuda().requires_grad_(True) for n in names}
    v = side.v.cuda().requires_grad_(True)
    q, k, g, beta = gdn.gated_delta_rule_prologue(*(x[n] for n in names))
    o, ht = gdn.chunk_gated_delta_rule(q, k, v, g, beta, scale=side.scale,
                                       initial_state=side.h0.cuda(), output_final_state=True)
    loss = (o.float() * side.dO.cuda().float()).sum() + (ht * side.dht.cuda()).sum()
    loss.backward()

    rq, rk, rg, rb = pro.fwd(*(np64(d[n]) for n in names))
    ro, rht = orc.fwd(rq, rk, np64(side.v), rg, rb, side.scale, h0=np64(side.h0))
    assert rel_err(np64(o.detach()), ro) <= BF16_TOL
    dq, dk, dv, dg, dbeta, _ = orc.bwd(rq, rk, np64(side.v), rg, rb, side.scale, np64(side.dO),
                                       h0=np64(side.h0), dht=np64(side.dht))
    ref = pro.bwd(*(np64(d[n]) for n in names), dq, dk, dg, dbeta)
    for n, r in zip(names, ref):
        assert rel_err(np64(x[n].grad), r) <= BF16_TOL, n
    assert rel_err(np64(v.grad), dv) <= BF16_TOL
