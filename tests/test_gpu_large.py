"""Offsets past 2^31 elements: a packed batch of two sequences whose second, short sequence
starts after token 16.8M, so that its q/k/v/o rows, its chunk records and its per-chunk states
sit beyond 32-bit element (and byte) offsets.  The GPU runs the whole batch (forward and
backward); the fp64 oracle checks the short sequence, which depends on nothing else.

Inputs are drawn on the device (a seeded generator) with the recipe of the other workloads;
only the short sequence's slice is copied to the host for the oracle."""
import numpy as np
import pytest
import torch

from tests.gpu_util import BF16_TOL, oracle_bwd, oracle_fwd, rel_err

pytestmark = pytest.mark.gpu

T_LONG, T_SHORT = (1 << 24) + 4096, 300   # 16.78M + 300 tokens; 128 x 16.78M > 2^31


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_prefill_gb300 import build
    build.build()


class _Sub:  # the short sequence as an oracle input set
    pass


def test_forward_and_backward_past_32bit_offsets():
    from chunked_prefill_gb300 import gdn
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev).manual_seed(77)
    T = T_LONG + T_SHORT
    nrm = lambda x: x / x.norm(dim=-1, keepdim=True)
    q = nrm(torch.randn(1, T, 1, 128, device=dev, generator=gen)).to(torch.bfloat16)
    k = nrm(torch.randn(1, T, 1, 128, device=dev, generator=gen)).to(torch.bfloat16)
    v = torch.randn(1, T, 1, 128, device=dev, generator=gen).to(torch.bfloat16)
    g = -torch.nn.functional.softplus(torch.randn(1, T, 1, device=dev, generator=gen))
    beta = torch.sigmoid(torch.randn(1, T, 1, device=dev, generator=gen))
    h0 = 0.1 * torch.randn(2, 1, 128, 128, device=dev, generator=gen)
    dO = torch.randn(1, T, 1, 128, device=dev, generator=gen).to(torch.bfloat16)
    dht = 0.1 * torch.randn(2, 1, 128, 128, device=dev, generator=gen)
    cu_host = torch.tensor([0, T_LONG, T], dtype=torch.int32)
    cu = cu_host.to(dev)
    scale = 128 ** -0.5
    o, ht = gdn.gdn_chunk_fwd(q, k, v, g, beta, scale, h0=h0, cu_seqlens=cu,
                              cu_seqlens_host=cu_host)
    grads = gdn.gdn_chunk_bwd(q, k, v, g, beta, scale, dO, h0=h0, dht=dht, cu_seqlens=cu,
                              cu_seqlens_host=cu_host)
    torch.cuda.synchronize()

    sl = slice(T_LONG, T)
    sub = _Sub()
    sub.q, sub.k, sub.v = (x[:, sl].cpu() for x in (q, k, v))
    sub.g, sub.beta, sub.dO = g[:, sl].cpu(), beta[:, sl].cpu(), dO[:, sl].cpu()
    sub.h0, sub.dht = h0[1:].cpu(), dht[1:].cpu()
    sub.scale, sub.cu_seqlens = scale, None
    ro, rht = oracle_fwd(sub)
    assert rel_err(o[:, sl].float().cpu().numpy(), ro) <= BF16_TOL
    assert rel_err(ht[1:].cpu().numpy(), rht) <= BF16_TOL
    ref = oracle_bwd(sub)
    for name, a, r in zip(["dq", "dk", "dv", "dg", "dbeta"], grads[:5], ref[:5]):
        got = a[:, sl].float().cpu().numpy()
        assert rel_err(got.reshape(r.shape), r) <= BF16_TOL, name
    assert rel_err(grads[5][1:].cpu().numpy(), ref[5]) <= BF16_TOL, "dh0"
