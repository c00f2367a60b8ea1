"""Shared helpers of the GPU parity tests: run the CUDA path through the binding and the
fp64 oracle on the same (already rounded) CPU inputs."""
import numpy as np
import torch

from oracle import oracle as orc

BF16_TOL = 1e-2   # max|err| <= 1e-2 max|ref| for bf16 inputs with fp32 accumulation
FP32_TOL = 1e-4   # max|err| <= 1e-4 max|ref| in the fp32 test mode


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def to_dev(inp):
    d = {}
    for name in ("q", "k", "v", "g", "beta", "h0", "dO", "dht"):
        t = getattr(inp, name)
        d[name] = None if t is None else t.cuda().contiguous()
    d["cu"] = None if inp.cu_seqlens is None else inp.cu_seqlens.cuda()
    return d


def oracle_fwd(inp):
    return orc.fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, h0=inp.h0,
                   cu_seqlens=None if inp.cu_seqlens is None else inp.cu_seqlens.numpy())


def oracle_bwd(inp):
    return orc.bwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, inp.dO, h0=inp.h0,
                   dht=inp.dht,
                   cu_seqlens=None if inp.cu_seqlens is None else inp.cu_seqlens.numpy())


def gpu_fwd(inp, **kw):
    from chunked_prefill_gb300 import gdn
    d = to_dev(inp)
    o, ht = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], inp.scale,
                              h0=d["h0"], cu_seqlens=d["cu"],
                              cu_seqlens_host=inp.cu_seqlens, **kw)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), (None if ht is None else ht.cpu().numpy())


def gpu_bwd(inp, **kw):
    from chunked_prefill_gb300 import gdn
    d = to_dev(inp)
    res = gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], inp.scale, d["dO"],
                            h0=d["h0"], dht=d["dht"], cu_seqlens=d["cu"],
                            cu_seqlens_host=inp.cu_seqlens, **kw)
    torch.cuda.synchronize()
    return [None if r is None else r.float().cpu().numpy() for r in res]


def as_packed(inp):
    """The same equal-length batch as varlen sequences packed along one row (cu_seqlens at
    multiples of T): the library then reads the planner kernel's segmentation arrays instead
    of the closed form it uses for an equal-length batch."""
    import dataclasses
    B, T = inp.q.shape[:2]
    fields = {}
    for name in ("q", "k", "v", "g", "beta", "dO"):
        t = getattr(inp, name)
        fields[name] = None if t is None else t.reshape(1, B * T, *t.shape[2:]).contiguous()
    fields["cu_seqlens"] = torch.arange(0, B * T + 1, T, dtype=torch.int32)
    return dataclasses.replace(inp, **fields)
