"""Seeded synthetic inputs for the gated delta rule workloads.

This module holds no arithmetic of the method itself: it only draws random tensors with the
distributions of the FlashQLA benchmark workloads (1 x 32768 tokens, q/k heads shared by
grouped v heads, K = V = 128; FlashQLA pages, "performance benchmark" table) and the usual
GDN input conventions (L2-normalised q/k, log-decay gate g = -softplus(x), write strength
beta = sigmoid(x)).  Both the CUDA path's tests and the oracle read the same CPU tensors, so
they see identical bits.

Draw order from one CPU generator: q, k, v, x_g, x_beta, h0, dO, dht, then (varlen only)
the sequence lengths.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int                 # tokens per sequence (or total tokens when varlen)
    Hqk: int
    Hv: int
    K: int = 128
    V: int = 128
    B: int = 1
    h0_std: float = 0.0    # 0 -> no initial state
    backward: bool = False
    varlen_seqs: int = 0   # >0 -> that many packed sequences summing to T tokens
    varlen_range: tuple = (256, 8192)
    seed: int = 1000


# The five workloads: a small one the oracle finishes in seconds, the small-head and the
# wider-head 32K-token forwards, a 16-sequence varlen forward and a 32K-token training step.
WORKLOADS = {
    w.name: w for w in [
        Workload("fwd_t256_hqk2_hv4", T=256, Hqk=2, Hv=4, seed=1000),
        Workload("fwd_t32k_hqk2_hv8", T=32768, Hqk=2, Hv=8, seed=1001),
        Workload("fwd_t32k_hqk8_hv24", T=32768, Hqk=8, Hv=24, h0_std=0.1, seed=1002),
        Workload("fwd_varlen16_64k_hqk4_hv16", T=65536, Hqk=4, Hv=16, h0_std=0.1,
                 varlen_seqs=16, seed=1003),
        Workload("fwdbwd_t32k_hqk16_hv16", T=32768, Hqk=16, Hv=16, h0_std=0.1,
                 backward=True, seed=1004),
    ]
}


# Head / length sweep (the pages benchmark the head settings h_v in {64, 48, 32, 24, 16, 8}
# across tensor-parallel degrees 1-8 and several lengths; FlashQLA pages, "performance
# benchmark" paragraph).  Reading: two model families with 16 q/k heads and 64 or 48 v-heads
# split over TP = 1, 2, 4, 8, keeping the splits whose v-head count is in that set; lengths
# 1 x 8192, 4 x 8192 and 1 x 32768 tokens.
def _sweep() -> dict:
    pts = []
    for hqk_all, hv_all in ((16, 64), (16, 48)):
        for tp in (1, 2, 4, 8):
            hqk, hv = hqk_all // tp, hv_all // tp
            if hv not in (64, 48, 32, 24, 16, 8):
                continue
            for B, T in ((1, 8192), (4, 8192), (1, 32768)):
                pts.append(Workload(f"sweep_b{B}_t{T // 1024}k_hqk{hqk}_hv{hv}", T=T, Hqk=hqk, Hv=hv, B=B,
                                    seed=2000 + len(pts)))
    return {w.name: w for w in pts}


SWEEP = _sweep()


def varlen_lengths(gen: torch.Generator, n: int, total: int, lo: int, hi: int) -> list[int]:
    """n lengths drawn uniformly from [lo, hi], rescaled to sum to exactly ``total`` by the
    largest-remainder method (ties go to the lower index).  Lengths may leave [lo, hi]."""
    raw = torch.randint(lo, hi + 1, (n,), generator=gen, dtype=torch.int64).tolist()
    s = sum(raw)
    base = [r * total // s for r in raw]
    frac = [(r * total) % s for r in raw]
    short = total - sum(base)
    order = sorted(range(n), key=lambda i: (-frac[i], i))
    for i in order[:short]:
        base[i] += 1
    return base


@dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    scale: float
    h0: torch.Tensor | None
    cu_seqlens: torch.Tensor | None      # int32 [N+1] or None
    dO: torch.Tensor | None = None
    dht: torch.Tensor | None = None
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return self.q.shape[0] if self.cu_seqlens is None else self.cu_seqlens.numel() - 1


def _l2n(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-6)


def make_inputs(B: int, T: int, Hqk: int, Hv: int, K: int = 128, V: int = 128, *,
                seed: int = 0, dtype: torch.dtype = torch.bfloat16, h0_std: float = 0.0,
                lengths: list[int] | None = None, backward: bool = False,
                varlen_seqs: int = 0, varlen_range=(256, 8192),
                gate_scale: float = 1.0) -> Inputs:
    """Draw one input set on the CPU.

    ``lengths`` packs explicit sequence lengths (B must be 1, T must equal their sum);
    ``varlen_seqs`` > 0 draws that many lengths after all tensors (see module docstring).
    ``gate_scale`` multiplies x before g = -softplus(x) (tests use it for extreme decay).
    """
    gen = torch.Generator().manual_seed(seed)
    q = _l2n(torch.randn(B, T, Hqk, K, generator=gen)).to(dtype)
    k = _l2n(torch.randn(B, T, Hqk, K, generator=gen)).to(dtype)
    v = torch.randn(B, T, Hv, V, generator=gen).to(dtype)
    g = -torch.nn.functional.softplus(gate_scale * torch.randn(B, T, Hv, generator=gen))
    beta = torch.sigmoid(torch.randn(B, T, Hv, generator=gen))
    if varlen_seqs:
        n_seq = varlen_seqs
    elif lengths is not None:
        n_seq = len(lengths)
    else:
        n_seq = B
    h0 = None
    if h0_std > 0:
        h0 = h0_std * torch.randn(n_seq, Hv, K, V, generator=gen)
    dO = dht = None
    if backward:
        dO = torch.randn(B, T, Hv, V, generator=gen).to(dtype)
        dht = 0.1 * torch.randn(n_seq, Hv, K, V, generator=gen)
    cu = None
    if varlen_seqs:
        assert B == 1
        lengths = varlen_lengths(gen, varlen_seqs, T, *varlen_range)
    if lengths is not None:
        assert B == 1 and sum(lengths) == T
        cu = torch.tensor([0] + list(torch.tensor(lengths).cumsum(0).tolist()), dtype=torch.int32)
    return Inputs(q, k, v, g.float().contiguous(), beta.float().contiguous(), K ** -0.5, h0, cu,
                  dO, dht, meta=dict(B=B, T=T, Hqk=Hqk, Hv=Hv, K=K, V=V))


def workload_inputs(name: str, dtype: torch.dtype = torch.bfloat16) -> Inputs:
    w = WORKLOADS[name] if name in WORKLOADS else SWEEP[name]
    return make_inputs(w.B, w.T, w.Hqk, w.Hv, w.K, w.V, seed=w.seed, dtype=dtype,
                       h0_std=w.h0_std, backward=w.backward, varlen_seqs=w.varlen_seqs,
                       varlen_range=w.varlen_range)


def make_prologue_inputs(B: int, T: int, Hqk: int, Hv: int, K: int = 128, *, seed: int = 0,
                         dtype: torch.dtype = torch.bfloat16, backward: bool = False) -> dict:
    """Raw projections for the fused prologue, drawn on the CPU: q_raw, k_raw ~ N(0, 1)
    [B, T, Hqk, K]; gate and beta pre-activations a, b ~ N(0, 1) [B, T, Hv]; per-head
    A_log = log U[1, 16] and dt_bias ~ N(0, 1) [Hv]; with ``backward`` also upstream
    gradients dq, dk ~ N(0, 1) and dg, dbeta ~ N(0, 1)."""
    gen = torch.Generator().manual_seed(seed)
    d = {
        "q_raw": torch.randn(B, T, Hqk, K, generator=gen).to(dtype),
        "k_raw": torch.randn(B, T, Hqk, K, generator=gen).to(dtype),
        "a": torch.randn(B, T, Hv, generator=gen),
        "b": torch.randn(B, T, Hv, generator=gen),
        "A_log": torch.log(1 + 15 * torch.rand(Hv, generator=gen)),
        "dt_bias": torch.randn(Hv, generator=gen),
    }
    if backward:
        d["dq"] = torch.randn(B, T, Hqk, K, generator=gen).to(dtype)
        d["dk"] = torch.randn(B, T, Hqk, K, generator=gen).to(dtype)
        d["dg"] = torch.randn(B, T, Hv, generator=gen)
        d["dbeta"] = torch.randn(B, T, Hv, generator=gen)
    return d
