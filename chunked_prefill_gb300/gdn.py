"""Thin Python binding of libgdn.so (argument marshalling only; every step of the
computation runs in the library's CUDA kernels).

The names follow the C ABI (``gdn_chunk_fwd``, ``gdn_chunk_bwd``, ``*_workspace_size``)
and, on top, the FlashQLA pages' high-level call (aisparkup page, "usage":
``chunk_gated_delta_rule(q, k, v, g, beta, scale, initial_state, output_final_state,
cu_seqlens) -> (o, final_state)``) as a ``torch.autograd.Function``.

PyTorch supplies device memory and the stream; the library never allocates.  When
libgdn.so is missing this module raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# GDN_LIB selects another in-tree build of the same library (the checked variant
# libgdn_check.so in the bounds tests); the default is the release build
LIB_PATH = os.environ.get("GDN_LIB") or os.path.join(_HERE, "libgdn.so")

(GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE, GDN_ERR_CUDA, GDN_ERR_TIMEOUT,
 GDN_ERR_BOUNDS) = range(7)
GDN_BF16, GDN_FP32 = 0, 1
CP_AUTO, CP_OFF, CP_EXACT, CP_WARMUP, CP_EXACT_FULL = 0, 1, 2, 3, 4
_STATUS = {1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_WORKSPACE",
           4: "GDN_ERR_CUDA"}


class GdnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


class GdnProblem(ctypes.Structure):
    """Mirror of ``gdn_problem`` in include/gdn.h."""
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("Hqk", ctypes.c_int32),
                ("Hv", ctypes.c_int32), ("K", ctypes.c_int32), ("V", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float),
                ("cu_seqlens", ctypes.c_void_p), ("cu_seqlens_host", ctypes.c_void_p),
                ("num_seqs", ctypes.c_int32), ("cp_mode", ctypes.c_int32),
                ("cp_segment_chunks", ctypes.c_int32), ("warmup_chunks", ctypes.c_int32),
                ("cp_lambda", ctypes.c_float)]


class GdnKernelTime(ctypes.Structure):
    """Mirror of ``gdn_kernel_time``."""
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int32),
                ("total_ms", ctypes.c_float)]


_lib = None


def lib():
    """Load libgdn.so (built in-tree by ``chunked_prefill_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m chunked_prefill_gb300.build` (no fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        vp, P = ctypes.c_void_p, ctypes.POINTER(GdnProblem)
        L.gdn_chunk_fwd_workspace_size.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
        L.gdn_chunk_bwd_workspace_size.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
        L.gdn_chunk_fwd.argtypes = [P] + [vp] * 9 + [ctypes.c_size_t, vp]
        L.gdn_chunk_bwd.argtypes = [P] + [vp] * 15 + [ctypes.c_size_t, vp]
        L.gdn_chunk_layout.argtypes = [P, ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_int64)]
        L.gdn_debug_plan.argtypes = [P, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                                     ctypes.POINTER(ctypes.c_int32)]
        L.gdn_chunk_fwd_saved.argtypes = [P] + [vp] * 12 + [ctypes.c_size_t, vp]
        L.gdn_chunk_bwd_saved.argtypes = [P] + [vp] * 15 + [ctypes.c_size_t, vp]
        L.gdn_prologue_fwd.argtypes = [P] + [vp] * 10 + [vp]
        L.gdn_prologue_bwd_workspace_size.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
        L.gdn_prologue_bwd.argtypes = [P] + [vp] * 17 + [ctypes.c_size_t, vp]
        for f in ("gdn_chunk_fwd_workspace_size", "gdn_chunk_bwd_workspace_size",
                  "gdn_chunk_fwd", "gdn_chunk_bwd", "gdn_chunk_layout", "gdn_chunk_fwd_saved",
                  "gdn_chunk_bwd_saved", "gdn_prologue_fwd", "gdn_prologue_bwd_workspace_size",
                  "gdn_prologue_bwd"):
            getattr(L, f).restype = ctypes.c_int
        L.gdn_device_status.argtypes = [vp, vp]
        L.gdn_device_status.restype = ctypes.c_int
        L.gdn_debug_wait_timeout.argtypes = [vp, ctypes.c_int32, vp]
        L.gdn_debug_wait_timeout.restype = ctypes.c_int
        L.gdn_last_error.restype = ctypes.c_char_p
        L.gdn_timing_enable.argtypes = [ctypes.c_int32]
        L.gdn_timing_enable.restype = ctypes.c_int
        L.gdn_timing_collect.argtypes = [ctypes.POINTER(GdnKernelTime), ctypes.c_int32,
                                         ctypes.POINTER(ctypes.c_int32)]
        L.gdn_timing_collect.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(rc: int):
    if rc != GDN_OK:
        raise GdnError(rc, lib().gdn_last_error().decode())


def gdn_device_status(workspace, stream=None) -> int:
    """Wait for the stream and read the error word of a call's workspace: GDN_OK,
    GDN_ERR_BOUNDS when a checked build skipped an out-of-range store, or GDN_ERR_TIMEOUT
    when a device-side wait of that call gave up (see include/gdn.h)."""
    return lib().gdn_device_status(_ptr(workspace), _stream(stream))


def gdn_debug_wait_timeout(workspace, limit_us: int, stream=None):
    """Test hook: a kernel whose bounded wait runs out after limit_us, setting its bit in the
    error word of `workspace`."""
    _check(lib().gdn_debug_wait_timeout(_ptr(workspace), int(limit_us), _stream(stream)))


def gdn_timing_enable(on: bool = True):
    """Bracket every library kernel launch with CUDA events (see include/gdn.h)."""
    _check(lib().gdn_timing_enable(1 if on else 0))


def gdn_timing_collect() -> dict:
    """{kernel name: (launches, total ms)} since the last collect; waits on the events."""
    buf = (GdnKernelTime * 64)()
    n = ctypes.c_int32(0)
    _check(lib().gdn_timing_collect(buf, 64, ctypes.byref(n)))
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms))
            for i in range(min(n.value, 64))}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return GDN_BF16
    if dt == torch.float32:
        return GDN_FP32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {dt}")


class Problem:
    """A ``gdn_problem`` plus the host copy of cu_seqlens it points to (kept alive)."""

    def __init__(self, q, v, scale, cu_seqlens=None, cu_seqlens_host=None, cp_mode=CP_AUTO,
                 cp_segment_chunks=0, warmup_chunks=0, cp_lambda=0.0):
        B, T, Hqk, K = q.shape
        Hv, V = v.shape[2], v.shape[3]
        p = GdnProblem(B=B, T=T, Hqk=Hqk, Hv=Hv, K=K, V=V, dtype=_dtype_code(q.dtype),
                       scale=float(scale), cp_mode=cp_mode, cp_segment_chunks=cp_segment_chunks,
                       warmup_chunks=warmup_chunks, cp_lambda=cp_lambda)
        self._cu_host = None
        self.num_seqs = B
        if cu_seqlens is not None:
            if cu_seqlens_host is None:
                cu_seqlens_host = cu_seqlens.detach().to("cpu")
            self._cu_host = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous()
            self._cu_dev = cu_seqlens
            p.cu_seqlens = cu_seqlens.data_ptr()
            p.cu_seqlens_host = self._cu_host.data_ptr()
            p.num_seqs = self._cu_host.numel() - 1
            self.num_seqs = p.num_seqs
        self.p = p
        self.Hv, self.K, self.V = Hv, K, V

    def ref(self):
        return ctypes.byref(self.p)


def gdn_chunk_fwd_workspace_size(prob: Problem) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().gdn_chunk_fwd_workspace_size(prob.ref(), ctypes.byref(n)))
    return n.value


def gdn_chunk_bwd_workspace_size(prob: Problem) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().gdn_chunk_bwd_workspace_size(prob.ref(), ctypes.byref(n)))
    return n.value


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _workspace(nbytes, device, workspace):
    if workspace is not None and workspace.numel() * workspace.element_size() >= nbytes:
        return workspace
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


def _validate_tensors(q, k, v, g, beta):
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if k.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q and k must match in shape; q, k, v in dtype")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise ValueError("g and beta must be float32")
    if g.shape != v.shape[:3] or beta.shape != v.shape[:3]:
        raise ValueError("g and beta must be [B, T, Hv]")


def gdn_chunk_fwd(q, k, v, g, beta, scale, h0=None, output_final_state=True, cu_seqlens=None,
                  cu_seqlens_host=None, cp_mode=CP_AUTO, cp_segment_chunks=0, warmup_chunks=0,
                  cp_lambda=0.0, o=None, ht=None, workspace=None, stream=None):
    """Forward through the C ABI.  Returns (o, ht); ht is None unless requested."""
    _validate_tensors(q, k, v, g, beta)
    prob = Problem(q, v, scale, cu_seqlens, cu_seqlens_host, cp_mode, cp_segment_chunks,
                   warmup_chunks, cp_lambda)
    if o is None:
        o = torch.empty_like(v)
    if ht is None and output_final_state:
        ht = torch.empty(prob.num_seqs, prob.Hv, prob.K, prob.V, device=q.device,
                         dtype=torch.float32)
    if h0 is not None:
        h0 = h0.contiguous().float()
    nbytes = gdn_chunk_fwd_workspace_size(prob)
    ws = _workspace(nbytes, q.device, workspace)
    _check(lib().gdn_chunk_fwd(prob.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                               _ptr(h0), _ptr(o), _ptr(ht), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream)))
    return o, ht


def gdn_chunk_bwd(q, k, v, g, beta, scale, dO, h0=None, dht=None, cu_seqlens=None,
                  cu_seqlens_host=None, cp_mode=CP_AUTO, cp_segment_chunks=0, warmup_chunks=0,
                  cp_lambda=0.0, want_dh0=True, workspace=None, stream=None, out=None):
    """Backward through the C ABI.  Returns (dq, dk, dv, dg, dbeta, dh0)."""
    _validate_tensors(q, k, v, g, beta)
    if dO.shape != v.shape or dO.dtype != v.dtype or not dO.is_contiguous():
        raise ValueError("dO must be contiguous and match v")
    prob = Problem(q, v, scale, cu_seqlens, cu_seqlens_host, cp_mode, cp_segment_chunks,
                   warmup_chunks, cp_lambda)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dg, db = torch.empty_like(g), torch.empty_like(beta)
        dh0 = (torch.empty(prob.num_seqs, prob.Hv, prob.K, prob.V, device=q.device)
               if want_dh0 else None)
    else:
        dq, dk, dv, dg, db, dh0 = out
    if h0 is not None:
        h0 = h0.contiguous().float()
    if dht is not None:
        dht = dht.contiguous().float()
    nbytes = gdn_chunk_bwd_workspace_size(prob)
    ws = _workspace(nbytes, q.device, workspace)
    _check(lib().gdn_chunk_bwd(prob.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                               _ptr(h0), _ptr(dO), _ptr(dht), _ptr(dq), _ptr(dk), _ptr(dv),
                               _ptr(dg), _ptr(db), _ptr(dh0), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream)))
    return dq, dk, dv, dg, db, dh0


def gdn_chunk_layout(prob: Problem):
    """(chunk size C, chunks over all sequences) of the per-chunk saved outputs."""
    c, n = ctypes.c_int32(0), ctypes.c_int64(0)
    _check(lib().gdn_chunk_layout(prob.ref(), ctypes.byref(c), ctypes.byref(n)))
    return c.value, n.value


def gdn_debug_plan(prob: Problem, sms: int):
    """Test hook: (chunks per segment, segments) the planner picks for `prob` on `sms` SMs."""
    L, n = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib().gdn_debug_plan(prob.ref(), int(sms), ctypes.byref(L), ctypes.byref(n)))
    return L.value, n.value


def gdn_chunk_fwd_saved(q, k, v, g, beta, scale, h0=None, output_final_state=True,
                        cu_seqlens=None, cu_seqlens_host=None, cp_mode=CP_AUTO,
                        cp_segment_chunks=0, cp_lambda=0.0, want_g_cum=True, want_A=True,
                        workspace=None, stream=None, o=None, ht=None, h=None):
    """Low-level forward through the C ABI.  Returns (g_cum, A, o, h, ht, ctx): the in-chunk
    cumulative gate [B,T,Hv] (or None), every token's row of its chunk's (I + A)^-1
    [B,T,Hv,C] (or None), the output, the state entering every chunk [total_chunks,Hv,K,V],
    the final state (or None) and the workspace that gdn_chunk_bwd_saved reads back."""
    _validate_tensors(q, k, v, g, beta)
    prob = Problem(q, v, scale, cu_seqlens, cu_seqlens_host, cp_mode, cp_segment_chunks, 0,
                   cp_lambda)
    C, nchunks = gdn_chunk_layout(prob)
    B, T, Hv = v.shape[:3]
    if o is None:
        o = torch.empty_like(v)
    if ht is None and output_final_state:
        ht = torch.empty(prob.num_seqs, Hv, prob.K, prob.V, device=q.device, dtype=torch.float32)
    g_cum = torch.empty_like(g) if want_g_cum else None
    A = torch.empty(B, T, Hv, C, device=q.device, dtype=q.dtype) if want_A else None
    if h is None:
        h = torch.empty(max(nchunks, 0), Hv, prob.K, prob.V, device=q.device, dtype=q.dtype)
    if h0 is not None:
        h0 = h0.contiguous().float()
    nbytes = gdn_chunk_bwd_workspace_size(prob)
    ws = _workspace(nbytes, q.device, workspace)
    _check(lib().gdn_chunk_fwd_saved(prob.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                     _ptr(h0), _ptr(o), _ptr(ht), _ptr(g_cum), _ptr(A), _ptr(h),
                                     _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))
    return g_cum, A, o, h, ht, ws


def gdn_chunk_bwd_saved(q, k, v, g, beta, scale, h, ctx, dO, dht=None, cu_seqlens=None,
                        cu_seqlens_host=None, cp_mode=CP_AUTO, cp_segment_chunks=0,
                        cp_lambda=0.0, want_dh0=True, stream=None, out=None):
    """Backward from the saved states h and workspace ctx of gdn_chunk_fwd_saved (same
    problem arguments).  Returns (dq, dk, dv, dg, dbeta, dh0)."""
    _validate_tensors(q, k, v, g, beta)
    if dO.shape != v.shape or dO.dtype != v.dtype or not dO.is_contiguous():
        raise ValueError("dO must be contiguous and match v")
    prob = Problem(q, v, scale, cu_seqlens, cu_seqlens_host, cp_mode, cp_segment_chunks, 0,
                   cp_lambda)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dg, db = torch.empty_like(g), torch.empty_like(beta)
        dh0 = (torch.empty(prob.num_seqs, prob.Hv, prob.K, prob.V, device=q.device)
               if want_dh0 else None)
    else:
        dq, dk, dv, dg, db, dh0 = out
    if dht is not None:
        dht = dht.contiguous().float()
    _check(lib().gdn_chunk_bwd_saved(prob.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                     _ptr(h), _ptr(dO), _ptr(dht), _ptr(dq), _ptr(dk), _ptr(dv),
                                     _ptr(dg), _ptr(db), _ptr(dh0), _ptr(ctx),
                                     ctx.numel() * ctx.element_size(), _stream(stream)))
    return dq, dk, dv, dg, db, dh0


def chunk_gated_delta_rule_fwd(q, k, v, g, beta, scale=None, initial_state=None,
                               output_final_state=True, cu_seqlens=None, stream=None):
    """Low-level forward under the FlashQLA name (usage page, "low-level API"): returns
    (g_cum, A, o, h, final_state) -- the in-chunk cumulative gate, every token's row of its
    chunk's (I + A)^-1, the output, the state entering every chunk and the final state (None
    unless output_final_state).  The chunk records that chunk_gated_delta_rule_bwd reads back
    stay attached to h (attribute gdn_ctx), so h must be passed to it unchanged."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    g_cum, A, o, h, ht, ctx = gdn_chunk_fwd_saved(q, k, v, g, beta, scale, h0=initial_state,
                                                  output_final_state=output_final_state,
                                                  cu_seqlens=cu_seqlens, stream=stream)
    h.gdn_ctx = ctx
    return g_cum, A, o, h, ht


def chunk_gated_delta_rule_bwd(q, k, v, g, beta, h, do, dht=None, scale=None,
                               cu_seqlens=None, stream=None):
    """Low-level backward from chunk_gated_delta_rule_fwd's h (same q, k, v, g, beta, scale and
    cu_seqlens): returns (dq, dk, dv, dg, dbeta, dh0).  g and beta are the forward's inputs,
    not its cumulative gate."""
    ctx = getattr(h, "gdn_ctx", None)
    if ctx is None:
        raise ValueError("h must be the state tensor returned by chunk_gated_delta_rule_fwd")
    if scale is None:
        scale = q.shape[-1] ** -0.5
    return gdn_chunk_bwd_saved(q, k, v, g, beta, scale, h, ctx, do, dht=dht,
                               cu_seqlens=cu_seqlens, stream=stream)


def _prologue_problem(q_raw, a):
    if q_raw.dim() != 4 or a.dim() != 3 or a.shape[:2] != q_raw.shape[:2]:
        raise ValueError("q_raw must be [B,T,Hqk,K] and a [B,T,Hv]")
    B, T, Hqk, K = q_raw.shape
    Hv = a.shape[2]
    return GdnProblem(B=B, T=T, Hqk=Hqk, Hv=Hv, K=K, V=K, dtype=_dtype_code(q_raw.dtype),
                      scale=1.0, cp_mode=CP_AUTO)


def _check_prologue_inputs(q_raw, k_raw, a, b, A_log, dt_bias):
    for name, t in (("q_raw", q_raw), ("k_raw", k_raw), ("a", a), ("b", b), ("A_log", A_log),
                    ("dt_bias", dt_bias)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if k_raw.shape != q_raw.shape or k_raw.dtype != q_raw.dtype:
        raise ValueError("q_raw and k_raw must match in shape and dtype")
    for name, t in (("a", a), ("b", b), ("A_log", A_log), ("dt_bias", dt_bias)):
        if t.dtype != torch.float32:
            raise ValueError(f"{name} must be float32")
    if b.shape != a.shape or A_log.shape != (a.shape[2],) or dt_bias.shape != (a.shape[2],):
        raise ValueError("b must match a; A_log and dt_bias must be [Hv]")


def gdn_prologue_fwd(q_raw, k_raw, a, b, A_log, dt_bias, stream=None):
    """Fused prologue through the C ABI: (q, k, g, beta) from the raw projections."""
    _check_prologue_inputs(q_raw, k_raw, a, b, A_log, dt_bias)
    p = _prologue_problem(q_raw, a)
    q, k = torch.empty_like(q_raw), torch.empty_like(k_raw)
    g, beta = torch.empty_like(a), torch.empty_like(b)
    _check(lib().gdn_prologue_fwd(ctypes.byref(p), _ptr(q_raw), _ptr(k_raw), _ptr(a), _ptr(b),
                                  _ptr(A_log), _ptr(dt_bias), _ptr(q), _ptr(k), _ptr(g),
                                  _ptr(beta), _stream(stream)))
    return q, k, g, beta


def gdn_prologue_bwd(q_raw, k_raw, a, b, A_log, dt_bias, dq, dk, dg, dbeta, stream=None):
    """Reverse mode of the prologue: (dq_raw, dk_raw, da, db, dA_log, ddt_bias)."""
    _check_prologue_inputs(q_raw, k_raw, a, b, A_log, dt_bias)
    p = _prologue_problem(q_raw, a)
    dq, dk = dq.contiguous(), dk.contiguous()
    dg, dbeta = dg.contiguous().float(), dbeta.contiguous().float()
    dq_raw, dk_raw = torch.empty_like(q_raw), torch.empty_like(k_raw)
    da, db = torch.empty_like(a), torch.empty_like(b)
    dA_log, ddt_bias = torch.empty_like(A_log), torch.empty_like(dt_bias)
    n = ctypes.c_size_t(0)
    _check(lib().gdn_prologue_bwd_workspace_size(ctypes.byref(p), ctypes.byref(n)))
    ws = torch.empty(max(n.value, 16), dtype=torch.uint8, device=q_raw.device)
    _check(lib().gdn_prologue_bwd(ctypes.byref(p), _ptr(q_raw), _ptr(k_raw), _ptr(a), _ptr(b),
                                  _ptr(A_log), _ptr(dt_bias), _ptr(dq), _ptr(dk), _ptr(dg),
                                  _ptr(dbeta), _ptr(dq_raw), _ptr(dk_raw), _ptr(da), _ptr(db),
                                  _ptr(dA_log), _ptr(ddt_bias), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)))
    return dq_raw, dk_raw, da, db, dA_log, ddt_bias


class _Prologue(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q_raw, k_raw, a, b, A_log, dt_bias):
        ctx.save_for_backward(q_raw, k_raw, a, b, A_log, dt_bias)
        return gdn_prologue_fwd(q_raw, k_raw, a, b, A_log, dt_bias)

    @staticmethod
    def backward(ctx, dq, dk, dg, dbeta):
        q_raw, k_raw, a, b, A_log, dt_bias = ctx.saved_tensors
        zero = lambda t, like: torch.zeros_like(like) if t is None else t
        return gdn_prologue_bwd(q_raw, k_raw, a, b, A_log, dt_bias, zero(dq, q_raw),
                                zero(dk, k_raw), zero(dg, a), zero(dbeta, b))


def gated_delta_rule_prologue(q_raw, k_raw, a, b, A_log, dt_bias):
    """Differentiable fused prologue: q, k L2-normalised over K; g = -exp(A_log)
    softplus(a + dt_bias); beta = sigmoid(b).  Returns (q, k, g, beta)."""
    return _Prologue.apply(q_raw, k_raw, a, b, A_log, dt_bias)


class _ChunkGDN(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, h0, scale, output_final_state, cu_seqlens, save_states):
        if save_states:
            _, _, o, h, ht, ws = gdn_chunk_fwd_saved(q, k, v, g, beta, scale, h0=h0,
                                                     output_final_state=output_final_state,
                                                     cu_seqlens=cu_seqlens, want_g_cum=False,
                                                     want_A=False)
            ctx.save_for_backward(q, k, v, g, beta, h0, cu_seqlens, h, ws)
        else:
            o, ht = gdn_chunk_fwd(q, k, v, g, beta, scale, h0=h0,
                                  output_final_state=output_final_state, cu_seqlens=cu_seqlens)
            ctx.save_for_backward(q, k, v, g, beta, h0, cu_seqlens)
        ctx.scale = scale
        ctx.save_states = save_states
        return o, ht

    @staticmethod
    def backward(ctx, do, dht):
        if ctx.save_states:
            q, k, v, g, beta, h0, cu, h, ws = ctx.saved_tensors
            grads = gdn_chunk_bwd_saved(q, k, v, g, beta, ctx.scale, h, ws, do.contiguous(),
                                        dht=dht, cu_seqlens=cu, want_dh0=h0 is not None)
        else:
            q, k, v, g, beta, h0, cu = ctx.saved_tensors
            grads = gdn_chunk_bwd(q, k, v, g, beta, ctx.scale, do.contiguous(), h0=h0, dht=dht,
                                  cu_seqlens=cu, want_dh0=h0 is not None)
        return (*grads, None, None, None, None)


def chunk_gated_delta_rule(q, k, v, g, beta, scale=None, initial_state=None,
                           output_final_state=False, cu_seqlens=None, save_states=False):
    """High-level call with the FlashQLA/FLA signature; differentiable.
    q, k [B,T,Hqk,K]; v [B,T,Hv,V]; g, beta [B,T,Hv] (fp32); initial_state [N,Hv,K,V].
    save_states=True keeps the state entering every chunk (and the chunk records) from the
    forward for the backward, which then skips its recompute of the forward."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    return _ChunkGDN.apply(q, k, v, g, beta, initial_state, scale, output_final_state,
                           cu_seqlens, save_states)
