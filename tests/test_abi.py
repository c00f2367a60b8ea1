"""The C ABI without a GPU: libgdn.so builds, loads, exports every function include/gdn.h
declares, and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest

from chunked_prefill_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    from chunked_prefill_gb300 import gdn
    return gdn


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(gdn_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"gdn_chunk_fwd", "gdn_chunk_bwd", "gdn_chunk_fwd_workspace_size",
            "gdn_chunk_bwd_workspace_size", "gdn_last_error"} <= set(names)
    lib = ctypes.CDLL(L.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def problem(L, **kw):
    base = dict(B=1, T=256, Hqk=2, Hv=4, K=128, V=128, dtype=0, scale=128 ** -0.5,
                cp_mode=L.CP_OFF)
    base.update(kw)
    return L.GdnProblem(**base)


def fwd_status(L, p, ptrs=None, ws_bytes=1 << 30):
    fake = ctypes.c_void_p(0x10000)
    args = ptrs or [fake] * 5 + [None, fake, fake, fake]  # q k v g beta h0 o ht ws
    lib = L.lib()
    rc = lib.gdn_chunk_fwd(ctypes.byref(p), *args[:8], args[8], ws_bytes, None)
    return rc, lib.gdn_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(K=64, V=64), 2),          # unsupported head dim
    (dict(K=0), 1),
    (dict(Hv=3), 1),                # Hv not a multiple of Hqk
    (dict(dtype=7), 1),
    (dict(T=-1), 1),
    (dict(cp_mode=9), 1),
    (dict(scale=float("nan")), 1),
    (dict(scale=0.0), 1),           # the scale must be > 0
    (dict(scale=-0.5), 1),
])
def test_rejects_bad_problems(L, kw, code):
    rc, msg = fwd_status(L, problem(L, **kw))
    assert rc == code and msg


def test_rejects_bad_cu_seqlens(L):
    for cu in ([0, 100, 90, 256], [1, 100, 256], [0, 100, 200]):
        host = (ctypes.c_int32 * len(cu))(*cu)
        p = problem(L, cu_seqlens=0x10000, cu_seqlens_host=ctypes.addressof(host),
                    num_seqs=len(cu) - 1)
        rc, msg = fwd_status(L, p)
        assert rc == 1, (cu, rc, msg)
    p = problem(L, B=2, cu_seqlens=0x10000, cu_seqlens_host=0x10000, num_seqs=1)
    assert fwd_status(L, p)[0] == 1
    p = problem(L, cu_seqlens=0x10000)  # device copy without the host copy
    assert fwd_status(L, p)[0] == 1


def test_rejects_misaligned_and_null(L):
    fake = ctypes.c_void_p(0x10000)
    bad = ctypes.c_void_p(0x10002)
    rc, _ = fwd_status(L, problem(L), [bad] + [fake] * 4 + [None, fake, fake, fake])
    assert rc == 1
    rc, _ = fwd_status(L, problem(L), [None] + [fake] * 4 + [None, fake, fake, fake])
    assert rc == 1


def test_workspace_size_and_too_small_workspace(L):
    p = problem(L, T=32768, Hqk=2, Hv=8, cp_mode=L.CP_EXACT, cp_segment_chunks=16)
    n = ctypes.c_size_t(0)
    assert L.lib().gdn_chunk_fwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == 0
    # 32 segments x 8 heads x (entering state + transition) of 64 KiB each, plus the plan
    assert n.value >= 2 * 32 * 8 * 128 * 128 * 4
    rc, msg = fwd_status(L, p, ws_bytes=n.value - 1)
    assert rc == 3 and "workspace" in msg
    # no context parallelism: the plan arrays, plus (bf16 tensor-core path) the TW, TU, P
    # tiles of every (chunk, v-head): 3 x 8 KiB each
    p2 = problem(L, T=32768, Hqk=2, Hv=8, cp_mode=L.CP_OFF, dtype=1)
    assert L.lib().gdn_chunk_fwd_workspace_size(ctypes.byref(p2), ctypes.byref(n)) == 0
    assert n.value < 4096
    p3 = problem(L, T=32768, Hqk=2, Hv=8, cp_mode=L.CP_OFF, dtype=0)
    assert L.lib().gdn_chunk_fwd_workspace_size(ctypes.byref(p3), ctypes.byref(n)) == 0
    assert 512 * 8 * 32768 <= n.value < 512 * 8 * 32768 + 4096


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from chunked_prefill_gb300 import gdn
    monkeypatch.setattr(gdn, "_lib", None)
    monkeypatch.setattr(gdn, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        gdn.lib()


def test_device_status_rejects_bad_arguments(L):
    """The failure-report entry points validate on the host and launch nothing."""
    lib = L.lib()
    assert lib.gdn_device_status(None, None) == L.GDN_ERR_INVALID_ARG
    assert lib.gdn_device_status(ctypes.c_void_p(0x1008), None) == L.GDN_ERR_INVALID_ARG  # misaligned
    assert lib.gdn_debug_wait_timeout(None, 1000, None) == L.GDN_ERR_INVALID_ARG
    assert lib.gdn_debug_wait_timeout(ctypes.c_void_p(0x1000), 0, None) == L.GDN_ERR_INVALID_ARG
    assert lib.gdn_debug_wait_timeout(ctypes.c_void_p(0x1000), 2000000, None) == L.GDN_ERR_INVALID_ARG
    lib.gdn_noalloc_debug_wait_timeout.argtypes = [ctypes.c_int32, ctypes.c_void_p]
    assert lib.gdn_noalloc_debug_wait_timeout(0, None) == L.GDN_ERR_INVALID_ARG


def test_status_codes_match_the_header(L):
    """Every GDN_* status value the header's enum declares has the same value in the binding."""
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    codes = dict((n, int(v)) for n, v in re.findall(r"\b(GDN_(?:OK|ERR_\w+))\s*=\s*(\d+)", src))
    assert {"GDN_OK", "GDN_ERR_TIMEOUT", "GDN_ERR_BOUNDS"} <= set(codes)
    for name, value in codes.items():
        assert getattr(L, name) == value, name


# The planner's segmentation on a 152-SM GB300 for the benchmark shapes, pinned to the plans
# measured fastest there (CUDA events, same GPU, the same workload forced to each segment
# length): 1 x 32768 tokens at 8 / 24 heads took 0.351 ms with 86-chunk segments (one wave of
# scan CTAs) against 0.366 ms with 43 and 0.378 ms with 27 (two and three waves); the training
# step at 16 / 16 heads 1.409 ms with 57 (one wave) against 1.466 ms with 27 (two waves) and
# 1.436 ms with 64; at 2 / 8 heads 27-chunk segments fill the 152 SMs once (54: 0.177 against
# 0.141 ms); 16 packed sequences of 64 chunks at 4 / 16 heads ran best unsplit.
@pytest.mark.parametrize("shape, expect", [
    (dict(B=1, T=32768, Hqk=2, Hv=8), (27, 19)),
    (dict(B=1, T=32768, Hqk=8, Hv=24), (86, 6)),
    (dict(B=1, T=32768, Hqk=16, Hv=16), (57, 9)),
    (dict(B=1, T=256, Hqk=2, Hv=4), (4, 1)),
])
def test_planner_choice_on_152_sms(L, shape, expect):
    p = problem(L, cp_mode=L.CP_AUTO, **shape)
    seg_len, segs = ctypes.c_int32(0), ctypes.c_int32(0)
    assert L.lib().gdn_debug_plan(ctypes.byref(p), 152, ctypes.byref(seg_len), ctypes.byref(segs)) == 0
    assert (seg_len.value, segs.value) == expect


def test_planner_choice_packed_sequences(L):
    import torch
    cu = torch.arange(0, 16 * 4096 + 1, 4096, dtype=torch.int32)
    p = problem(L, B=1, T=16 * 4096, Hqk=4, Hv=16, cp_mode=L.CP_AUTO, num_seqs=16,
                cu_seqlens=0x10000, cu_seqlens_host=cu.data_ptr())
    seg_len, segs = ctypes.c_int32(0), ctypes.c_int32(0)
    assert L.lib().gdn_debug_plan(ctypes.byref(p), 152, ctypes.byref(seg_len), ctypes.byref(segs)) == 0
    assert (seg_len.value, segs.value) == (64, 16)
    # the binding's wrapper, and the hook's argument checks
    q = torch.empty(1, 32768, 16, 128, dtype=torch.bfloat16)
    assert L.gdn_debug_plan(L.Problem(q, q, 128 ** -0.5), 152) == (57, 9)
    assert L.lib().gdn_debug_plan(ctypes.byref(p), 0, ctypes.byref(seg_len), ctypes.byref(segs)) == 1
