"""Checked build (libgdn_check.so, compiled with -DGDN_CHECK): every output store of the bf16
path tests its element index against the tensor's extent and, out of range, records
GDN_ERR_BOUNDS in the call's error word instead of writing.  The edge cases below (empty and
partial sequences, a single token, grouped heads with G = 3, forced context-parallel segments,
the low-level outputs) run through that build in a child process (the library a process
loads is fixed at its first call): every call's error word must stay clear and the results
must match the fp64 oracle."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import torch
from chunked_prefill_gb300 import gdn
from chunked_prefill_gb300.inputs import make_inputs
from tests.gpu_util import BF16_TOL, oracle_bwd, oracle_fwd, rel_err, to_dev

assert gdn.LIB_PATH.endswith("libgdn_check.so"), gdn.LIB_PATH
cases = [
    (dict(B=1, T=276, Hqk=2, Hv=4, lengths=[0, 5, 64, 130, 0, 77]), {}),
    (dict(B=2, T=64 * 3 + 17, Hqk=1, Hv=3), {}),
    (dict(B=1, T=1, Hqk=1, Hv=1), {}),
    (dict(B=1, T=64 * 9 + 5, Hqk=2, Hv=2), dict(cp_mode=2, cp_segment_chunks=2)),
]
for n, (shape, kw) in enumerate(cases):
    inp = make_inputs(shape["B"], shape["T"], shape["Hqk"], shape["Hv"], seed=70 + n,
                      h0_std=0.1, lengths=shape.get("lengths"), backward=True)
    d = to_dev(inp)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], inp.scale)
    prob = gdn.Problem(d["q"], d["v"], inp.scale, d["cu"], inp.cu_seqlens, **kw)
    ws = torch.zeros(gdn.gdn_chunk_bwd_workspace_size(prob), dtype=torch.uint8, device="cuda")
    o, ht = gdn.gdn_chunk_fwd(*args, h0=d["h0"], cu_seqlens=d["cu"],
                              cu_seqlens_host=inp.cu_seqlens, workspace=ws, **kw)
    assert gdn.gdn_device_status(ws) == gdn.GDN_OK, (n, "fwd", gdn.lib().gdn_last_error())
    ro, rht = oracle_fwd(inp)
    assert rel_err(o.float().cpu().numpy(), ro) <= BF16_TOL, (n, "o")
    assert rel_err(ht.cpu().numpy(), rht) <= BF16_TOL, (n, "ht")
    got = gdn.gdn_chunk_bwd(*args, d["dO"], h0=d["h0"], dht=d["dht"], cu_seqlens=d["cu"],
                            cu_seqlens_host=inp.cu_seqlens, workspace=ws, **kw)
    assert gdn.gdn_device_status(ws) == gdn.GDN_OK, (n, "bwd", gdn.lib().gdn_last_error())
    for name, a, r in zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), got, oracle_bwd(inp)):
        assert rel_err(a.float().cpu().numpy().reshape(r.shape), r) <= BF16_TOL, (n, name)
    g_cum, A, o2, h, ht2, ctx = gdn.gdn_chunk_fwd_saved(*args, h0=d["h0"], cu_seqlens=d["cu"],
                                                        cu_seqlens_host=inp.cu_seqlens, **kw)
    assert gdn.gdn_device_status(ctx) == gdn.GDN_OK, (n, "saved", gdn.lib().gdn_last_error())
    assert torch.equal(o2, o), (n, "saved o")
print("CHECKED OK")
'''


@pytest.fixture(scope="module")
def checked_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_prefill_gb300 import build
    return build.build(checked=True)


def test_checked_build_stores_stay_in_range(checked_lib):
    env = dict(os.environ, GDN_LIB=checked_lib)
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0 and "CHECKED OK" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
