"""Device-side failure report without a GPU fault: a bounded wait that runs out (an mbarrier
that nothing completes) sets its bit in the call's error word, gdn_device_status returns
GDN_ERR_TIMEOUT, the context stays usable, and the next call clears the word."""
import numpy as np
import pytest
import torch

from chunked_prefill_gb300.inputs import make_inputs
from tests.gpu_util import BF16_TOL, oracle_fwd, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_prefill_gb300 import build
    build.build()


def test_wait_timeout_reported_then_cleared():
    from chunked_prefill_gb300 import gdn
    inp = make_inputs(1, 256, 2, 4, seed=3)
    q, k, v, g, beta = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    nbytes = gdn.gdn_chunk_fwd_workspace_size(gdn.Problem(q, v, inp.scale))
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")

    gdn.gdn_debug_wait_timeout(ws, 2000)  # gives up after 2 ms
    assert gdn.gdn_device_status(ws) == gdn.GDN_ERR_TIMEOUT
    assert "gave up" in gdn.lib().gdn_last_error().decode()

    # the context is still usable; the next call starts from a clear error word
    o, ht = gdn.gdn_chunk_fwd(q, k, v, g, beta, inp.scale, workspace=ws)
    assert gdn.gdn_device_status(ws) == gdn.GDN_OK
    ro, rht = oracle_fwd(inp)
    assert rel_err(o.float().cpu().numpy(), ro) <= BF16_TOL
    assert rel_err(ht.cpu().numpy(), rht) <= BF16_TOL
