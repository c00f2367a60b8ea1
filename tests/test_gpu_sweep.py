"""GPU parity of the forward at points of the head / length sweep (inputs.SWEEP): the full
problem runs on the GPU, the fp64 oracle checks the outputs of the first and the last q/k
group (all their v-heads), which is a complete sub-problem of its own."""
import copy

import numpy as np
import pytest
import torch

from chunked_prefill_gb300.inputs import workload_inputs
from tests.gpu_util import BF16_TOL, gpu_fwd, oracle_fwd, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_prefill_gb300 import build
    build.build()


@pytest.mark.parametrize("name", ["sweep_b4_t8k_hqk16_hv64", "sweep_b1_t8k_hqk16_hv64", "sweep_b1_t32k_hqk8_hv24",
                                  "sweep_b1_t8k_hqk2_hv8"])
def test_sweep_point_sampled_groups(name):
    inp = workload_inputs(name)
    o, ht = gpu_fwd(inp)
    Hqk, Hv = inp.q.shape[2], inp.v.shape[2]
    G = Hv // Hqk
    groups = sorted({0, Hqk - 1})
    vh = [j for g in groups for j in range(g * G, (g + 1) * G)]
    sub = copy.copy(inp)
    sub.q, sub.k = inp.q[:, :, groups].contiguous(), inp.k[:, :, groups].contiguous()
    sub.v = inp.v[:, :, vh].contiguous()
    sub.g, sub.beta = inp.g[:, :, vh].contiguous(), inp.beta[:, :, vh].contiguous()
    sub.h0 = None if inp.h0 is None else inp.h0[:, vh].contiguous()
    ro, rht = oracle_fwd(sub)
    got_o = np.take(o, vh, axis=2)
    got_ht = np.take(ht, vh, axis=1)
    assert rel_err(got_o.reshape(ro.shape), ro) <= BF16_TOL
    assert rel_err(got_ht.reshape(rht.shape), rht) <= BF16_TOL
