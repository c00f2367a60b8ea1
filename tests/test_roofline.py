"""The benchmark's roofline arithmetic on the host: the compulsory bytes of a step counted
from the tensors' sizes (bf16 activations, fp32 gates and states), independently of
chunked_prefill_gb300.roofline and bench.method_bytes, which must agree with them."""
import pytest

import bench
from chunked_prefill_gb300 import roofline as rl
from chunked_prefill_gb300.inputs import WORKLOADS


def by_hand(T, N, Hqk, Hv, h0, backward):
    act_qk, act_v = T * Hqk * 128 * 2, T * Hv * 128 * 2     # one bf16 [T, H, 128] tensor
    gate, state = T * Hv * 4, N * Hv * 128 * 128 * 4         # one fp32 gate, one fp32 state
    fwd = 2 * act_qk + act_v + 2 * gate + act_v + state * (int(h0) + 1)   # q k v g b in; o ht out
    if not backward:
        return fwd
    # the backward call: q k v dO g b (h0, dht) in; dq dk dv dg db (dh0) out
    bwd = 2 * act_qk + 2 * act_v + 2 * gate + 2 * act_qk + act_v + 2 * gate + state * (2 * int(h0) + 1)
    return fwd + bwd


def test_forward_step_bytes_of_the_benchmark_workload():
    # 1 x 32768 tokens, 2 / 8 heads, no initial state: 170.39 MB
    assert by_hand(32768, 1, 2, 8, False, False) == 170_393_600
    assert rl.fwd_bytes(32768, 1, 2, 8, h0=False) == 170_393_600
    w = WORKLOADS["fwd_t32k_hqk2_hv8"]
    mb = bench.method_bytes(32768, [32768], w)
    assert sum(mb[n] for n in bench.step_tensors(False)) == 170_393_600
    # the preparation's method tensors: q, k, g, beta
    assert bench.kernel_bytes("fwd_prep", mb)[0] == 2 * 32768 * 2 * 128 * 2 + 2 * 32768 * 8 * 4


def test_training_step_bytes_count_each_call():
    # 1 x 32768 tokens, 16 / 16 heads, h0 and dht: the forward call 543.16 MB, the backward
    # call 951.06 MB (it reads the inputs again), 1494.22 MB per step
    assert by_hand(32768, 1, 16, 16, True, False) == 543_162_368
    assert by_hand(32768, 1, 16, 16, True, True) == 1_494_220_800
    assert rl.fwd_bytes(32768, 1, 16, 16, h0=True) + rl.bwd_bytes(32768, 1, 16, 16, h0=True) == 1_494_220_800


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_every_workload_matches_the_hand_count(name):
    w = WORKLOADS[name]
    lens = [w.T] * w.B if not w.varlen_seqs else None
    if lens is None:
        pytest.skip("packed lengths are drawn by the input generator")
    T = w.B * w.T
    got = rl.fwd_bytes(T, len(lens), w.Hqk, w.Hv, h0=w.h0_std > 0)
    if w.backward:
        got += rl.bwd_bytes(T, len(lens), w.Hqk, w.Hv, h0=w.h0_std > 0)
    assert got == by_hand(T, len(lens), w.Hqk, w.Hv, w.h0_std > 0, w.backward)
