"""GPU parity at the DeepSeek-V3 shape (H=7168, E=256, K=8, I=I_shared=2048) in the launch
configuration the benchmark times: routing, counts and affinity bit-exact over every token,
Y on sampled tokens that the oracle evaluates one by one."""
import numpy as np
import pytest

from expert_routed_ffn_router_gb300 import synth

from gpu_common import DEV, Problem, check_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv3_weights():
    w = synth.workload("decode")
    return synth.expert_weights_device(w, DEV)


def _sample(T, n):
    return sorted({0, T - 1, *np.linspace(0, T - 1, n).astype(int).tolist()})


def test_decode_T128(dsv3_weights):
    w = synth.workload("decode")
    check_layer(Problem(w, weights_dev=dsv3_weights), tokens=_sample(w.T, 4))


@pytest.mark.parametrize("T", [2, 64])
def test_batch_sweep(dsv3_weights, T):
    w = synth.workload(f"sweep{T}")
    r = check_layer(Problem(w, weights_dev=dsv3_weights),
                    tokens=None if T <= 2 else _sample(T, 3))
    n_act = int((r["disp"]["counts"] > 0).sum())
    assert n_act <= min(w.E, T * w.K)


def test_prefill_T16384(dsv3_weights):
    w = synth.workload("prefill")
    check_layer(Problem(w, weights_dev=dsv3_weights), tokens=_sample(w.T, 2))


def test_skewed_T8192(dsv3_weights):
    w = synth.workload("skewed")
    r = check_layer(Problem(w, weights_dev=dsv3_weights), tokens=_sample(w.T, 2))
    assert r["disp"]["counts"].max() >= 0.95 * w.T  # the most popular experts: nearly every token
