"""FP8 experts on the GPU against the oracle ("Lower latency and higher throughput with
multi-node DeepSeek deployment", Quantization: E4M3 with 128 x 128 weight-tile scales and
1 x 128 activation-vector scales).  Weight and activation quantisation bit-exact; the layer's
routing bit-exact and Y within the stated tolerances of the oracle's FP8 layer."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8
from expert_routed_ffn_router_gb300 import binding as B
from expert_routed_ffn_router_gb300 import synth

from gpu_common import (DEV, W_MAX_ABS, Y_MAX_ABS, Y_REL_FROB, Problem, bits, check_dispatch,
                        host_to_device_bf16, rel_frob)

pytestmark = pytest.mark.gpu


def _e4m3_bytes_to_values(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.float8_e4m3fn).double().numpy()


def _bf16_values(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits_to_f32(bits(t)).astype(np.float64)


def test_weight_quantisation_is_bit_exact():
    rng = np.random.default_rng(0)
    W = rng.standard_normal((3, 256, 384)).astype(np.float32) * 0.02
    W[0, :128, :128] *= 1e4            # large tile
    W[1, 128:, 128:256] = 0.0          # all-zero tile: k = 0
    W[2, :128, 256:] *= 1e-30          # tiny values: the clamped exponent
    W[2, 5, 300] = 448.0 * 2.0 ** -20  # a tile whose maximum sits exactly on 448 * 2^k
    Wb = synth.f32_to_bf16_bits(W)
    Wq, S = B.moe_quantize_weight_fp8(host_to_device_bf16(Wb))
    torch.cuda.synchronize()
    q_ref, k_ref = ofp8.quantize_weight(synth.bf16_bits_to_f32(Wb).astype(np.float64))
    assert np.array_equal(S.cpu().numpy().astype(np.int64), k_ref)
    # the bytes are stored transposed ([G, C, R]: K-major rows for the FP8 tensor-core MMA)
    assert tuple(Wq.shape) == (3, 384, 256)
    np.testing.assert_array_equal(_e4m3_bytes_to_values(Wq), np.swapaxes(q_ref, -1, -2))


@pytest.mark.parametrize("rows,n", [(1, 128), (37, 512), (300, 7168)])
def test_row_quantisation_is_bit_exact(rows, n):
    rng = np.random.default_rng(rows + n)
    x = rng.standard_normal((rows, n)).astype(np.float32) * np.exp(rng.uniform(-10, 6, (rows, 1)))
    x[0, :128] = 0.0
    xb = synth.f32_to_bf16_bits(x.astype(np.float32))
    out = B.moe_quantize_rows_fp8(host_to_device_bf16(xb))
    torch.cuda.synchronize()
    ref = ofp8.fake_quant_rows(synth.bf16_bits_to_f32(xb).astype(np.float64))
    np.testing.assert_array_equal(_bf16_values(out), ref)


def _oracle_Y_fp8(p: Problem, idx, wts, tokens):
    """Y[t] = sum_j w_tj FFN8_{e_tj}(x_t) + FFN8_shared(x_t) on the oracle's quantisation."""
    X = synth.bf16_bits_to_f32(p.routing["X"]).astype(np.float64)
    deq = {}

    def expert(name, e=None):
        key = (name, e)
        if key not in deq:
            w = synth.bf16_bits_to_f32(p.expert_host(name, e)).astype(np.float64)
            deq[key] = ofp8.dequantize_weight(*ofp8.quantize_weight(w))
        return deq[key]

    Y = np.zeros((len(tokens), p.w.H))
    for qi, t in enumerate(tokens):
        x = X[t:t + 1]
        for j in range(p.w.K):
            e = int(idx[t, j])
            Y[qi] += wts[t, j] * ofp8.expert_rows_fp8(x, expert("W1", e), expert("W3", e),
                                                       expert("W2", e))[0]
        if p.w.Is > 0:
            Y[qi] += ofp8.expert_rows_fp8(x, expert("W1s"), expert("W3s"), expert("W2s"))[0]
    return Y


def check_layer_fp8(p: Problem, tokens=None):
    layer = B.MoELayer(p.dev, p.w.T, p.w.K, routing=p.opts, fp8=True)
    layer.forward(p.X)
    torch.cuda.synchronize()
    assert layer.status() == 0
    idx_o, w_o = p.oracle_routing()
    assert np.array_equal(layer.topk_idx.cpu().numpy(), idx_o)
    assert np.abs(layer.topk_w.cpu().numpy().astype(np.float64) - w_o).max() <= W_MAX_ABS
    d = oracle.dispatch(idx_o, p.w.E)
    assert np.array_equal(layer.counts.cpu().numpy(), d["counts"])
    assert np.array_equal(layer.affinity.cpu().numpy(), d["affinity"])
    check_dispatch(layer, p.X, d)     # offsets, perm, slot_pos and Xp = X[perm], bit-exact
    tokens = np.arange(p.w.T) if tokens is None else np.asarray(tokens)
    Y_o = _oracle_Y_fp8(p, idx_o, w_o, tokens)
    Y_g = layer.Y.cpu().numpy()[tokens].astype(np.float64)
    rf, ma = rel_frob(Y_g, Y_o), float(np.abs(Y_g - Y_o).max())
    assert rf <= Y_REL_FROB and ma <= Y_MAX_ABS, (rf, ma)
    return rf, ma


@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("T,H,E,K,I,Is", [
    (3, 256, 16, 2, 128, 128),        # one valid row per tile
    (45, 256, 16, 2, 128, 128),
    (300, 384, 40, 5, 256, 128),      # H % 256 == 128: pair tiles past the last column
    (513, 256, 8, 6, 128, 0),         # 256-row token tiles, no shared expert
])
def test_fp8_layer_matches_the_oracle(T, H, E, K, I, Is, variant):
    w = synth.Workload("f8", T=T, H=H, E=E, K=K, I=I, Is=Is, seed=T + 3, x_seed=T + 4)
    B.moe_debug_set_ffn_variant(variant)
    try:
        check_layer_fp8(Problem(w))
    finally:
        B.moe_debug_set_ffn_variant(0)


def test_fp8_weights_with_subnormal_codes():
    # every 128 x 128 tile of the up projections holds one large weight, in a row that meets
    # a zero column of X, and otherwise values that quantise to E4M3 subnormals (below 2^-6
    # of the tile scale): the whole up projection comes from subnormal codes, which the
    # weight path must keep exactly
    w = synth.Workload("f8sub", T=40, H=256, E=8, K=2, I=128, Is=128, seed=41, x_seed=42)
    r = synth.routing_inputs(w)
    r["X"][:, 0] = 0
    r["X"][:, 128] = 0
    p = Problem(w, routing=r)
    rng = np.random.default_rng(43)
    for name in ("W1", "W3", "W1s", "W3s"):
        shape = p.host_w[name].shape
        v = rng.uniform(-1, 1, shape) * 2.0 ** -16          # tile scale 2^-10: codes m * 2^-9
        v[..., ::128, ::128] = 0.4                           # 0.4 = 409.6 * 2^-10
        b = synth.f32_to_bf16_bits(v.astype(np.float32))
        p.host_w[name] = b
        p.dev[name] = host_to_device_bf16(b)
    q, k = ofp8.quantize_weight(synth.bf16_bits_to_f32(p.host_w["W1"]).astype(np.float64))
    sub = (np.abs(q) < 2.0 ** -6) & (q != 0)
    assert np.all(k == -10) and sub.mean() > 0.8
    check_layer_fp8(p)


def test_fp8_layer_with_grouped_routing():
    w = synth.Workload("f8r", T=150, H=256, E=32, K=4, I=128, Is=128, seed=31, x_seed=32)
    check_layer_fp8(Problem(w, opts=dict(scoring="sigmoid", n_group=4, topk_group=2, group_top=2)))


def test_fp8_layer_dsv3_two_tokens():
    # DeepSeek-V3 shape, 2 tokens (16 routed experts + the shared expert), every token
    w = synth.workload("sweep2")
    check_layer_fp8(Problem(w, host_weights=False))


def test_fp8_layer_dsv3_decode():
    # DeepSeek-V3 decode step (128 tokens, 32-row FP8 token tiles, 256-row weight tiles):
    # routing, counts and affinity bit-exact over every token; Y on four tokens spread over
    # the batch (the oracle quantises each of their ~30 experts' weights in numpy)
    w = synth.workload("decode")
    check_layer_fp8(Problem(w, host_weights=False), tokens=[0, 37, 77, 127])


def test_fp8_layer_is_deterministic_and_graph_capturable():
    # the FP8 layer (router, dispatch, row and h quantisation, the up and down launches,
    # combine: ten launches) captured in a CUDA graph and replayed on new activations gives
    # what an ordinary call on them gives, bit for bit; two ordinary calls agree too
    w = synth.Workload("f8g", T=70, H=256, E=16, K=4, I=128, Is=128, seed=61, x_seed=62)
    p = Problem(w)
    layer = B.MoELayer(p.dev, w.T, w.K, fp8=True)
    layer.forward(p.X)
    torch.cuda.synchronize()
    y1 = layer.Y.clone()
    layer.forward(p.X)
    torch.cuda.synchronize()
    assert torch.equal(y1, layer.Y)
    s = torch.cuda.Stream()
    X2 = p.X.clone()
    with torch.cuda.stream(s):
        layer.forward(X2, stream=s)            # warm-up on the capture stream
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            layer.forward(X2, stream=s)
    torch.cuda.synchronize()
    Xn = host_to_device_bf16(synth.f32_to_bf16_bits(
        np.random.default_rng(63).standard_normal((w.T, w.H)).astype(np.float32)))
    X2.copy_(Xn)
    g.replay()
    torch.cuda.synchronize()
    y_graph = layer.Y.clone()
    layer.forward(Xn)
    torch.cuda.synchronize()
    assert torch.equal(y_graph, layer.Y)
    assert layer.status() == 0


def test_fp8_rejects_shapes_off_the_128_grid():
    w = synth.Workload("f8bad", T=8, H=192, E=8, K=2, I=128, Is=0, seed=1, x_seed=2)
    p = Problem(w)
    with pytest.raises(B.MoeError) as ei:
        B.MoELayer(p.dev, w.T, w.K, fp8=True)
    assert ei.value.status == -2
