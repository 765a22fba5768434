"""The layer captured in a CUDA graph and replayed for bucketed batches, and
the dense SwiGLU MLP entry point, against eager calls and the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import assert_close, prepare, prepared
from sparse_moe_ffn_gb300 import binding
from sparse_moe_ffn_gb300.inputs import MoEShape, make_inputs

pytestmark = pytest.mark.gpu


def _eager(shape, dev, x):
    shared = {n: dev[n] for n in binding.SHARED_KEYS} if shape.I_s else None
    return binding.moe_forward(x, dev["router"], dev["w_gate"], dev["w_up"], dev["w_down"],
                               shape.k, shape.norm_topk_prob, shared)


@pytest.mark.parametrize("name", ["decode", "talker"])
def test_graph_replay_matches_eager(name):
    shape, dev, _ = prepared(name)
    weights = {n: t for n, t in dev.items() if n != "x"}
    g = binding.ForwardGraph(weights, shape.k, shape.norm_topk_prob, bucket=shape.N)
    for seed in (11, 12, 13):  # fresh activations into the captured buffers
        x = make_inputs(shape.with_tokens(shape.N), seed=seed)["x"].cuda()
        got = g(x).clone()
        assert torch.equal(got, _eager(shape, dev, x)), f"seed {seed}"


def test_graph_bucket_padding_is_exact():
    shape, dev, _ = prepared("decode")
    weights = {n: t for n, t in dev.items() if n != "x"}
    g = binding.ForwardGraph(weights, shape.k, shape.norm_topk_prob, bucket=64)
    x = dev["x"][:37].contiguous()
    assert torch.equal(g(x), _eager(shape, dev, x))


@pytest.mark.parametrize("N,H,I", [(300, 256, 192), (1, 128, 64), (129, 64, 200), (2048, 2048, 768)])
def test_dense_mlp_matches_oracle(N, H, I):
    shape, dev, bits = prepare(MoEShape("dense", N=N, H=H, E=1, k=1, I=I), seed=5)
    out = binding.moe_dense_mlp(dev["x"], dev["w_gate"][0], dev["w_up"][0], dev["w_down"][0])
    rows = np.arange(0, N, max(1, N // 256), dtype=np.int64)
    ref = oracle.moe_forward(bits, 1, True, rows=rows)  # E = k = 1: the dense MLP
    assert_close(out[torch.from_numpy(rows).cuda()], ref, f"dense N={N}")
    # and it agrees with the layer's own E = k = 1 path bit for bit
    assert torch.equal(out, _eager(shape, dev, dev["x"]))
