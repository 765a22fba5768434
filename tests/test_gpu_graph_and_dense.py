"""The layer captured in a CUDA graph and replayed for bucketed batches, and
the dense SwiGLU MLP entry point, against eager calls and the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import FORMS, assert_close, prepare, prepared
from sparse_moe_ffn_gb300 import binding
from sparse_moe_ffn_gb300.inputs import MoEShape, make_inputs, make_tokens

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


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("name", ["decode", "talker"])
def test_forward_host_buffers_match_device_call(name, form):
    """moe_forward_host (pinned host x in, pinned host out) equals the device
    call bit for bit."""
    shape, dev, _ = prepared(name, form=form)
    weights = {n: t for n, t in dev.items() if n != "x"}
    x_host = dev["x"].cpu().pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    x_dev, out_dev = torch.empty_like(dev["x"]), torch.empty_like(dev["x"])
    ws = binding.alloc_workspace(shape.N, shape.H, shape.E, shape.I, shape.k, shape.I_s)
    binding.moe_forward_from_host(x_host, out_host, x_dev, out_dev, weights, shape.k,
                                  shape.norm_topk_prob, ws)
    torch.cuda.synchronize()
    assert binding.moe_read_device_status(ws) == 0
    assert torch.equal(out_host, _eager(shape, dev, dev["x"]).cpu())


@pytest.mark.parametrize("form", FORMS)
def test_graph_set_decode_loop_matches_oracle(form):
    """A multi-step decode loop under CUDA-graph replay: ten steps whose batch
    sizes change from step to step (buckets 1, 4, 8, 32, 64 and 128 among
    the captured 1, 2, 4, ... 128), each with fresh activations, every step's
    output against the oracle over all its tokens and against an eager call
    bit for bit."""
    shape, dev, bits = prepared("decode", form=form)
    weights = {n: t for n, t in dev.items() if n != "x"}
    graphs = binding.ForwardGraphSet(weights, shape.k, shape.norm_topk_prob)
    assert graphs.buckets == (1, 2, 4, 8, 16, 32, 64, 128)
    sizes = [1, 3, 64, 8, 27, 128, 5, 64, 33, 2]
    steps = [make_tokens(shape, dev["router"], n, seed=100 + i).cuda()
             for i, n in enumerate(sizes)]
    outs = binding.decode_loop(graphs, steps)
    used = {graphs.bucket_of(n) for n in sizes}
    assert len(used) >= 5, used
    for i, (x, out) in enumerate(zip(steps, outs)):
        assert out.shape == x.shape
        step_bits = dict(bits, x=oracle.bf16_bits(x))
        ref = oracle.moe_forward(step_bits, shape.k, shape.norm_topk_prob)
        assert_close(out, ref, f"step {i} (n={x.shape[0]}, {form})")
        assert torch.equal(out, _eager(shape, dev, x)), f"step {i}"


def test_graph_bucket_padding_is_exact():
    shape, dev, _ = prepared("decode")
    weights = {n: t for n, t in dev.items() if n != "x"}
    g = binding.ForwardGraph(weights, shape.k, shape.norm_topk_prob, bucket=64)
    x = dev["x"][:37].contiguous()
    assert torch.equal(g(x), _eager(shape, dev, x))


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("N,H,I", [(300, 256, 192), (1, 128, 64), (129, 64, 200), (2048, 2048, 768)])
def test_dense_mlp_matches_oracle(N, H, I, form):
    shape, dev, bits = prepare(MoEShape("dense", N=N, H=H, E=1, k=1, I=I), seed=5, form=form)
    out = binding.moe_dense_mlp(dev["x"], dev["w_gate"][0], dev["w_up"][0], dev["w_down"][0])
    ref = oracle.moe_forward(bits, 1, True)  # E = k = 1: the dense MLP
    assert_close(out, ref, f"dense N={N} ({form})")
    # and it agrees with the layer's own E = k = 1 path bit for bit
    assert torch.equal(out, _eager(shape, dev, dev["x"]))


@pytest.mark.parametrize("N,H,gemma", [(64, 2048, False), (8192, 2048, False), (37, 200, True),
                                       (1, 64, False)])
def test_add_rmsnorm_matches_oracle(N, H, gemma):
    rng = np.random.default_rng(N + H)
    x = torch.from_numpy(rng.standard_normal((N, H)).astype(np.float32)).to(torch.bfloat16)
    res = torch.from_numpy((3 * rng.standard_normal((N, H))).astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy((1 + 0.1 * rng.standard_normal(H)).astype(np.float32)).to(torch.bfloat16)
    r_ref, n_ref = oracle.add_rmsnorm(oracle.bf16_bits(x), oracle.bf16_bits(res),
                                      oracle.bf16_bits(w), 1e-6, gemma)
    res_d = res.cuda()
    normed = binding.moe_add_rmsnorm(x.cuda(), res_d, w.cuda(), 1e-6, gemma)
    assert np.array_equal(oracle.bf16_bits(res_d), r_ref)   # the new residual, bit for bit
    got = normed.float().cpu().numpy().astype(np.float64)
    # one bf16 rounding (half an ulp is 2^-9 relative) plus the fp32 sum of squares
    assert np.all(np.abs(got - n_ref) <= 2.0 ** -8 * np.abs(n_ref) + 1e-30)
