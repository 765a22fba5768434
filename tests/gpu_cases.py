"""Shared helpers of the GPU parity tests: seeded inputs on the device, their
exact bf16 bits for the oracle, and the output tolerance.

Output tolerance (bf16 outputs against the fp64 oracle), per token batch:
    max |out - ref| <= 2e-2 * rms(ref)   and   mean|out - ref| / mean|ref| <= 5e-3
where rms(ref) = sqrt(mean(ref^2)) over every compared element.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from sparse_moe_ffn_gb300 import binding
from sparse_moe_ffn_gb300.inputs import CONFIGS, MoEShape, make_inputs, to_device

MAX_ERR_OF_RMS = 2e-2
MEAN_REL_ERR = 5e-3
# fp32 routing weights against fp64: the logits accumulate H bf16 products in
# fp32 (error ~ sqrt(H) * 2^-24 * |partial sums|), softmax adds a few ulp.
WEIGHT_ATOL = 2e-5


@functools.lru_cache(maxsize=5)
def prepared(name: str, seed: int = 0):
    """(shape, device tensors, oracle bit arrays) of a named configuration."""
    return prepare(CONFIGS[name], seed)


def prepare(shape: MoEShape, seed: int = 0):
    cpu = make_inputs(shape, seed)
    dev = to_device(cpu, "cuda")
    if shape.cast_on_gpu:
        bits = {n: oracle.bf16_bits(t) for n, t in dev.items()}  # the GPU's cast
    else:
        bits = {n: oracle.bf16_bits(t) for n, t in cpu.items()}
    # the oracle takes the model's bf16 weights; the library its fp16 down weights
    return shape, binding.prepare_weights(dev), bits


def shared_of(shape, dev):
    return {n: dev[n] for n in binding.SHARED_KEYS} if shape.I_s else None


def run_forward(shape, dev, x=None, workspace=None):
    x = dev["x"] if x is None else x
    N = x.shape[0]
    if workspace is None:
        workspace = binding.alloc_workspace(N, shape.H, shape.E, shape.I, shape.k, shape.I_s)
    out = binding.moe_forward(x, dev["router"], dev["w_gate"], dev["w_up"], dev["w_down"],
                              shape.k, shape.norm_topk_prob, shared_of(shape, dev),
                              workspace=workspace)
    status = binding.moe_read_device_status(workspace)
    assert status == 0, f"device status {status}: {binding.moe_status_string(status)}"
    return out, workspace


def error_stats(out, ref):
    got = out.float().cpu().numpy().astype(np.float64) if torch.is_tensor(out) else out
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return float(err.max()), rms, float(err.mean() / np.abs(ref).mean())


def assert_close(out, ref, what=""):
    mx, rms, mean_rel = error_stats(out, ref)
    assert mx <= MAX_ERR_OF_RMS * rms and mean_rel <= MEAN_REL_ERR, (
        f"{what}: max|err| {mx:.3e} vs {MAX_ERR_OF_RMS} * rms {rms:.3e}; "
        f"mean rel err {mean_rel:.3e} vs {MEAN_REL_ERR}")


def sample_rows(N: int, n: int, seed: int = 0) -> np.ndarray:
    """First, last and n-2 random rows (sorted, unique)."""
    if N <= n:
        return np.arange(N, dtype=np.int64)
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(N, size=n - 2, replace=False).tolist()) | {0, N - 1}
    return np.array(sorted(rows), dtype=np.int64)
