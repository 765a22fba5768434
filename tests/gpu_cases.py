"""Shared helpers of the GPU parity tests: seeded inputs on the device, their
exact bf16 bits for the oracle, the oracle's full outputs (computed once per
configuration), and the output tolerance.

Output tolerance (bf16 outputs against the fp64 oracle), per token batch:
    max |out - ref| <= 2e-2 * rms(ref)   and   mean|out - ref| / mean|ref| <= 5e-3
where rms(ref) = sqrt(mean(ref^2)) over every compared element.

The layer runs with the model's bf16 down weights ("bf16": moe_forward, hi/lo
activation) or with their fp16 copies ("f16": moe_forward_prepared); FORMS
lists both, and the tests that hold for either run for both.
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


FORMS = ("bf16", "f16")
ALL = ("tiny", "decode", "prefill", "talker", "skewed")


@functools.lru_cache(maxsize=16)
def prepared(name: str, seed: int = 0, form: str = "bf16"):
    """(shape, device tensors, oracle bit arrays) of a named configuration;
    form "f16" gives the down projections as their fp16 copies."""
    shape, dev, bits = _prepared_bf16(name, seed)
    return shape, with_form(dev, form), bits


@functools.lru_cache(maxsize=5)
def _prepared_bf16(name: str, seed: int):
    return prepare(CONFIGS[name], seed)


def prepare(shape: MoEShape, seed: int = 0, form: str = "bf16"):
    cpu = make_inputs(shape, seed)
    dev = to_device(cpu, "cuda")
    if shape.cast_on_gpu:
        bits = {n: oracle.bf16_bits(t) for n, t in dev.items()}  # the GPU's cast
    else:
        bits = {n: oracle.bf16_bits(t) for n, t in cpu.items()}
    # the oracle takes the model's bf16 weights, as does moe_forward
    return shape, with_form(dev, form), bits


def with_form(dev: dict, form: str) -> dict:
    """The device tensors with the down projections in the given form."""
    if form == "bf16":
        return dev
    if form == "f16":
        return binding.prepare_weights(dev)
    raise ValueError(form)


@functools.lru_cache(maxsize=5)
def oracle_outputs(name: str, seed: int = 0) -> np.ndarray:
    """The oracle's output for every token of a named configuration (fp64)."""
    shape, _, bits = _prepared_bf16(name, seed)
    return oracle.moe_forward(bits, shape.k, shape.norm_topk_prob)


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


def decode_pair_rows(y) -> np.ndarray:
    """The values held by pair rows (hi bf16, res int8), as moe.h defines the
    format: v = hi + res * 2^(f - 142), f = max(16, exponent field of hi)."""
    hi = y[0].float().cpu()
    res = y[1].cpu().to(torch.float64)
    f = ((hi.view(torch.int32) >> 23) & 0xFF).clamp(min=16).to(torch.float64)
    return (hi.double() + res * torch.pow(2.0, f - 142)).numpy()


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
