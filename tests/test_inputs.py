"""Seeded input generators: determinism, the near-tie filter and the skewed
routing construction, checked through the oracle (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
from sparse_moe_ffn_gb300.inputs import (CONFIGS, DEAD_EXPERTS, HOT_EXPERTS, MARGIN,
                                         MoEShape, make_inputs)


def _bits(t):
    return oracle.bf16_bits(t.to(torch.bfloat16))


def _min_gap(x, router, k):
    logits, _, _, _ = oracle.route(_bits(x), _bits(router), k, True)
    m = min(k + 1, logits.shape[1])
    top = -np.sort(-logits, axis=1)[:, :m]
    return (top[:, :-1] - top[:, 1:]).min()


def test_deterministic_per_seed():
    shp = MoEShape("d", N=32, H=64, E=8, k=2, I=32, I_s=16)
    a, b, c = make_inputs(shp, 1), make_inputs(shp, 1), make_inputs(shp, 2)
    for key in a:
        assert torch.equal(a[key], b[key]), key
    assert not torch.equal(a["x"], c["x"])


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_margin_filter_in_logit_space(name):
    shp = CONFIGS[name]
    w = make_inputs(shp, seed=0)
    assert _min_gap(w["x"], w["router"], shp.k) >= MARGIN


def test_tiny_is_fp32_cast_later():
    w = make_inputs(CONFIGS["tiny"], seed=0)
    assert all(t.dtype == torch.float32 for t in w.values())
    # the raw draws are not all bf16-exact: the cast really happens later
    assert not torch.equal(w["x"], w["x"].to(torch.bfloat16).float())


def test_skewed_routing_invariants():
    """8 hot experts take roughly half the pairs and >= 10 experts get none,
    at the skewed workload's N=16384, E=128, k=8 (small I: only the router matters)."""
    full = CONFIGS["skewed"]
    small_weights = MoEShape("skewed-router", N=full.N, H=full.H, E=full.E, k=full.k, I=8,
                             skew=True)
    w = make_inputs(small_weights, seed=0)
    _, _, _, ids = oracle.route(_bits(w["x"]), _bits(w["router"]), full.k, True)
    counts = np.bincount(ids.reshape(-1), minlength=full.E)
    hot_share = counts[:HOT_EXPERTS].sum() / counts.sum()
    assert 0.45 <= hot_share <= 0.70, hot_share
    assert (counts == 0).sum() >= 10
    assert np.all(counts[full.E - DEAD_EXPERTS:] == 0)


def test_prefill_router_is_near_uniform():
    shp = CONFIGS["prefill"]
    router_only = MoEShape("prefill-router", N=shp.N, H=shp.H, E=shp.E, k=shp.k, I=8)
    w = make_inputs(router_only, seed=0)
    _, _, _, ids = oracle.route(_bits(w["x"]), _bits(w["router"]), shp.k, True)
    counts = np.bincount(ids.reshape(-1), minlength=shp.E)
    mean = shp.pairs / shp.E
    assert counts.min() > 0.5 * mean and counts.max() < 1.6 * mean, (counts.min(), counts.max())


def test_make_tokens_fresh_rows_without_near_ties():
    """Fresh decode-step activations: seeded, bf16, the requested shape, and
    no near-tie among each row's k+1 largest logits against the given router."""
    from sparse_moe_ffn_gb300.inputs import MARGIN, make_tokens
    shape = CONFIGS["decode"].with_tokens(4)
    router = make_inputs(shape, seed=0)["router"]
    a = make_tokens(shape, router, 37, seed=5)
    b = make_tokens(shape, router, 37, seed=5)
    assert a.dtype == torch.bfloat16 and a.shape == (37, shape.H)
    assert torch.equal(a, b)
    assert not torch.equal(a, make_tokens(shape, router, 37, seed=6))
    top = torch.topk(a.double() @ router.double().T, shape.k + 1, dim=1).values
    assert float((top[:, :-1] - top[:, 1:]).min()) >= MARGIN
