"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Every check takes an ``oracle.Oracle`` and raises AssertionError on failure, so
the same checks run against the real oracle (tests/test_oracle_pins.py) and
against deliberately broken copies of it (tests/test_oracle_mutants.py).

Sources of truth:
  * values printed on the M03 "Sparse MoE" drill page (tests/golden/
    m03_worked_examples.json, each entry citing its section);
  * brute force: every expert evaluated on every token with dense numpy
    matmuls, then masked by the top-k weights (numpy's stable argsort picks
    the top k);
  * closed forms and special cases: E = k = 1 is a dense SwiGLU MLP computed
    with torch's silu; k = E with renormalisation gives the full softmax
    (scipy); renormalised weights equal a softmax over the top-k logits;
    unrenormalised weights sum to less than one;
  * grouping: numpy's bincount, cumsum and stable argsort.
"""
from __future__ import annotations

import json
import os

import numpy as np
import scipy.special
import torch

from oracle import widen

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "m03_worked_examples.json")
PRINT_TOL = 5e-5 + 1e-12  # the page prints 4 decimals


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def bits(a) -> np.ndarray:
    """float values -> bf16 bit patterns (round to nearest even)."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def close_printed(got, printed, what):
    got = np.asarray(got, np.float64)
    printed = np.asarray(printed, np.float64)
    assert got.shape == printed.shape, f"{what}: shape {got.shape} vs {printed.shape}"
    err = np.abs(got - printed).max() if got.size else 0.0
    assert err <= PRINT_TOL, f"{what}: {got.tolist()} vs printed {printed.tolist()}"


# ---------------------------------------------------------------------------
# printed worked examples
# ---------------------------------------------------------------------------

def check_bookkeeping(orc):
    g = golden()["bookkeeping"]
    r = orc.align(np.array(g["ids"]), g["E"], 1)
    assert r["flat_e"].tolist() == g["flat_e"], r["flat_e"]
    assert r["flat_tok"].tolist() == g["flat_tok"], r["flat_tok"]
    assert r["order"].tolist() == g["order"], f"order {r['order']}"
    assert r["counts"].tolist() == g["counts"], f"counts {r['counts']}"
    starts = r["offsets"]
    for e, pairs in enumerate(g["expert_pairs"]):
        seg = r["order"][starts[e]:starts[e + 1]].tolist()
        assert seg == pairs, f"expert {e}: pairs {seg} vs {pairs}"
        toks = [p // g["k"] for p in seg]
        assert toks == g["expert_tokens"][e], f"expert {e}: tokens {toks}"
    # each token receives contributions from exactly the experts it chose
    for n, experts in enumerate(g["token_experts"]):
        got = sorted(int(r["flat_e"][p]) for p in range(len(r["flat_e"]))
                     if r["flat_tok"][p] == n)
        assert got == experts, f"token {n}: {got}"


def check_route_io(orc):
    g = golden()["route_io"]
    x, router = bits(g["x"]), bits(g["router"])
    _, probs, w, ids = orc.route(x, router, g["k"], True)
    close_printed(probs, g["probs"], "route probs")
    assert ids.tolist() == g["ids"], f"route ids {ids.tolist()}"
    close_printed(w, g["weights_norm"], "route weights (norm)")
    _, _, w_raw, ids_raw = orc.route(x, router, g["k"], False)
    assert ids_raw.tolist() == g["ids"]
    close_printed(w_raw, g["weights_raw"], "route weights (raw)")
    close_printed(w_raw[0].sum(), g["raw_sum_token0"], "raw weight sum")


def _scalar_weights(g):
    return {
        "x": bits(g["x"]),
        "router": bits(g["router"]),
        "w_gate": bits(g["w_gate"]).reshape(g["E"], 1, 1),
        "w_up": bits(g["w_up"]).reshape(g["E"], 1, 1),
        "w_down": bits(g["w_down"]).reshape(g["E"], 1, 1),
    }


def check_scalar_e2e(orc):
    g = golden()["scalar_e2e"]
    w = _scalar_weights(g)
    logits, _, wt, ids = orc.route(w["x"], w["router"], g["k"], g["norm_topk_prob"])
    close_printed(logits, g["logits"], "scalar logits")
    assert ids.tolist() == g["ids"], f"scalar ids {ids.tolist()}"
    close_printed(wt, g["weights"], "scalar weights")
    # per-expert outputs: a one-expert layer with k = 1 and renorm is that expert
    for e in range(g["E"]):
        one = {"x": w["x"], "router": bits([[0.0]]), "w_gate": w["w_gate"][e:e + 1],
               "w_up": w["w_up"][e:e + 1], "w_down": w["w_down"][e:e + 1]}
        y = orc.moe_forward(one, 1, True)[:, 0]
        close_printed(y, [row[e] for row in g["expert_out"]], f"expert {e} output")
    out = orc.moe_forward(w, g["k"], g["norm_topk_prob"])
    close_printed(out, g["out"], "scalar moe_forward")
    assert abs(out[0, 0] - g["out_if_assigned_token0"]) > 0.1


def check_shared(orc):
    g = golden()["scalar_e2e"]
    s = golden()["shared"]
    w = _scalar_weights(g)
    for key in ("shared_gate_proj", "shared_up_proj", "shared_down_proj", "shared_gate"):
        w[key] = bits(s[key])
    out = orc.moe_forward(w, g["k"], g["norm_topk_prob"])
    close_printed(out, s["out"], "scalar moe_forward + shared")
    one = {"x": w["x"], "router": bits([[0.0]]), "w_gate": bits(s["shared_gate_proj"])[None],
           "w_up": bits(s["shared_up_proj"])[None], "w_down": bits(s["shared_down_proj"])[None]}
    close_printed(orc.moe_forward(one, 1, True)[:, 0], s["shared_expert_out"], "shared expert")


def check_shape_trace(orc):
    from sparse_moe_ffn_gb300.inputs import MoEShape, make_inputs
    g = golden()["shape_trace"]
    shp = MoEShape("trace", N=g["N"], H=g["H"], E=g["E"], k=g["k"], I=g["I"], I_s=g["I"])
    w = {n: bits_of(t) for n, t in make_inputs(shp, seed=5).items()}
    logits, probs, wt, ids = orc.route(w["x"], w["router"], g["k"], True)
    assert list(logits.shape) == g["logits"] and list(probs.shape) == g["probs"]
    assert list(wt.shape) == g["weights"] and list(ids.shape) == g["ids"]
    r = orc.align(ids, g["E"], 1)
    assert [len(r["flat_e"])] == g["flat"] and [len(r["flat_tok"])] == g["flat"]
    assert [len(r["order"])] == g["order"] and [len(r["counts"])] == g["counts"]
    assert int(r["counts"].sum()) == g["counts_sum"]
    out = orc.moe_forward(w, g["k"], True)
    assert list(out.shape) == g["out"]
    assert list((widen(w["x"]) @ widen(w["shared_gate"]).T).shape) == g["shared_gate"]


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# brute force and closed forms
# ---------------------------------------------------------------------------

def _silu(z):
    return z / (1.0 + np.exp(-z))


def brute_force(w, k, norm):
    """Every expert on every token, masked by the top-k weights (dense numpy)."""
    x = widen(w["x"])
    R = widen(w["router"])
    Wg, Wu, Wd = widen(w["w_gate"]), widen(w["w_up"]), widen(w["w_down"])
    N, E = x.shape[0], R.shape[0]
    probs = scipy.special.softmax(x @ R.T, axis=1)
    top = np.argsort(-probs, axis=1, kind="stable")[:, :k]
    rows = np.arange(N)[:, None]
    wsel = probs[rows, top]
    if norm:
        wsel = wsel / wsel.sum(axis=1, keepdims=True)
    mask = np.zeros_like(probs)
    mask[rows, top] = wsel
    Y = np.stack([(_silu(x @ Wg[e].T) * (x @ Wu[e].T)) @ Wd[e].T for e in range(E)], axis=1)
    out = np.einsum("ne,neh->nh", mask, Y)
    if "shared_gate" in w:
        gamma = scipy.special.expit(x @ widen(w["shared_gate"]).T)
        s = (_silu(x @ widen(w["shared_gate_proj"]).T) * (x @ widen(w["shared_up_proj"]).T)) \
            @ widen(w["shared_down_proj"]).T
        out = out + gamma * s
    return out, top, wsel


BRUTE_CASES = [
    # (name, N, H, E, k, I, I_s, norm)
    ("b1", 9, 16, 8, 2, 32, 0, True),
    ("b2", 7, 24, 6, 3, 16, 0, False),
    ("b3", 11, 16, 5, 2, 8, 24, False),
    ("b4", 6, 32, 4, 4, 16, 8, True),
]


def check_brute_force(orc):
    from sparse_moe_ffn_gb300.inputs import MoEShape, make_inputs
    for name, N, H, E, k, I, I_s, norm in BRUTE_CASES:
        shp = MoEShape(name, N=N, H=H, E=E, k=k, I=I, I_s=I_s, norm_topk_prob=norm)
        w = {n: bits_of(t) for n, t in make_inputs(shp, seed=11).items()}
        ref, top, wsel = brute_force(w, k, norm)
        _, _, wt, ids = orc.route(w["x"], w["router"], k, norm)
        assert np.array_equal(ids, top), f"{name}: ids {ids} vs {top}"
        np.testing.assert_allclose(wt, wsel, rtol=1e-12, atol=1e-15, err_msg=name)
        out = orc.moe_forward(w, k, norm)
        np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12, err_msg=name)


def check_closed_forms(orc):
    from sparse_moe_ffn_gb300.inputs import MoEShape, make_inputs
    # E = k = 1 with renorm: a dense SwiGLU MLP
    shp = MoEShape("dense", N=5, H=32, E=1, k=1, I=24)
    w = {n: bits_of(t) for n, t in make_inputs(shp, seed=3).items()}
    x = torch.from_numpy(widen(w["x"]))
    mlp = (torch.nn.functional.silu(x @ torch.from_numpy(widen(w["w_gate"][0])).T)
           * (x @ torch.from_numpy(widen(w["w_up"][0])).T)) @ torch.from_numpy(widen(w["w_down"][0])).T
    np.testing.assert_allclose(orc.moe_forward(w, 1, True), mlp.numpy(), rtol=1e-10, atol=1e-13)

    # k = E with renorm: the weights are the full softmax, sorted descending
    shp = MoEShape("kE", N=6, H=16, E=5, k=5, I=8)
    w = {n: bits_of(t) for n, t in make_inputs(shp, seed=4).items()}
    logits, _, wt, ids = orc.route(w["x"], w["router"], 5, True)
    sm = scipy.special.softmax(widen(w["x"]) @ widen(w["router"]).T, axis=1)
    np.testing.assert_allclose(wt, np.take_along_axis(sm, ids.astype(np.int64), 1), rtol=1e-12)
    assert np.all(np.diff(wt, axis=1) <= 0), "k=E weights not descending"

    # renormalised weights == softmax over the top-k logits; raw weights sum < 1
    shp = MoEShape("norm", N=12, H=16, E=8, k=3, I=8)
    w = {n: bits_of(t) for n, t in make_inputs(shp, seed=6).items()}
    logits, _, wn, ids = orc.route(w["x"], w["router"], 3, True)
    _, _, wr, ids_r = orc.route(w["x"], w["router"], 3, False)
    assert np.array_equal(ids, ids_r)
    topl = np.take_along_axis(logits, ids.astype(np.int64), 1)
    np.testing.assert_allclose(wn, scipy.special.softmax(topl, axis=1), rtol=1e-12)
    np.testing.assert_allclose(wn.sum(1), 1.0, rtol=1e-14)
    assert np.all(wr.sum(1) < 1.0)
    # raw top-k weights differ from a softmax over the top-k logits (the
    # "top-k logits then softmax" pitfall only coincides when renormalising)
    assert np.abs(wr - scipy.special.softmax(topl, axis=1)).max() > 1e-3


def check_ties(orc):
    """Exact ties in the probabilities go to the lower expert index, which is
    what numpy's stable argsort of the negated probabilities gives."""
    rng = np.random.default_rng(12)
    H, E = 16, 6
    x = bits(rng.standard_normal((5, H)))
    # all logits zero: every probability is 1/E
    _, probs, w, ids = orc.route(x, bits(np.zeros((E, H))), 3, True)
    assert ids.tolist() == [[0, 1, 2]] * 5, f"all-equal ties {ids.tolist()}"
    np.testing.assert_allclose(w, 1.0 / 3.0, rtol=1e-14)
    # duplicated router rows give bit-identical logits
    base = rng.standard_normal((E, H)) * 0.5
    base[2] = base[1]
    base[4] = base[1]
    router = bits(base)
    for k in (2, 3, 4):
        _, probs, _, ids = orc.route(x, router, k, False)
        want = np.argsort(-probs, axis=1, kind="stable")[:, :k]
        assert np.array_equal(ids, want), f"duplicated-row ties k={k}: {ids} vs {want}"


def check_align_vs_numpy(orc):
    rng = np.random.default_rng(7)
    for (N, k, E, BM) in [(1000, 8, 64, 128), (37, 3, 11, 16), (5, 2, 9, 4), (0, 4, 7, 128),
                          (1, 1, 1, 1)]:
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(N)]) \
            if N else np.zeros((0, k), np.int32)
        if N > 50:
            ids[ids == 5] = 6  # an expert with no pairs (align needs no distinct ids)
        ids = ids.astype(np.int32)
        r = orc.align(ids, E, BM)
        flat = ids.reshape(-1)
        P = flat.size
        assert np.array_equal(r["counts"], np.bincount(flat, minlength=E))
        assert np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
        assert np.array_equal(r["order"], np.argsort(flat, kind="stable"))
        seg = -(-np.bincount(flat, minlength=E) // BM) * BM
        pad_off = np.concatenate([[0], np.cumsum(seg)])
        assert r["num_padded"] == pad_off[-1]
        sp = r["sorted_pair"]
        for e in range(E):
            c = r["counts"][e]
            s = sp[pad_off[e]:pad_off[e + 1]]
            assert np.array_equal(s[:c], r["order"][r["offsets"][e]:r["offsets"][e + 1]])
            assert np.all(s[c:] == P), f"expert {e} padding not sentinel"
            assert np.all(r["block_expert"][pad_off[e] // BM:pad_off[e + 1] // BM] == e)


def check_batch_invariance(orc):
    from sparse_moe_ffn_gb300.inputs import MoEShape, make_inputs
    shp = MoEShape("bi", N=10, H=32, E=8, k=2, I=16, I_s=16)
    w = {n: bits_of(t) for n, t in make_inputs(shp, seed=9).items()}
    full = orc.moe_forward(w, 2, True)
    for i in (0, 4, 9):
        one = dict(w)
        one["x"] = w["x"][i:i + 1]
        assert np.array_equal(orc.moe_forward(one, 2, True)[0], full[i])
        assert np.array_equal(orc.moe_forward(w, 2, True, rows=[i])[0], full[i])


def check_add_rmsnorm(orc):
    """Residual add in bf16, then RMSNorm: against torch's rms_norm in fp64 on
    the bf16 sum, a closed form (constant rows) and the Gemma (1 + w) form."""
    rng = np.random.default_rng(21)
    N, H, eps = 9, 96, 1e-6
    x = bits(rng.standard_normal((N, H)))
    res = bits(rng.standard_normal((N, H)) * 3)
    w = bits(1 + 0.1 * rng.standard_normal(H))
    r_bits, normed = orc.add_rmsnorm(x, res, w, eps)
    r_ref = (torch.from_numpy(widen(x)) + torch.from_numpy(widen(res))).to(torch.bfloat16)
    assert np.array_equal(r_bits, r_ref.view(torch.int16).numpy().view(np.uint16))
    want = torch.nn.functional.rms_norm(r_ref.double(), (H,), torch.from_numpy(widen(w)), eps)
    np.testing.assert_allclose(normed, want.numpy(), rtol=1e-12, atol=1e-14)
    _, g = orc.add_rmsnorm(x, res, w, eps, gemma=True)
    want_g = torch.nn.functional.rms_norm(r_ref.double(), (H,), 1 + torch.from_numpy(widen(w)), eps)
    np.testing.assert_allclose(g, want_g.numpy(), rtol=1e-12, atol=1e-14)
    # a constant row c normalises to c / sqrt(c^2 + eps) * w
    c = np.full((1, H), 0.75)
    _, one = orc.add_rmsnorm(bits(c), bits(np.zeros((1, H))), w, eps)
    np.testing.assert_allclose(one[0], 0.75 / np.sqrt(0.5625 + eps) * widen(w), rtol=1e-13)


ALL_CHECKS = [check_bookkeeping, check_route_io, check_scalar_e2e, check_shared,
              check_shape_trace, check_brute_force, check_closed_forms, check_ties,
              check_align_vs_numpy, check_batch_invariance, check_add_rmsnorm]


def failures(orc):
    """Names of the checks that fail (or crash) for ``orc``."""
    bad = []
    for chk in ALL_CHECKS:
        try:
            chk(orc)
        except Exception as exc:  # noqa: BLE001 -- a crash is a failure too
            bad.append(f"{chk.__name__}: {type(exc).__name__}")
    return bad
