"""GPU parity: every kernel of the layer against the fp64 oracle, through the
C ABI (ctypes binding).  Routing and grouping are compared bit for bit, the
layer's outputs element by element over every token of every configuration
within the tolerance stated in gpu_cases.py, for both forms of the down
weights (the model's bf16, and the fp16 copies of the prepared entry
points)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import (ALL, FORMS, WEIGHT_ATOL, assert_close, decode_pair_rows, error_stats,
                       oracle_outputs, prepare, prepared, run_forward, shared_of)
from sparse_moe_ffn_gb300 import binding
from sparse_moe_ffn_gb300.inputs import MoEShape

pytestmark = pytest.mark.gpu

# Per-pair outputs w * Expert(x) are kept as pair rows (16 significant bits,
# error <= 2^-16 relative), so they can be held to a far tighter bound than
# the layer's bf16 output: the hi/lo activation carries 16 significant bits
# (error ~2^-17 relative per element), the fp16 one 11 (~2^-12).  Max |err|
# over the sampled pairs, relative to their rms.
PAIR_TOL = {"bf16": 2e-4, "f16": 3e-3}


# ----------------------------------------------------------------- routing

@pytest.mark.parametrize("name", ALL)
def test_route_matches_oracle(name):
    shape, dev, bits = prepared(name)
    sg = dev.get("shared_gate")
    w, ids, gamma, wb = binding.moe_route_raw(dev["x"], dev["router"], shape.k,
                                              shape.norm_topk_prob, shared_gate=sg,
                                              want_bf16=True)
    logits, _, w_ref, ids_ref = oracle.route(bits["x"], bits["router"], shape.k,
                                             shape.norm_topk_prob)
    got_ids = ids.cpu().numpy()
    assert np.array_equal(got_ids, ids_ref), \
        f"{name}: {np.sum(got_ids != ids_ref)} ids differ"
    werr = np.abs(w.cpu().numpy() - w_ref).max()
    assert werr <= WEIGHT_ATOL, f"{name}: routing weight error {werr:.3e}"
    # exported bf16 weights are the fp32 weights rounded to nearest even
    assert torch.equal(wb, w.to(torch.bfloat16))
    if sg is not None:
        g_ref = 1.0 / (1.0 + np.exp(-(oracle.widen(bits["x"]) @ oracle.widen(bits["shared_gate"]).T)[:, 0]))
        gerr = np.abs(gamma.cpu().numpy() - g_ref).max()
        assert gerr <= WEIGHT_ATOL, f"{name}: shared gate error {gerr:.3e}"
    # the page's route(): weights in x.dtype, ids int64
    wt, it = binding.moe_route(dev["x"], dev["router"], shape.k, shape.norm_topk_prob)
    assert wt.dtype == dev["x"].dtype and it.dtype == torch.int64
    assert np.array_equal(it.cpu().numpy(), ids_ref)


def test_route_sums():
    """Renormalised weights sum to 1; unrenormalised ones to less than 1."""
    shape, dev, _ = prepared("decode")
    w, _, _, _ = binding.moe_route_raw(dev["x"], dev["router"], shape.k, True)
    assert torch.allclose(w.sum(1), torch.ones(shape.N, device="cuda"), atol=1e-6)
    w, _, _, _ = binding.moe_route_raw(dev["x"], dev["router"], shape.k, False)
    assert bool((w.sum(1) < 1.0).all())


# ---------------------------------------------------------------- grouping

def _align_vs_oracle(ids_np, E, block_m):
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
    r = binding.moe_align(ids, E, block_m)
    torch.cuda.synchronize()
    ref = oracle.align(ids_np, E, block_m)
    npad = int(r["num_padded"].item())
    assert npad == ref["num_padded"]
    assert np.array_equal(r["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(r["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(r["sorted_pair"][:npad].cpu().numpy(), ref["sorted_pair"])
    assert np.array_equal(r["block_expert"][:npad // block_m].cpu().numpy(),
                          ref["block_expert"])
    assert binding.moe_read_device_status(r["workspace"]) == 0


@pytest.mark.parametrize("name", ALL)
def test_align_matches_oracle(name):
    shape, dev, bits = prepared(name)
    _, _, _, ids = oracle.route(bits["x"], bits["router"], shape.k, shape.norm_topk_prob)
    _align_vs_oracle(ids, shape.E, 128)


@pytest.mark.parametrize("N,k,E,block_m", [(1, 1, 1, 1), (3, 2, 5, 4), (1000, 8, 64, 16),
                                           (5000, 4, 1024, 128), (70000, 2, 3, 1),
                                           (513, 8, 128, 128), (4096, 8, 256, 64)])
def test_align_random(N, k, E, block_m):
    rng = np.random.default_rng(N + E)
    ids = rng.integers(0, E, size=(N, k)).astype(np.int32)
    if E > 4:
        ids[ids == 3] = 4  # an expert with no pairs
    _align_vs_oracle(ids, E, block_m)


@pytest.mark.parametrize("N,H,E,k", [(1, 2048, 128, 8), (7, 64, 6, 2), (64, 2048, 128, 8),
                                     (100, 200, 32, 12), (127, 128, 256, 4), (128, 512, 16, 16)])
def test_routing_kernel_grouping(N, H, E, k):
    """One cluster routes every token (N <= 128, no shared expert): the
    routing kernel groups the pairs itself, and what it writes into the
    forward workspace equals moe_align's result on the same ids, bit for bit,
    and the oracle's grouping (H spans cluster sizes 1, 2, 4 and 8; k = 12
    and 16 place more pairs per CTA than one pass)."""
    shape, dev, _ = prepare(MoEShape("grouped-in-router", N=N, H=H, E=E, k=k, I=64), seed=11)
    out, ws = run_forward(shape, dev)
    v = binding.workspace_views(ws, N, H, E, 64, k)
    ids = v["topk_ids"].clone()
    ref = oracle.align(ids.cpu().numpy(), E, 128)
    npad = int(v["num_padded"].item())
    assert npad == ref["num_padded"]
    assert np.array_equal(v["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(v["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(v["sorted_pair"][:npad].cpu().numpy(), ref["sorted_pair"])
    assert np.array_equal(v["block_expert"][:npad // 128].cpu().numpy(), ref["block_expert"])
    r = binding.moe_align(ids, E, 128)
    torch.cuda.synchronize()
    assert np.array_equal(r["sorted_pair"][:npad].cpu().numpy(),
                          v["sorted_pair"][:npad].cpu().numpy())
    assert np.array_equal(r["counts"].cpu().numpy(), v["counts"].cpu().numpy())


def test_align_flags_bad_ids():
    """An id outside [0, E) is skipped and recorded in the status word."""
    ids = torch.tensor([[0, 1], [7, 2]], dtype=torch.int32, device="cuda")
    r = binding.moe_align(ids, 4, 8)
    assert binding.moe_read_device_status(r["workspace"]) == 5  # MOE_ERR_DEVICE_CHECK


# ------------------------------------------------------------ whole layer

@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("name", ALL)
def test_forward_matches_oracle(name, form):
    """Every output element of the layer against the oracle."""
    shape, dev, bits = prepared(name, form=form)
    out, ws = run_forward(shape, dev)
    assert_close(out, oracle_outputs(name), f"{name} ({form} down weights)")
    # the stages inside the workspace: routing and grouping bit-exact
    v = binding.workspace_views(ws, shape.N, shape.H, shape.E, shape.I, shape.k, shape.I_s)
    _, _, _, ids_ref = oracle.route(bits["x"], bits["router"], shape.k, shape.norm_topk_prob)
    assert np.array_equal(v["routed_ids"].cpu().numpy(), ids_ref)
    # the shared expert's chunks: virtual experts E, E+1, ... in the slots
    # after the routed ones, for every token
    C = v["slots"] - shape.k
    assert C == (-(-shape.I_s // shape.I) if shape.I_s else 0)
    all_ids = np.concatenate(
        [ids_ref, np.tile(np.arange(shape.E, shape.E + C, dtype=ids_ref.dtype), (shape.N, 1))],
        axis=1)
    assert np.array_equal(v["topk_ids"].cpu().numpy(), all_ids)
    al = oracle.align(all_ids, shape.E + C, 128)
    npad = int(v["num_padded"].item())
    assert npad == al["num_padded"]
    assert np.array_equal(v["counts"].cpu().numpy(), al["counts"])
    assert np.array_equal(v["sorted_pair"][:npad].cpu().numpy(), al["sorted_pair"])


PAIR_CASES = {
    # the three GEMM tilings: 32-row passes (decode), one CTA per row block
    # (between 32 and 128 pairs per expert), CTA pairs (prefill)
    "decode": None,
    "ragged": MoEShape("ragged", N=300, H=256, E=16, k=4, I=192),
    "prefill": None,
}


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("case", list(PAIR_CASES))
def test_pair_outputs(case, form):
    """K3 + K4 per pair: ypair[p] = w_p * Expert_{e_p}(x_n) (decoded pair rows)
    for sampled pairs, the expert evaluated by the oracle as a one-expert
    layer."""
    if PAIR_CASES[case] is None:
        shape, dev, bits = prepared(case, form=form)
    else:
        shape, dev, bits = prepare(PAIR_CASES[case], seed=6, form=form)
    out, ws = run_forward(shape, dev)
    v = binding.workspace_views(ws, shape.N, shape.H, shape.E, shape.I, shape.k)
    ids = v["topk_ids"].cpu().numpy()
    w = v["topk_w"].cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(1)
    pairs = rng.choice(shape.N * shape.k, size=24, replace=False)
    sel = torch.from_numpy(pairs).cuda()
    ypair = decode_pair_rows((v["ypair"][0][sel], v["ypair"][1][sel]))
    ref = []
    for p in pairs:
        n, j = divmod(int(p), shape.k)
        e = int(ids[n, j])
        one = {"x": bits["x"][n:n + 1], "router": bits["router"][:1],
               "w_gate": bits["w_gate"][e:e + 1], "w_up": bits["w_up"][e:e + 1],
               "w_down": bits["w_down"][e:e + 1]}
        # the fp32 weight the kernel used, times the expert's exact output
        ref.append(w[n, j] * oracle.moe_forward(one, 1, True)[0])
    ref = np.array(ref)
    err = np.abs(ypair - ref).max()
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert err <= PAIR_TOL[form] * rms, f"{case}/{form}: pair max|err| {err / rms:.3e} * rms"


EDGE = [
    # name, N, H, E, k, I, I_s, norm
    ("ragged", 300, 256, 16, 4, 192, 0, True),
    ("one-token", 1, 128, 8, 2, 64, 0, True),
    ("tile-plus-one", 129, 64, 8, 2, 128, 0, False),
    ("k-equals-E", 40, 64, 4, 4, 64, 0, True),
    ("dense-E1-k1", 77, 128, 1, 1, 96, 0, True),
    ("odd-E-shared", 50, 64, 6, 2, 128, 64, False),
    ("ragged-H-I", 200, 200, 10, 3, 72, 40, True),
    ("wide-E", 256, 128, 256, 8, 64, 0, True),
    ("E248-shared", 64, 64, 248, 4, 32, 16, False),
    # fewer than 32 pairs per expert: the GEMMs with 32-row activation
    # passes (K tails in both GEMMs, a partial N tile)
    ("sparse-ragged-H-I", 40, 200, 32, 4, 72, 0, True),
    # at least two row blocks per expert: the CTA-pair GEMMs (odd block
    # counts leave half-empty pairs; ragged H and I give K and N tails)
    ("pairs-3-blocks", 600, 256, 4, 2, 256, 0, True),
    ("pairs-ragged-H-I", 700, 200, 5, 3, 200, 0, False),
    ("pairs-E1-k1", 520, 128, 1, 1, 128, 0, True),
    ("pairs-shared", 600, 128, 4, 2, 128, 64, True),
    # the shared expert cut into three chunks of I rows, the last one partly
    # zero padding: one-CTA tiles, CTA pairs, expert-indexed sparse tiles
    ("shared-3-chunks", 200, 128, 8, 2, 64, 160, False),
    ("pairs-shared-3-chunks", 600, 128, 4, 2, 96, 200, True),
    ("sparse-shared-3-chunks", 24, 128, 16, 2, 64, 136, False),
    # the limits on experts with a shared expert: E = 248 (the shared gate's
    # router column follows E rounded up to 8) and E + C = 256 (C = 8 chunks)
    ("shared-at-expert-limit", 40, 64, 248, 4, 32, 256, False),
]


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("case", EDGE, ids=[c[0] for c in EDGE])
def test_forward_edge_shapes(case, form):
    name, N, H, E, k, I, I_s, norm = case
    shape, dev, bits = prepare(MoEShape(name, N=N, H=H, E=E, k=k, I=I, I_s=I_s,
                                        norm_topk_prob=norm), seed=3, form=form)
    out, _ = run_forward(shape, dev)
    ref = oracle.moe_forward(bits, k, norm)
    assert_close(out, ref, f"{name} ({form})")


@pytest.mark.parametrize("form", FORMS)
def test_forward_every_expert_per_token(form):
    """The largest top-k: k = E = 256, every token routed to every expert.
    Random logits over 256 experts leave gaps below the near-tie margin, so
    column 0 spreads them instead: x[:, 0] = 4 and router[e, 0] = (e - 128)
    / 64 put expert e's logit near (e - 128) / 16, the rest of the router
    scaled down to noise (std ~0.01), so the descending order of all 256 is
    unambiguous.  Ids bit for bit, outputs within the tolerance."""
    from sparse_moe_ffn_gb300.inputs import MARGIN, _near_tie_rows, make_inputs, to_device
    shape = MoEShape("k-equals-E-256", N=3, H=64, E=256, k=256, I=32, norm_topk_prob=True)
    cpu = make_inputs(MoEShape("k-equals-E-256-draw", N=3, H=64, E=256, k=1, I=32), seed=13)
    x = cpu["x"].float()
    router = cpu["router"].float() * 0.05
    x[:, 0] = 4.0
    router[:, 0] = (torch.arange(256, dtype=torch.float32) - 128.0) / 64.0
    cpu["x"], cpu["router"] = x.to(torch.bfloat16), router.to(torch.bfloat16)
    assert _near_tie_rows(cpu["x"], cpu["router"], shape.k, MARGIN).numel() == 0
    bits = {n: oracle.bf16_bits(t) for n, t in cpu.items()}
    dev = to_device(cpu, "cuda")
    if form == "f16":
        dev = binding.prepare_weights(dev)
    out, ws = run_forward(shape, dev)
    _, _, _, ids_ref = oracle.route(bits["x"], bits["router"], shape.k, True)
    ids = binding.workspace_views(ws, shape.N, shape.H, shape.E, shape.I, shape.k)["topk_ids"]
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.array_equal(ids_ref[:, 0], np.full(3, 255))  # descending: expert 255 first
    assert_close(out, oracle.moe_forward(bits, shape.k, True), shape.name)


def _random_shapes(n, seed):
    """Seeded random layer shapes spanning the three GEMM tilings, ragged H
    and I (multiples of 8), k up to E, and the shared expert in one or
    several chunks."""
    rng = np.random.default_rng(seed)
    shapes = []
    for i in range(n):
        E = int(rng.choice([1, 3, 8, 24, 64, 160]))
        k = int(rng.integers(1, min(E, 10) + 1))
        N = int(rng.choice([1, 5, 37, 128, 129, 300, 900]))
        H = int(rng.integers(1, 40)) * 8
        I = int(rng.integers(1, 33)) * 8
        I_s = int(rng.integers(1, 50)) * 8 if (E + 8 <= 240 and rng.random() < 0.4) else 0
        shapes.append(MoEShape(f"fuzz{i}", N=N, H=H, E=E, k=k, I=I, I_s=I_s,
                               norm_topk_prob=bool(rng.random() < 0.5)))
    return shapes


FUZZ = _random_shapes(16, 2024)


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("shape", FUZZ, ids=[f"{s.name}-N{s.N}-H{s.H}-E{s.E}-k{s.k}-I{s.I}-Is{s.I_s}"
                                              for s in FUZZ])
def test_forward_random_shapes(shape, form):
    """Random shapes (seeded) against the oracle, every output element."""
    shape, dev, bits = prepare(shape, seed=12, form=form)
    out, _ = run_forward(shape, dev)
    assert_close(out, oracle.moe_forward(bits, shape.k, shape.norm_topk_prob), shape.name)


def _forward_status(shape, dev, x):
    ws = binding.alloc_workspace(x.shape[0], shape.H, shape.E, shape.I, shape.k, shape.I_s)
    out = binding.moe_forward(x, dev["router"], dev["w_gate"], dev["w_up"], dev["w_down"],
                              shape.k, shape.norm_topk_prob, shared_of(shape, dev),
                              workspace=ws)
    return out, binding.moe_read_device_status(ws)


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("bad", ["nan", "inf"])
@pytest.mark.parametrize("N", [40, 300, 600])  # 32-row passes, one-CTA tiles, CTA pairs
def test_non_finite_token_is_reported(form, bad, N):
    """A token whose x row holds a NaN or an infinity gives non-finite
    activations and pair outputs: the layer records MOE_ERR_DEVICE_CHECK,
    its ids stay in [0, E), and every other token's output still matches the
    oracle (tokens do not mix)."""
    shape, dev, bits = prepare(MoEShape("non-finite", N=N, H=128, E=8, k=2, I=64, I_s=64,
                                        norm_topk_prob=False), seed=9, form=form)
    x = dev["x"].clone()
    x[7, 5] = float("nan") if bad == "nan" else float("inf")
    out, status = _forward_status(shape, dev, x)
    assert status == 5  # MOE_ERR_DEVICE_CHECK
    keep = np.array([n for n in range(N) if n != 7])
    ref = oracle.moe_forward(bits, shape.k, shape.norm_topk_prob)
    assert_close(out[torch.from_numpy(keep).cuda()], ref[keep], f"{bad} token, other rows")


@pytest.mark.parametrize("form", FORMS)
def test_activation_range(form):
    """One token scaled by 2^12 gives activations of ~1e5-1e6: past fp16's
    65504, so the prepared path (fp16 activation) records
    MOE_ERR_DEVICE_CHECK, while the bf16 hi/lo activation holds them and the
    layer stays within the tolerance of the oracle."""
    shape, dev, bits = prepare(MoEShape("range", N=40, H=128, E=8, k=2, I=64), seed=10,
                               form=form)
    x = dev["x"].clone()
    x[3] *= 4096.0
    out, status = _forward_status(shape, dev, x)
    assert status == (5 if form == "f16" else 0)
    if form == "bf16":
        big = dict(bits)
        big["x"] = oracle.bf16_bits(x)
        ref = oracle.moe_forward(big, shape.k, shape.norm_topk_prob)
        assert_close(out[3:4], ref[3:4], "scaled token")
        rest = np.array([n for n in range(shape.N) if n != 3])
        assert_close(out[torch.from_numpy(rest).cuda()], ref[rest], "other tokens")


@pytest.mark.parametrize("form", FORMS)
def test_forward_mixed_sparse_and_dense_row_blocks(form):
    """Skewed routing at a small size with top-10: each token takes the 8 hot
    experts (160 pairs each: one full row block loaded as a tiled box, then a
    block of exactly 32 rows, gathered) and two of the others (3 to 21 pairs,
    gathered four rows at a time), all in one call."""
    shape, dev, bits = prepare(MoEShape("skewed-small", N=160, H=256, E=64, k=10, I=128,
                                        skew=True), seed=4, form=form)
    out, ws = run_forward(shape, dev)
    v = binding.workspace_views(ws, shape.N, shape.H, shape.E, shape.I, shape.k)
    counts = v["counts"].cpu()
    assert int(counts.max()) > 64 and int(counts[counts > 0].min()) <= 32
    ref = oracle.moe_forward(bits, shape.k, shape.norm_topk_prob)
    assert_close(out, ref, shape.name)


@pytest.mark.parametrize("form", FORMS)
def test_forward_expert_indexed_tiles_with_passes_and_empty_experts(form):
    """N <= 128 with fewer than 32 pairs per expert on average: gate/up tiles
    are indexed by expert.  Skewed routing gives the 8 hot experts 45-52
    pairs (two 32-row passes each; three or four 16-row passes in the down
    GEMM of the hi/lo activation) and 16 experts none (their tiles take no
    pass)."""
    shape, dev, bits = prepare(MoEShape("expert-tiles", N=128, H=256, E=24, k=3, I=128,
                                        skew=True), seed=5, form=form)
    out, ws = run_forward(shape, dev)
    counts = binding.workspace_views(ws, shape.N, shape.H, shape.E, shape.I, shape.k)["counts"]
    counts = counts.cpu()
    assert int(counts.max()) > 32 and int((counts == 0).sum()) >= 10
    ref = oracle.moe_forward(bits, shape.k, shape.norm_topk_prob)
    assert_close(out, ref, shape.name)


@pytest.mark.parametrize("form", FORMS)
def test_batch_invariance_skewed(form):
    """A token computed alone equals the same token inside the skewed batch,
    bit for bit (routing, grouping position and GEMM order do not depend on
    the rest of the batch)."""
    shape, dev, _ = prepared("skewed", form=form)
    out, _ = run_forward(shape, dev)
    for i in (0, 1, 4097, shape.N - 1):
        one, _ = run_forward(shape, dev, x=dev["x"][i:i + 1].contiguous())
        assert torch.equal(one[0], out[i]), f"row {i} differs"
    w_all, ids_all, _, _ = binding.moe_route_raw(dev["x"], dev["router"], shape.k, True)
    w_one, ids_one, _, _ = binding.moe_route_raw(dev["x"][5:6].contiguous(), dev["router"],
                                                 shape.k, True)
    assert torch.equal(ids_all[5], ids_one[0]) and torch.equal(w_all[5], w_one[0])


def test_repeatable_and_status_clean():
    shape, dev, _ = prepared("talker")
    a, ws = run_forward(shape, dev)
    b, _ = run_forward(shape, dev, workspace=ws)
    assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["talker", "skewed", "prefill"])
def test_repeated_calls_with_fresh_workspaces(name):
    """Back-to-back layer calls (kernels chained by programmatic dependent
    launch), each with a newly allocated workspace, give bit-identical
    outputs: no kernel reads a stale copy of its predecessor's results."""
    shape, dev, _ = prepared(name)
    first, _ = run_forward(shape, dev)
    for _ in range(3):
        again, _ = run_forward(shape, dev)
        assert torch.equal(first, again)
    # and calls queued without a synchronisation in between
    outs = []
    for _ in range(3):
        ws = binding.alloc_workspace(shape.N, shape.H, shape.E, shape.I, shape.k, shape.I_s)
        outs.append(binding.moe_forward(dev["x"], dev["router"], dev["w_gate"], dev["w_up"],
                                        dev["w_down"], shape.k, shape.norm_topk_prob,
                                        shared_of(shape, dev), workspace=ws))
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(first, o)


def test_zero_tokens_is_a_noop():
    shape, dev, _ = prepared("tiny")
    x = dev["x"][:0]
    out = binding.moe_forward(x, dev["router"], dev["w_gate"], dev["w_up"], dev["w_down"],
                              shape.k, True)
    assert out.shape == (0, shape.H)


def test_error_summary_is_reported(capsys):
    """Print the measured error figures of every configuration, over every
    output element, for both forms of the down weights, next to the error of
    the oracle's own result rounded once to bf16 -- the floor that no bf16
    output can go below (information)."""
    for name in ALL:
        ref = oracle_outputs(name)
        floor, rms, _ = error_stats(torch.from_numpy(ref).to(torch.bfloat16), ref)
        for form in FORMS:
            shape, dev, _ = prepared(name, form=form)
            out, _ = run_forward(shape, dev)
            mx, rms, mean_rel = error_stats(out, ref)
            print(f"{name} [{form}]: max|err|/rms = {mx / rms:.4e} (bf16 rounding of the exact "
                  f"result: {floor / rms:.4e}), mean rel err = {mean_rel:.3e}")
