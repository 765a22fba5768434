"""The expert-parallel compute steps on one GPU: moe_experts (the receiving
side of dispatch) and moe_combine (the last step of the combine), and the
whole exchange path of ep_forward with one rank, against moe_forward.  Each
(token, slot) pair is computed by the same tile kernels whatever batch it
sits in, so all of these agree with moe_forward bit for bit.

Two ranks are emulated in one process by running moe_experts once per half
of the experts, one call after the other; no kernel waits on another."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import (FORMS, assert_close, decode_pair_rows, oracle_outputs, prepare, prepared,
                       run_forward, shared_of)
from sparse_moe_ffn_gb300 import binding
from sparse_moe_ffn_gb300.ep import ep_dispatch_reference, ep_forward, ep_plan
from sparse_moe_ffn_gb300.inputs import MoEShape

pytestmark = pytest.mark.gpu


def _pairs(shape, ws):
    v = binding.workspace_views(ws, shape.N, shape.H, shape.E, shape.I, shape.k)
    return (v["topk_w"].reshape(-1).clone(), v["topk_ids"].reshape(-1).clone(),
            tuple(t.clone() for t in v["ypair"]))


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("name", ["tiny", "decode", "prefill"])
def test_experts_rows_and_combine_match_forward(name, form):
    shape, dev, _ = prepared(name, form=form)
    out, ws = run_forward(shape, dev)
    w, ids, ypair = _pairs(shape, ws)
    rows = dev["x"].index_select(0, torch.arange(shape.N * shape.k, device="cuda") // shape.k)
    y, ews = binding.moe_experts(rows, ids, w, dev["w_gate"], dev["w_up"], dev["w_down"])
    torch.cuda.synchronize()
    assert binding.moe_read_device_status(ews) == 0
    assert torch.equal(y[0], ypair[0]) and torch.equal(y[1], ypair[1])
    assert torch.equal(binding.moe_combine(ypair, shape.N, shape.k), out)


def _shifted(t, elems):
    """A contiguous copy of t whose data starts `elems` elements into a fresh
    buffer (16 bytes in: 16-byte but not 32-byte aligned)."""
    buf = torch.empty(t.numel() + elems, dtype=t.dtype, device=t.device)
    view = buf[elems:].view(t.shape)
    view.copy_(t)
    return view


@pytest.mark.parametrize("name", ["prefill", "talker"])
def test_combine_forms_agree_on_unaligned_planes(name):
    """Large batches sum 16 columns per thread with 32-byte loads when the
    planes and the output are 32-byte aligned, else 8 columns per thread;
    both add the same values in the same order, so the bits agree."""
    shape, dev, _ = prepared(name)
    out, ws = run_forward(shape, dev)
    v = binding.workspace_views(ws, shape.N, shape.H, shape.E, shape.I, shape.k, shape.I_s)
    slots, k, H = v["slots"], shape.k, shape.H
    hi = v["ypair"][0].view(shape.N, slots, H)
    res = v["ypair"][1].view(shape.N, slots, H)
    routed = (hi[:, :k].reshape(-1, H).contiguous(), res[:, :k].reshape(-1, H).contiguous())
    shared = None
    if slots > k:
        shared = (hi[:, k:].reshape(-1, H).contiguous(), res[:, k:].reshape(-1, H).contiguous())
    aligned = binding.moe_combine(routed, shape.N, k, yshared=shared)
    assert torch.equal(aligned, out)
    moved = (_shifted(routed[0], 8), _shifted(routed[1], 16))
    moved_shared = None if shared is None else (_shifted(shared[0], 8), _shifted(shared[1], 16))
    target = _shifted(torch.zeros_like(out), 8)
    assert target.data_ptr() % 32 == 16 and moved[0].data_ptr() % 32 == 16
    got = binding.moe_combine(moved, shape.N, k, yshared=moved_shared, out=target)
    assert torch.equal(got, out)


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("name", ["decode", "prefill", "talker"])
def test_ep_forward_one_rank_equals_forward(name, form):
    """talker: the shared expert runs as moe_shared_expert (chunk rows, no
    exchange), and matches moe_forward's shared slots."""
    shape, dev, _ = prepared(name, form=form)
    out, _ = run_forward(shape, dev)
    got = ep_forward(dev["x"], dev["router"], dev["w_gate"], dev["w_up"], dev["w_down"],
                     shape.E, shape.k, shape.norm_topk_prob, shared=shared_of(shape, dev))
    assert torch.equal(got, out)


SHARED_CASES = {
    "talker": None,  # I_s = 2048 in three chunks of I = 768 (the last one 512 rows)
    "three-chunks": MoEShape("three-chunks", N=200, H=128, E=8, k=2, I=64, I_s=160,
                             norm_topk_prob=False),
    # decode-sized: the 32-row-pass GEMMs with expert-indexed tiles
    "sparse-chunks": MoEShape("sparse-chunks", N=24, H=128, E=16, k=2, I=64, I_s=136,
                              norm_topk_prob=True),
}


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("case", list(SHARED_CASES))
def test_shared_expert_rows_equal_forward_slots(case, form):
    """moe_shared_expert's chunk rows equal the pair rows moe_forward holds in
    slots k .. k+C-1 bit for bit, and combining the routed slots with them
    gives the layer's output."""
    if SHARED_CASES[case] is None:
        shape, dev, _ = prepared(case, form=form)
    else:
        shape, dev, _ = prepare(SHARED_CASES[case], seed=8, form=form)
    out, ws = run_forward(shape, dev)
    v = binding.workspace_views(ws, shape.N, shape.H, shape.E, shape.I, shape.k, shape.I_s)
    slots, k, H = v["slots"], shape.k, shape.H
    C = slots - k
    assert C == binding.moe_shared_chunks(shape.I, shape.I_s)
    y, sws = binding.moe_shared_expert(dev["x"], v["gamma"].clone(), shape.I,
                                       dev["shared_gate_proj"], dev["shared_up_proj"],
                                       dev["shared_down_proj"])
    torch.cuda.synchronize()
    assert binding.moe_read_device_status(sws) == 0
    hi = v["ypair"][0].view(shape.N, slots, H)
    res = v["ypair"][1].view(shape.N, slots, H)
    assert torch.equal(y[0], hi[:, k:].reshape(-1, H))
    assert torch.equal(y[1], res[:, k:].reshape(-1, H))
    routed = (hi[:, :k].reshape(-1, H).contiguous(), res[:, :k].reshape(-1, H).contiguous())
    assert torch.equal(binding.moe_combine(routed, shape.N, k, yshared=y), out)


def _fuzz_shapes():
    from test_gpu_parity import FUZZ
    return FUZZ


@pytest.mark.parametrize("shape", _fuzz_shapes(), ids=lambda s: s.name)
def test_ep_forward_one_rank_random_shapes(shape):
    """ep_forward with one rank (device dispatch plan, moe_experts,
    moe_shared_expert, indexed combine) equals moe_forward bit for bit on the
    seeded random shapes."""
    shape, dev, _ = prepare(shape, seed=12)
    out, _ = run_forward(shape, dev)
    got = ep_forward(dev["x"], dev["router"], dev["w_gate"], dev["w_up"], dev["w_down"],
                     shape.E, shape.k, shape.norm_topk_prob, shared=shared_of(shape, dev))
    assert torch.equal(got, out)


@pytest.mark.parametrize("name,world", [("decode", 2), ("prefill", 2), ("prefill", 3),
                                        ("tiny", 4)])
def test_expert_slices_in_one_process_equal_forward(name, world):
    """Each 'rank' holds a contiguous slice of the experts (the last one
    smaller when E does not split evenly) and computes only the pairs the
    device dispatch plan sends it; the results, concatenated in send order
    and combined through each pair's send row, leave the layer unchanged."""
    shape, dev, bits = prepared(name)
    out, ws = run_forward(shape, dev)
    w, ids, _ = _pairs(shape, ws)
    ids2, w2 = ids.view(shape.N, shape.k), w.view(shape.N, shape.k)
    d = binding.moe_ep_dispatch(dev["x"], ids2, w2, shape.E, world)
    counts = d["send_counts"].cpu().tolist()
    E_loc = -(-shape.E // world)
    ys_hi, ys_res = [], []
    start = 0
    for r in range(world):
        n_r = counts[r]
        e0, e1 = r * E_loc, min(shape.E, (r + 1) * E_loc)
        if n_r == 0:
            continue
        sl = slice(start, start + n_r)
        start += n_r
        y, ews = binding.moe_experts(d["send_x"][sl], d["send_ids"][sl], d["send_w"][sl],
                                     dev["w_gate"][e0:e1], dev["w_up"][e0:e1],
                                     dev["w_down"][e0:e1])
        torch.cuda.synchronize()
        assert binding.moe_read_device_status(ews) == 0
        ys_hi.append(y[0])
        ys_res.append(y[1])
    y_back = (torch.cat(ys_hi), torch.cat(ys_res))
    got = binding.moe_combine_indexed(y_back, d["inv_order"], shape.N, shape.k)
    assert torch.equal(got, out)
    assert_close(got, oracle_outputs(name), f"{name} world {world}")


@pytest.mark.parametrize("N,k,E,world", [(1, 1, 1, 1), (64, 8, 128, 2), (700, 6, 64, 3),
                                         (5000, 8, 128, 8), (33, 4, 7, 5)])
def test_device_dispatch_matches_reference(N, k, E, world):
    """moe_ep_dispatch against the host reference plan, bit for bit: send
    rows (token rows, local ids, weights), counts and each pair's send row;
    the grouping runs the single-CTA path (<= 4096 pairs) and the
    three-kernel one."""
    g = torch.Generator().manual_seed(N + E + world)
    H = 64
    x = torch.randn(N, H, generator=g).to(torch.bfloat16)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(N)]).to(torch.int32)
    w = torch.rand(N, k, generator=g)
    d = binding.moe_ep_dispatch(x.cuda(), ids.cuda(), w.cuda(), E, world)
    torch.cuda.synchronize()
    assert binding.moe_read_device_status(d["workspace"]) == 0
    ref = ep_dispatch_reference(x, ids, w, E, world)
    for name, r in zip(("send_x", "send_ids", "send_w", "send_counts", "inv_order"), ref):
        assert torch.equal(d[name].cpu(), r), name


def test_device_dispatch_flags_a_bad_id():
    """An expert id outside [0, E) is not sent (its send row is -1), is
    reported as MOE_ERR_DEVICE_CHECK, and the indexed combine skips it."""
    N, H, E, k, world = 6, 64, 8, 2, 2
    x = torch.randn(N, H).to(torch.bfloat16).cuda()
    ids = torch.tensor([[0, 5], [1, 2], [9, 3], [4, 6], [7, 0], [2, 1]], dtype=torch.int32).cuda()
    w = torch.rand(N, k).cuda()
    d = binding.moe_ep_dispatch(x, ids, w, E, world)
    assert binding.moe_read_device_status(d["workspace"]) == 5  # MOE_ERR_DEVICE_CHECK
    assert int(d["inv_order"][4].item()) == -1                   # pair (2, 0) holds id 9
    assert int(d["send_counts"].sum().item()) == N * k - 1
    n_rows = N * k - 1
    rows = binding.alloc_pair_rows(n_rows, H)
    rows[0].fill_(1.0)
    rows[1].zero_()
    out = binding.moe_combine_indexed(rows, d["inv_order"], N, k)
    sums = out.float().sum(dim=1).cpu() / H
    assert sums.tolist() == [2.0, 2.0, 1.0, 2.0, 2.0, 2.0]


def test_experts_with_empty_experts_and_one_row():
    """Rows routed to a few of many experts, down to a single row."""
    shape, dev, wbits = prepare(MoEShape("slice", N=1, H=256, E=40, k=1, I=192), seed=9)
    for R in (1, 7, 130):
        g = torch.Generator().manual_seed(R)
        x = torch.randn(R, shape.H, generator=g).to(torch.bfloat16).cuda()
        ids = torch.randint(0, 3, (R,), generator=g).to(torch.int32).cuda() * 13  # 0, 13, 26
        w = torch.rand(R, generator=g).cuda()
        y, ews = binding.moe_experts(x, ids, w, dev["w_gate"], dev["w_up"], dev["w_down"])
        torch.cuda.synchronize()
        assert binding.moe_read_device_status(ews) == 0
        # reference: the oracle's E = k = 1 layer is expert e's SwiGLU with
        # routing weight 1; scale by the row's weight afterwards
        ids_h, w_h = ids.cpu().numpy(), w.cpu().numpy().astype(np.float64)
        ref = np.zeros((R, shape.H))
        for e in np.unique(ids_h):
            sel = np.nonzero(ids_h == e)[0]
            bits = {"x": oracle.bf16_bits(x[torch.from_numpy(sel).cuda()]),
                    "router": np.zeros((1, shape.H), np.uint16),
                    "w_gate": wbits["w_gate"][e:e + 1], "w_up": wbits["w_up"][e:e + 1],
                    "w_down": wbits["w_down"][e:e + 1]}
            ref[sel] = oracle.moe_forward(bits, 1, True) * w_h[sel, None]
        assert_close(decode_pair_rows(y), ref, f"R={R}")
