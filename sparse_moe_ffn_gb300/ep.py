"""Expert parallelism: the layer's experts split across ranks.  Every rank
routes its own tokens over all experts and exchanges its (token, slot) pairs
with the ranks that own the chosen experts.  This is the expert-parallel
follow-up of the M03 drill's level-3 hints, where the (token, expert) table
drives an all-to-all dispatch and an all-to-all combine.

Rank r owns experts [r * E_local, (r + 1) * E_local), E_local = ceil(E / R),
and holds only their weights.  Per layer call, on every rank:

1. route its N tokens over all E experts (moe_route: fp32 weights, ids);
2. dispatch plan, on the device (moe_ep_dispatch): pair p = n*k + j goes to
   rank ids[p] // E_local; the pairs are grouped by destination rank, in
   pair order within a rank (moe_align's grouping kernels with R groups),
   and packed in that order: token rows, expert ids local to the receiving
   rank, routing weights, the per-rank counts, and each pair's send row;
3. exchange: the counts first (the one host synchronisation: all_to_all
   needs the split sizes on the host), then the rows, ids and weights with
   one all_to_all each;
4. the receiving rank runs its experts on the rows it received
   (moe_experts: y = w * Expert(x) as pair rows, a bf16 plane and an int8
   residual plane);
5. combine: the results travel back with the reverse all_to_all, in send
   order, and moe_combine_indexed sums each token's k slots in slot order,
   reading pair p's row at its send row.

Step 4 computes each pair as moe_forward does, and step 5 is moe_forward's
own combine.  So the output equals moe_forward on the same tokens bit for
bit, whatever the number of ranks.

The shared expert (the talker layer) is dense: every rank holds its weights
and applies it to its own tokens, with no exchange.  It runs as
moe_shared_expert, which computes moe_forward's shared term gamma *
SharedMLP(x) the same way (its intermediate rows in chunks of the routed
experts' I, one pair row per chunk); the combine adds the chunk rows after
the k slots.

Transport: gloo and NCCL both carry int32, so bf16 rows and int8 residual
rows travel as their bit patterns viewed as int32 (H is a multiple of 8).
With one rank nothing is exchanged.  The compute steps can be replaced
(route_fn, dispatch_fn, experts_fn, shared_fn, combine_fn), which is how the
exchange logic is tested on CPU ranks; ``ep_dispatch_reference`` is the
dispatch plan written with host tensor operations for that purpose (and the
reference the device plan is tested against).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def ep_plan(ids: torch.Tensor, E: int, world: int):
    """Destination rank of every pair and the send order.

    Returns (order, dest, send_counts, E_local): ``order`` lists the pair
    indices p = n*k + j grouped by destination rank (stable within a rank),
    ``dest[p]`` is the rank owning expert ids[p], ``send_counts[r]`` the
    number of pairs sent to rank r."""
    if world < 1:
        raise ValueError("world must be >= 1")
    E_local = -(-E // world)
    flat = ids.reshape(-1).long()
    if flat.numel() and (int(flat.min()) < 0 or int(flat.max()) >= E):
        raise ValueError("expert ids must lie in [0, E)")
    dest = flat // E_local
    order = torch.sort(dest, stable=True).indices
    send_counts = torch.bincount(dest, minlength=world)
    return order, dest, send_counts, E_local


def ep_dispatch_reference(x, ids, w, E: int, world: int):
    """The dispatch plan of step 2 with torch operations (CPU ranks, tests):
    returns (send_x, send_ids, send_w, send_counts, inv_order) as
    moe_ep_dispatch defines them."""
    order, dest, send_counts, E_local = ep_plan(ids, E, world)
    k = ids.shape[1]
    send_x = x.index_select(0, order // k)
    send_e = (ids.reshape(-1).long()[order] - dest[order] * E_local).to(torch.int32)
    send_w = w.reshape(-1)[order].contiguous()
    inv = torch.empty_like(order)
    inv[order] = torch.arange(order.numel(), device=order.device)
    return send_x, send_e, send_w, send_counts.to(torch.int32), inv.to(torch.int32)


def _world(group):
    if not dist.is_available() or not dist.is_initialized():
        return 1
    return dist.get_world_size(group)


def _exchange(t: torch.Tensor, send_counts, recv_counts, group):
    """Rows of ``t`` (int32) sent in blocks of send_counts[r] rows to rank r;
    returns the rows received, recv_counts[r] from rank r."""
    out = torch.empty((int(sum(recv_counts)),) + tuple(t.shape[1:]), dtype=t.dtype,
                      device=t.device)
    dist.all_to_all_single(out, t.contiguous(), output_split_sizes=list(recv_counts),
                           input_split_sizes=list(send_counts), group=group)
    return out


def ep_forward(x, router, w_gate, w_up, w_down, E: int, k: int, norm_topk_prob: bool = True,
               group=None, shared=None, route_fn=None, dispatch_fn=None, experts_fn=None,
               shared_fn=None, combine_fn=None):
    """One MoE layer with experts split across the ranks of ``group``.

    x [N, H] bf16 (this rank's tokens), router [E, H] bf16 (all experts);
    w_gate, w_up [E_r, I, H] bf16 and w_down [E_r, H, I] (bf16, or the fp16
    copy of binding.prepare_weights): this rank's experts.  ``shared``: None
    or the shared expert (binding.SHARED_KEYS, shared_down_proj in the same
    form as w_down), the same on every rank.  route_fn(x) returns (weights,
    ids) or (weights, ids, gamma); dispatch_fn(x, ids, w, E, world) returns
    (send_x, send_ids, send_w, send_counts, inv_order); experts_fn and
    shared_fn return pair rows (hi bf16, res int8), each [rows, H] (the
    shared term: S rows per token); combine_fn(yrows, inv_order, N, k,
    yshared) returns the output.
    Returns out [N, H] bf16."""
    from sparse_moe_ffn_gb300 import binding

    world = _world(group)
    N, H = x.shape
    if route_fn is None:
        def route_fn(t):
            gate = shared["shared_gate"] if shared is not None else None
            w, ids, gamma, _ = binding.moe_route_raw(t, router, k, norm_topk_prob, gate)
            return w, ids, gamma
    if experts_fn is None:
        def experts_fn(rows, local_ids, weights):
            return binding.moe_experts(rows, local_ids, weights, w_gate, w_up, w_down)[0]
    if shared_fn is None and shared is not None:
        def shared_fn(t, gamma):
            return binding.moe_shared_expert(t, gamma, w_gate.shape[1],
                                             shared["shared_gate_proj"], shared["shared_up_proj"],
                                             shared["shared_down_proj"])[0]
    if dispatch_fn is None:
        def dispatch_fn(t, ids_, w_, E_, world_):
            d = binding.moe_ep_dispatch(t, ids_, w_, E_, world_)
            return d["send_x"], d["send_ids"], d["send_w"], d["send_counts"], d["inv_order"]
    if combine_fn is None:
        def combine_fn(yrows, inv, n, kk, yshared=None):
            return binding.moe_combine_indexed(yrows, inv, n, kk, yshared)

    routed = route_fn(x)
    w, ids = routed[0], routed[1]
    gamma = routed[2] if len(routed) > 2 else None
    # the shared term needs no exchange: it can run before the dispatch
    yshared = shared_fn(x, gamma) if shared_fn is not None else None
    send_x, send_e, send_w, send_counts, inv = dispatch_fn(x, ids, w, E, world)
    if world == 1:
        recv_x, recv_e, recv_w = send_x, send_e, send_w
    else:
        # counts first (gloo carries CPU tensors, NCCL device tensors)
        comm_dev = x.device if dist.get_backend(group) == "nccl" else torch.device("cpu")
        sc = send_counts.to(torch.int32).to(comm_dev)
        rc = torch.empty_like(sc)
        dist.all_to_all_single(rc, sc, group=group)
        send_list, recv_list = sc.tolist(), rc.tolist()
        n_send = sum(send_list)
        recv_x = _exchange(send_x[:n_send].view(torch.int32), send_list, recv_list,
                           group).view(torch.bfloat16)
        recv_e = _exchange(send_e[:n_send], send_list, recv_list, group)
        recv_w = _exchange(send_w[:n_send].view(torch.int32), send_list, recv_list,
                           group).view(torch.float32)
    y = experts_fn(recv_x, recv_e, recv_w)
    if world == 1:
        y_back = y
    else:
        y_back = (_exchange(y[0].view(torch.int32), recv_list, send_list,
                            group).view(torch.bfloat16),
                  _exchange(y[1].view(torch.int32), recv_list, send_list,
                            group).view(torch.int8))
    return combine_fn(y_back, inv, N, k, yshared)
