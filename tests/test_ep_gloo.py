"""Expert-parallel dispatch and combine (sparse_moe_ffn_gb300/ep.py) on CPU
ranks: two gloo processes, each routing its own tokens, with stand-in
compute steps (a per-pair function of the token row, the global expert id
and the weight; a slot-order fp32 sum).  Every rank's output must equal the
same stand-ins applied pair by pair without any exchange, bit for bit, also
when E does not split evenly and when a rank receives no pairs."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from sparse_moe_ffn_gb300.ep import ep_dispatch_reference, ep_plan


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rows(v):
    """Stand-in pair rows of values v: a bf16 plane and an int8 plane that
    both depend on v (the exchange must carry both bit for bit)."""
    hi = v.to(torch.bfloat16)
    res = ((v - hi.float()) * 4096).round().clamp(-127, 127).to(torch.int8)
    return hi, res


def _pair_value(row, e, w):
    """Stand-in for w * Expert_e(row): any function of all three inputs."""
    return (w * (row.float() * (e + 1) + e)).to(torch.float32)


def _combine(ypair, n, k, yshared=None):
    def val(y):
        return y[0].float() + y[1].float() / 4096
    acc = val(ypair).view(n, k, -1).sum(dim=1)
    if yshared is not None:
        acc = acc + val(yshared)
    return acc.to(torch.bfloat16)


def _combine_rows(yrows, inv, n, k, yshared=None):
    """Stand-in combine over rows in send order: pair p reads row inv[p]."""
    idx = inv.long()
    return _combine((yrows[0][idx], yrows[1][idx]), n, k, yshared)


def _shared_value(x, gamma):
    """Stand-in for gamma * SharedMLP(x), token-local."""
    return _rows((gamma[:, None] * (0.5 * x.float() - 1.0)).to(torch.float32))


def _inputs(rank, N, H, E, k, all_to_rank0):
    g = torch.Generator().manual_seed(100 + rank)
    x = torch.randn(N, H, generator=g).to(torch.bfloat16)
    scores = torch.rand(N, E, generator=g)
    if all_to_rank0:  # only experts of rank 0 ever chosen
        scores[:, (E + 1) // 2:] = -1.0
    ids = scores.topk(k, dim=1).indices.to(torch.int32)
    w = torch.rand(N, k, generator=g)
    return x, ids, w


def _worker(rank, world, port, q, N, H, E, k, all_to_rank0, with_shared=False):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from sparse_moe_ffn_gb300.ep import ep_dispatch_reference, ep_forward
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x, ids, w = _inputs(rank, N, H, E, k, all_to_rank0)
        E_local = -(-E // world)
        calls = []

        def experts_fn(rows, local_ids, weights):
            calls.append(rows.shape[0])
            if local_ids.numel():
                assert int(local_ids.min()) >= 0 and int(local_ids.max()) < E_local
            ge = local_ids.long() + rank * E_local
            return _rows(torch.stack([_pair_value(rows[i], int(ge[i]), float(weights[i]))
                                      for i in range(rows.shape[0])]) if rows.shape[0] else
                         torch.empty((0, H), dtype=torch.float32))

        gamma = torch.sigmoid(x.float()[:, 0]) if with_shared else None
        out = ep_forward(x, None, None, None, None, E, k, group=None,
                         route_fn=lambda t: (w, ids, gamma), experts_fn=experts_fn,
                         shared_fn=_shared_value if with_shared else None,
                         dispatch_fn=ep_dispatch_reference, combine_fn=_combine_rows)
        ref_pairs = _rows(torch.stack([_pair_value(x[p // k], int(ids.view(-1)[p]),
                                                   float(w.view(-1)[p])) for p in range(N * k)]))
        ref = _combine(ref_pairs, N, k, _shared_value(x, gamma) if with_shared else None)
        q.put((rank, bool(torch.equal(out, ref)), calls[0]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("N,H,E,k,all_to_rank0,with_shared",
                         [(12, 16, 6, 2, False, False), (9, 8, 5, 3, False, False),
                          (7, 16, 6, 2, True, False), (10, 16, 6, 2, False, True)])
def test_two_ranks_match_the_unsplit_layer(N, H, E, k, all_to_rank0, with_shared):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker,
                         args=(r, world, port, q, N, H, E, k, all_to_rank0, with_shared))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = dict((r, (ok, n)) for r, ok, n in (q.get(timeout=5) for _ in range(world)))
    assert got[0][0] and got[1][0], got
    if all_to_rank0:
        assert got[1][1] == 0  # rank 1 received no pairs


def test_plan_orders_pairs_by_destination_rank():
    ids = torch.tensor([[4, 0], [1, 5], [2, 3]], dtype=torch.int32)
    order, dest, counts, E_local = ep_plan(ids, E=6, world=2)
    assert E_local == 3
    assert dest.tolist() == [1, 0, 0, 1, 0, 1]
    assert order.tolist() == [1, 2, 4, 0, 3, 5]  # stable within each rank
    assert counts.tolist() == [3, 3]
    with pytest.raises(ValueError):
        ep_plan(torch.tensor([[6]], dtype=torch.int32), E=6, world=2)


@pytest.mark.parametrize("world", [1, 2, 3, 5, 8])
def test_plan_properties_on_random_routing(world):
    """For any routing table: the send order is a permutation of the pairs,
    grouped by destination rank in rank order, in pair order within a rank;
    every pair goes to the rank that owns its expert; counts add up."""
    g = torch.Generator().manual_seed(world)
    for N, k, E in [(1, 1, 1), (33, 4, 7), (64, 8, 128), (5, 3, 3)]:
        ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(N)]).to(torch.int32)
        order, dest, counts, E_local = ep_plan(ids, E, world)
        flat = ids.reshape(-1).long()
        assert E_local == -(-E // world)  # ceil(E / world); trailing ranks may own none
        assert sorted(order.tolist()) == list(range(N * k))
        assert torch.equal(dest, flat // E_local) and int(dest.max()) < world
        d_sorted = dest[order]
        assert torch.all(d_sorted[1:] >= d_sorted[:-1])
        for r in range(world):
            mine = order[d_sorted == r]
            assert torch.all(mine[1:] > mine[:-1])  # stable: pair order within a rank
        assert counts.tolist() == [int((dest == r).sum()) for r in range(world)]


def test_reference_dispatch_packs_rows_in_send_order():
    """The host reference of the dispatch plan: send row i is pair order[i]
    (its token row, local expert id and weight), and inv_order inverts the
    order, so reading row inv[p] gives pair p back."""
    g = torch.Generator().manual_seed(7)
    N, H, E, k, world = 9, 8, 7, 3, 3
    x = torch.randn(N, H, generator=g).to(torch.bfloat16)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(N)]).to(torch.int32)
    w = torch.rand(N, k, generator=g)
    send_x, send_e, send_w, counts, inv = ep_dispatch_reference(x, ids, w, E, world)
    order, dest, _, E_local = ep_plan(ids, E, world)
    assert counts.tolist() == [int((dest == r).sum()) for r in range(world)]
    for p in range(N * k):
        i = int(inv[p])
        assert int(order[i]) == p
        assert torch.equal(send_x[i], x[p // k])
        assert int(send_e[i]) == int(ids.view(-1)[p]) - int(dest[p]) * E_local
        assert float(send_w[i]) == float(w.view(-1)[p])
