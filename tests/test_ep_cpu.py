"""Expert parallelism on CPU ranks (gloo, world size 2, no GPU): the partition of
the routed experts and the data plane of mxfp4_expert_ffn_gb300.ep, with the
compute steps played by the fp64 oracle.  Each rank computes the share of y of
its own experts (the shared expert on rank 0), the shares are exchanged and
added in rank order, and every rank's tokens must come out as the oracle's
whole layer on the same routing."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from mxfp4_expert_ffn_gb300 import ep  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_expert_ranges_partition_the_experts():
    for E, R in [(16, 2), (384, 8), (385, 4), (7, 7), (10, 3)]:
        rg = ep.expert_ranges(E, R)
        assert rg[0][0] == 0 and rg[-1][1] == E
        assert all(a[1] == b[0] for a, b in zip(rg, rg[1:]))
        sizes = [hi - lo for lo, hi in rg]
        assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
        for e in range(E):
            lo, hi = rg[ep.owner_of_expert(e, rg)]
            assert lo <= e < hi
    with pytest.raises(ValueError):
        ep.expert_ranges(3, 4)


def _oracle_fns(wl, rank, ranges, touched):
    """The three compute steps by the oracle, as a rank would run them."""
    import oracle
    import synth
    lo, hi = ranges[rank]
    H, E = wl.hidden, wl.n_experts

    def route(x_all):
        xb = x_all.numpy().view(np.uint16)
        lg = oracle.router_logits(xb, synth.router_weights(wl), synth.router_bias(wl))
        idx, w = oracle.topk(lg, wl.top_k)
        return torch.from_numpy(idx), torch.from_numpy(w.astype(np.float32))

    def partial(x_all, idx, w):
        xb = x_all.numpy().view(np.uint16)
        xq, xs = oracle.quantize_act(xb)
        ids, ws = idx.numpy(), w.numpy().astype(np.float64)
        share = np.zeros((xb.shape[0], H), np.float64)
        shared = [synth.host_expert(wl, 0, E + s) for s in range(wl.n_shared)] if rank == 0 else []
        cache = {}
        for t in range(xb.shape[0]):
            for ex in shared:  # the shared experts first, then the slots in rank order
                share[t] += oracle.expert_ffn(ex, xq[t], xs[t])["o"]
            for j in range(ids.shape[1]):
                e = int(ids[t, j])
                if not lo <= e < hi:
                    continue
                touched.add(e)
                if e not in cache:
                    cache[e] = synth.host_expert(wl, 0, e)
                share[t] += ws[t, j] * oracle.expert_ffn(cache[e], xq[t], xs[t])["o"]
        return torch.from_numpy(share.astype(np.float32))

    def combine(shares, residual):
        import synth as sy
        acc = np.zeros(shares.shape[1:], np.float32)
        for r in range(shares.shape[0]):  # rank order, fp32 as the library adds them
            acc = acc + shares[r].numpy()
        y = sy.f32_to_bf16_bits(acc)
        return torch.from_numpy(y.view(np.int16))

    return route, partial, combine


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import synth
    from synth.workloads import TINY
    wl = TINY  # hidden 256, 16 routed experts top-2 + 1 shared, 4 tokens per rank
    ranges = ep.expert_ranges(wl.n_experts, world)
    x_local = synth.activations(wl, stream=70 + rank)  # this rank's own batch
    touched: set = set()
    route, partial, combine = _oracle_fns(wl, rank, ranges, touched)
    y = ep.ep_layer_step(dist, torch.from_numpy(x_local.view(np.int16)), route, partial, combine)
    out.put((rank, y.numpy().view(np.uint16).copy(), sorted(touched)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_match_the_oracle_layer():
    import oracle
    import synth
    from synth.workloads import TINY as wl
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # the whole batch on one process, by the oracle
    x_all = np.concatenate([synth.activations(wl, stream=70 + r) for r in range(world)])
    lg = oracle.router_logits(x_all, synth.router_weights(wl), synth.router_bias(wl))
    idx, w = oracle.topk(lg, wl.top_k)
    experts = {int(e): synth.host_expert(wl, 0, int(e)) for e in np.unique(idx)}
    shared = [synth.host_expert(wl, 0, wl.n_experts + s) for s in range(wl.n_shared)]
    ref, _ = oracle.moe_layer(x_all, idx, w, experts, shared, wl.n_experts, wl.inter)
    ranges = ep.expert_ranges(wl.n_experts, world)
    T = wl.tokens
    for rank, y, touched in res:
        lo, hi = ranges[rank]
        assert all(lo <= e < hi for e in touched), "a rank computed another rank's expert"
        want = synth.bf16_bits_to_f32(ref[rank * T:(rank + 1) * T]).astype(np.float64)
        got = synth.bf16_bits_to_f32(y).astype(np.float64)
        err = np.abs(got - want).max()
        assert err <= 2e-2 * np.abs(want).max()
        assert np.linalg.norm(got - want) <= 5e-3 * np.linalg.norm(want)
    # between them the ranks computed every routed expert the batch selects
    assert sorted(set(res[0][2]) | set(res[1][2])) == sorted(int(e) for e in np.unique(idx))
