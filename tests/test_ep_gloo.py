"""Expert parallelism's exchange logic on CPU ranks (gloo, world size 2).

group_limited_routing_gb300.ep splits a layer step into dispatch / compute /
finish phases around two all-to-all exchanges.  Here every phase's arithmetic
is done by HostOps (the CPU oracle for the expert rows, numpy for the
bookkeeping), so that two gloo ranks can run ep_forward on the CPU: each rank
routes its own batch, the rows travel to the rank holding their expert and
back, and the result must equal, bit for bit, the same HostOps arithmetic run
on one rank without any exchange -- and the oracle's layer output within the
layer tolerance.  The CUDA kernels of the same phases are checked against
moe_forward on the GPU (tests/test_gpu_ep.py).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

T, H, E, NG, TG, K, I = 48, 64, 32, 4, 2, 4, 32       # a tiny layer: 4 groups of 8 experts, top-2 groups, top-4


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _u16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


class HostOps:
    """The five operations of an expert-parallel step on the host."""

    def __init__(self, E, k):
        import oracle
        self.oracle, self.E, self.k = oracle, E, k

    def route(self, x, W_router, W_split, bias):
        o = self.oracle
        r = o.route(o.router_logits(_u16(x), W_router.numpy()), bias=bias.numpy(), n_group=NG, topk_group=TG, k=K)
        return torch.from_numpy(r["idx"]), torch.from_numpy(r["w"])

    def dispatch(self, ranks, x, idx):
        idx = idx.numpy()
        per = self.E // ranks
        dest = (idx // per).ravel()
        order = np.argsort(dest, kind="stable")          # pairs by rank, (token, j) ascending within one
        slot_of = np.empty(idx.size, dtype=np.int32)
        slot_of[order] = np.arange(idx.size, dtype=np.int32)
        x_send = x[torch.from_numpy(order // self.k)]
        e_send = torch.from_numpy((idx.ravel()[order] % per).astype(np.int32))
        counts = torch.from_numpy(np.bincount(dest, minlength=ranks).astype(np.int32))
        return counts, x_send, e_send, torch.from_numpy(slot_of.reshape(idx.shape))

    def expert_rows(self, cfg_local, x_recv, e_recv, Wgu, Wd):
        if x_recv.shape[0] == 0:
            return torch.empty(0, H, dtype=torch.bfloat16)
        y = self.oracle.experts(_u16(x_recv), _u16(Wgu), _u16(Wd), None, None, e_recv.numpy()[:, None],
                                np.ones((x_recv.shape[0], 1), dtype=np.float32))
        return torch.from_numpy(y).to(torch.bfloat16)

    def shared(self, x, sgu, sd, out):
        out.copy_(torch.from_numpy(self.oracle.dense_ffn(_u16(x), _u16(sgu), _u16(sd))).to(torch.bfloat16))
        return out

    def combine(self, Y, shared_row0, slot_of, w, residual):
        acc = torch.zeros(slot_of.shape[0], Y.shape[1], dtype=torch.float32)
        for j in range(slot_of.shape[1]):
            acc += w[:, j:j + 1] * Y[slot_of[:, j].long()].float()
        acc += Y[shared_row0:shared_row0 + slot_of.shape[0]].float()
        if residual is not None:
            acc += residual.float()
        return acc.to(torch.bfloat16)


def _layer(seed):
    g = torch.Generator().manual_seed(seed)
    return dict(W_router=torch.randn(E, H, generator=g) * 0.1,
                bias=(torch.rand(E, generator=g) - 0.5) * 0.02,
                Wgu=(torch.randn(E, 2 * I, H, generator=g) * 0.05).to(torch.bfloat16),
                Wd=(torch.randn(E, I, H, generator=g) * 0.05).to(torch.bfloat16),
                sgu=(torch.randn(2 * I, H, generator=g) * 0.05).to(torch.bfloat16),
                sd=(torch.randn(I, H, generator=g) * 0.05).to(torch.bfloat16))


def _batch(rank):
    return torch.randn(T, H, generator=torch.Generator().manual_seed(100 + rank)).to(torch.bfloat16)


def _shard(rank, world, L):
    from group_limited_routing_gb300 import ep, moe
    cfg = moe.MoeConfig(T=T, H=H, E=E, n_group=NG, topk_group=TG, k=K, I=I, Is=I)
    per = E // world
    return ep.ExpertShard(cfg, rank, world, L["W_router"], L["bias"], L["Wgu"][rank * per:(rank + 1) * per],
                          L["Wd"][rank * per:(rank + 1) * per], L["sgu"], L["sd"], ops=HostOps(E, K))


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import torch.distributed as dist
    from group_limited_routing_gb300 import ep

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        L = _layer(7)
        out = ep.ep_forward(_shard(rank, world, L), _batch(rank))
        q.put((rank, _u16(out).tobytes()))
    finally:
        dist.destroy_process_group()


def _single_rank_reference(rank):
    """The same HostOps arithmetic with every expert on one rank and no exchange."""
    from group_limited_routing_gb300 import ep
    L = _layer(7)
    return ep.ep_forward_local([_shard(0, 1, L)], [_batch(rank)])[0]


def test_two_gloo_ranks_equal_one_rank_bit_for_bit():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(world))
    for rank in range(world):
        ref = _u16(_single_rank_reference(rank)).tobytes()
        assert got[rank] == ref, "rank %d differs from the single-rank result" % rank


@pytest.mark.parametrize("world", [2, 4])
def test_local_driver_matches_the_oracle_layer(world):
    """All ranks in one process (ep_forward_local): every rank's output is
    the oracle's layer output for its batch within the layer tolerance, and
    equals the one-rank result bit for bit."""
    import oracle
    from group_limited_routing_gb300 import ep
    from parity import assert_output_close
    L = _layer(8)
    shards = [_shard(r, world, L) for r in range(world)]
    xs = [_batch(r) for r in range(world)]
    outs = ep.ep_forward_local(shards, xs)
    one = _shard(0, 1, L)
    for r in range(world):
        ref1 = ep.ep_forward_local([one], [xs[r]])[0]
        assert torch.equal(outs[r], ref1)
        idx, w = HostOps(E, K).route(xs[r], L["W_router"], None, L["bias"])
        ref = oracle.experts(_u16(xs[r]), _u16(L["Wgu"]), _u16(L["Wd"]), _u16(L["sgu"]), _u16(L["sd"]),
                             idx.numpy(), w.numpy())
        assert_output_close(outs[r].double().numpy(), ref, "EP rank %d of %d" % (r, world))


def test_shard_rejects_an_uneven_split():
    from group_limited_routing_gb300 import ep, moe
    L = _layer(9)
    cfg = moe.MoeConfig(T=T, H=H, E=E, n_group=NG, topk_group=TG, k=K, I=I, Is=I)
    with pytest.raises(ValueError):
        ep.ExpertShard(cfg, 0, 3, L["W_router"], L["bias"], L["Wgu"], L["Wd"], L["sgu"], L["sd"],
                       ops=HostOps(E, K))
