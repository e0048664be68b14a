"""Expert parallelism for the MoE layer: one rank per GPU, the expert stacks
sharded along their first dimension.

The InternLumina-U2 training-pitfalls article (section "专家并行（EP）怎么切")
shards the stacked expert weights W_gate_up [E, 2I, H] and W_down [E, I, H]
along the expert dimension over R ranks: rank r holds experts
[r E/R, (r + 1) E/R).  The router, its bias and the shared expert are
replicated.  Every rank routes its own batch, sends each (token, expert)
pair's hidden row to the rank that holds the expert, runs the rows it
receives through its local experts, sends the results back, and combines its
tokens' rows with their routing weights and the shared expert.

A step is three phases on each rank (ExpertShard), with two all-to-all
exchanges of rows between them:
  dispatch  moe_route + moe_ep_dispatch: routing, and the pairs' rows grouped
            by destination rank (stable: ascending (token, j) per rank);
  compute   moe_expert_rows on the rows received (unweighted expert outputs);
  finish    the shared expert (moe_dense_ffn) and moe_combine.
ep_forward runs them with torch.distributed (all_to_all_single) when every
rank is its own process; ep_forward_local runs all ranks' shards in one
process and hands the row pieces over directly (one GPU, or tests).  The
exchanges move raw bytes, so they work on any backend (NCCL on GPUs, gloo on
CPU tensors).

Every pair's expert output does not depend on the rank that computes it, and
the combine adds each token's rows in the same order as moe_forward, so the
result equals the single-GPU layer's bit for bit.

The arithmetic of every phase runs in the library's kernels (CudaOps); the
phases take an `ops` object so that the exchange logic can be exercised
against another implementation of the same five operations.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import torch

from . import moe


@dataclasses.dataclass
class Dispatched:
    """One rank's routed batch, ready to send."""
    idx: torch.Tensor          # [T, k] int32
    w: torch.Tensor            # [T, k] fp32
    send_counts: List[int]     # rows for each destination rank
    x_send: torch.Tensor       # [k T, H] bf16, grouped by destination rank
    e_send: torch.Tensor       # [k T] int32, local expert ids
    slot_of: torch.Tensor      # [T, k] int32, row of each pair in x_send


class CudaOps:
    """The five operations of an expert-parallel step in the library's CUDA
    kernels.  Each keeps its workspace across steps and grows it when a step
    needs more (the rows a rank receives change from step to step)."""

    def __init__(self, cfg: moe.MoeConfig, device):
        self.cfg = cfg
        self.device = device
        self.ws_route = moe.Workspace(cfg, 0, device)
        self.ws_dispatch = None
        self.ws_rows = None
        self.ws_dense = None

    def _sized(self, ws, need, what):
        if need and (ws is None or ws.nbytes < need):
            ws = moe.SizedWorkspace(need, what, self.device)
        return ws

    def route(self, x, W_router, W_split, expert_bias):
        idx, w, _, _, _ = moe.route(self.cfg, x, W_router, expert_bias, ws=self.ws_route, W_split=W_split)
        return idx, w

    def dispatch(self, ranks, x, idx):
        self.ws_dispatch = self._sized(self.ws_dispatch, moe.ep_dispatch_workspace_bytes(self.cfg, ranks),
                                       "moe_ep_dispatch")
        return moe.ep_dispatch(self.cfg, ranks, x, idx, ws=self.ws_dispatch)

    def expert_rows(self, cfg_local, x_recv, e_recv, W_gate_up, W_down):
        if x_recv.shape[0]:
            self.ws_rows = self._sized(self.ws_rows, moe.expert_rows_workspace_bytes(cfg_local, x_recv.shape[0]),
                                       "moe_expert_rows")
        return moe.expert_rows(cfg_local, x_recv, e_recv, W_gate_up, W_down, ws=self.ws_rows)

    def shared(self, x, shared_gate_up, shared_down, out):
        T, H = x.shape
        if self.ws_dense is None or self.ws_dense.shape != (T, H, shared_down.shape[0]):
            self.ws_dense = moe.DenseWorkspace(T, H, shared_down.shape[0], self.device)
        return moe.dense_ffn(x, shared_gate_up, shared_down, ws=self.ws_dense, out=out)

    def combine(self, Y, shared_row0, slot_of, w, residual):
        return moe.combine(self.cfg, Y, shared_row0, slot_of, w, residual)


class ExpertShard:
    """Rank `rank` of `world`: the replicated router, bias and shared expert,
    and its slice of the experts (W_gate_up_local [E/R, 2I, H], W_down_local
    [E/R, I, H]: experts rank E/R .. (rank + 1) E/R - 1)."""

    def __init__(self, cfg: moe.MoeConfig, rank: int, world: int, W_router, expert_bias, W_gate_up_local,
                 W_down_local, shared_gate_up, shared_down, ops=None):
        if cfg.E % world != 0:
            raise ValueError("E = %d experts do not split over %d ranks" % (cfg.E, world))
        self.cfg, self.rank, self.world = cfg, rank, world
        # the local experts' stage only (no routing happens on the received
        # rows); the routing fields are kept consistent for the checks
        n_group = max(1, cfg.n_group // world)
        self.cfg_local = dataclasses.replace(cfg, E=cfg.E // world, n_group=n_group,
                                             topk_group=min(cfg.topk_group, n_group))
        self.W_router, self.expert_bias = W_router, expert_bias
        self.W_gate_up_local, self.W_down_local = W_gate_up_local, W_down_local
        self.shared_gate_up, self.shared_down = shared_gate_up, shared_down
        self.ops = ops if ops is not None else CudaOps(cfg, W_router.device)
        self.W_split = moe.prepare_router(cfg, W_router) if isinstance(self.ops, CudaOps) else None

    def dispatch(self, x) -> Dispatched:
        idx, w = self.ops.route(x, self.W_router, self.W_split, self.expert_bias)
        counts, x_send, e_send, slot_of = self.ops.dispatch(self.world, x, idx)
        return Dispatched(idx, w, [int(c) for c in counts.tolist()], x_send, e_send, slot_of)

    def compute(self, x_recv, e_recv):
        return self.ops.expert_rows(self.cfg_local, x_recv, e_recv, self.W_gate_up_local, self.W_down_local)

    def result_rows(self, device):
        """The buffer finish() takes: [k T + T, H] bf16, whose first k T rows
        receive this rank's pairs' expert rows (in x_send's order)."""
        cfg = self.cfg
        return torch.empty(cfg.k * cfg.T + cfg.T, cfg.H, dtype=torch.bfloat16, device=device)

    def finish(self, x, Y, d: Dispatched, residual=None):
        """Y: result_rows() with its first k T rows filled; the shared expert
        goes into its last T rows, then the combine."""
        kT = self.cfg.k * self.cfg.T
        self.ops.shared(x, self.shared_gate_up, self.shared_down, Y[kT:])
        return self.ops.combine(Y, kT, d.slot_of, d.w, residual)


def _bytes(t):
    return t.contiguous().reshape(-1).view(torch.uint8)


def _all_to_all_rows(t, send_rows, recv_rows, group=None, out=None):
    """Rows of t ([n, ...], grouped by destination) to every rank by
    send_rows; returns the rows received, by recv_rows (source-rank order),
    in `out` when given."""
    import torch.distributed as dist
    row_bytes = t.element_size()
    for n in t.shape[1:]:
        row_bytes *= n
    if out is None:
        out = torch.empty((sum(recv_rows),) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
    dist.all_to_all_single(_bytes(out), _bytes(t), output_split_sizes=[r * row_bytes for r in recv_rows],
                           input_split_sizes=[r * row_bytes for r in send_rows], group=group)
    return out


def ep_forward(shard: ExpertShard, x, residual=None, group=None):
    """One expert-parallel layer step on this rank (every rank calls it
    together): dispatch, exchange rows and expert ids, compute, exchange the
    results back, finish."""
    import torch.distributed as dist
    d = shard.dispatch(x)
    send = torch.tensor(d.send_counts, dtype=torch.int64, device=x.device)
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv, send, group=group)
    recv_rows = [int(v) for v in recv.tolist()]
    x_recv = _all_to_all_rows(d.x_send, d.send_counts, recv_rows, group)
    e_recv = _all_to_all_rows(d.e_send, d.send_counts, recv_rows, group)
    y_recv = shard.compute(x_recv, e_recv)
    Y = shard.result_rows(x.device)
    _all_to_all_rows(y_recv, recv_rows, d.send_counts, group, out=Y[:shard.cfg.k * shard.cfg.T])
    return shard.finish(x, Y, d, residual)


def ep_forward_local(shards: List[ExpertShard], xs, residuals: Optional[list] = None):
    """All ranks of an expert-parallel layer in one process: shards[r] and
    its batch xs[r]; the exchanges are copies of row pieces.  Returns every
    rank's output."""
    R = len(shards)
    ds = [s.dispatch(x) for s, x in zip(shards, xs)]
    starts = []
    for d in ds:
        acc, st = 0, []
        for c in d.send_counts:
            st.append(acc)
            acc += c
        starts.append(st)
    # rows for rank r: every source's piece for r, sources in rank order
    y_recv = []
    for r in range(R):
        xr = torch.cat([d.x_send[starts[src][r]:starts[src][r] + d.send_counts[r]] for src, d in enumerate(ds)])
        er = torch.cat([d.e_send[starts[src][r]:starts[src][r] + d.send_counts[r]] for src, d in enumerate(ds)])
        y_recv.append(shards[r].compute(xr, er))
    outs = []
    for src, d in enumerate(ds):
        # src's rows sit, in rank r's received rows, after those of the lower sources
        pieces = []
        for r in range(R):
            o = sum(ds[s2].send_counts[r] for s2 in range(src))
            pieces.append(y_recv[r][o:o + d.send_counts[r]])
        Y = shards[src].result_rows(xs[src].device)
        torch.cat(pieces, out=Y[:len(d.e_send)])
        outs.append(shards[src].finish(xs[src], Y, d, None if residuals is None else residuals[src]))
    return outs
