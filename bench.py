"""Benchmark of the GB300 MoE layer forward (route + expert stage).

One step = the layer forward (moe_layer: routing and the expert stage in one
call; --two-call: moe_route + moe_forward) over one batch of T tokens of the full-size
skewed workload (T=32768, hidden 2048, 256 experts in 8 groups, top-4 groups,
top-8, SwiGLU experts [256, 512, 2048], one shared expert, 16 hot experts with
router rows x3 and expert_bias ~ N(0, 0.05)).  Inputs are seeded synthetic
tensors already resident in HBM; they are larger than L2 (1.61 GB of expert
weights and 134 MB of hidden states per step), so no L2 flush is needed.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle (the
plain C reference of the same method) on a bounded sample of the same
workload.  Multi-GPU (torchrun): every rank runs its own replica on its own
batch (weak scaling, no collective on the data path); the step time is the
maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "MoE layer fwd tokens/s on 1 GB300; % of tensor/HBM roofline per stage"
WORKLOAD_ID = 4


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def gemm_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when the GEMM sources have changed since that capture."""
    import hashlib
    csrc = os.path.join(ROOT, "group_limited_routing_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("gemm.cu", "ptx.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    try:
        with open(os.path.join(ROOT, "profiles", "gemm_dram_traffic_T32768.md")) as fh:
            text = fh.read()
    except OSError:
        return None
    tags = dict(line.split(": ", 1) for line in text.splitlines() if line.startswith(("gemm-source", "traffic-")))
    if tags.get("gemm-source-sha256-16") != h.hexdigest()[:16]:
        return None
    v = tags.get("traffic-" + kernel)
    return int(v) if v else None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 100 ms; summary() keeps those taken between
    mark('load') (start of the untimed loaded lead-in) and mark('end') (end of
    the timed region)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            sel = str(device_index)
        self.sel = sel

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.sel, "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark(self, name: str) -> None:
        """Record when the loaded window ('load') and the timed region ('end') start/finish."""
        setattr(self, "t_" + name, time.monotonic())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        t0 = getattr(self, "t_load", None)
        t1 = getattr(self, "t_end", None)
        for t, ln in self.lines:
            if t0 is not None and t1 is not None and not (t0 <= t <= t1 + 0.15):
                continue                  # only samples taken while the GPU ran the step
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------- work
def dense_work(T, H, I):
    """Algorithmic work of the dense MLP: its two GEMMs and the final copy."""
    return {
        "gemm_gate_up_swiglu": dict(bound="tensor", flops=2.0 * T * H * 2 * I,
                                    bytes=T * H * 2 + 2 * I * H * 2 + T * I * 2),
        "gemm_down": dict(bound="tensor", flops=2.0 * T * I * H, bytes=T * I * 2 + I * H * 2 + T * H * 2),
        "combine": dict(bound="hbm", bytes=T * H * 2 * 2),
    }


def algorithmic_work(T, H, E, I, k, hit=None, Is=None):
    """Per-launch algorithmic bytes / flops of each kernel (the method's own
    work: bytes every stage must move at least once, flops of the products).
    The grouped GEMMs read the weights of the `hit` experts that received at
    least one token (all E unless given) plus the shared expert's; each GEMM
    is reported against the roofline that binds it at this size (HBM when its
    bytes take longer at the measured copy rate than its flops at the
    measured sustained tensor rate)."""
    kT = k * T
    hit = E if hit is None else hit
    Is = I if Is is None else Is
    work = {
        # T <= 32: the CUDA-core router, which streams the fp32 weight once (HBM-bound)
        "router_gemm": dict(bound="hbm" if T <= 32 else "tensor", flops=2.0 * T * E * H,
                            bytes=T * H * 2 + E * H * 4 + T * E * 4),
        "route_select": dict(bound="hbm", bytes=T * E * 4 + T * k * 8),
        # the fused router: the router's hidden and weight reads, the routing
        # outputs, the pairs' bucket rows and the copied rows
        "router_route_bucket": dict(bound="hbm", bytes=T * H * 2 + E * H * 4 + T * k * 8 + T * k * 4 + kT * H * 2),
        "bucket_scatter": dict(bound="hbm", bytes=T * k * 4 * 2 + T * H * 2 + kT * H * 2),
        "gemm_gate_up_swiglu": dict(flops=2.0 * kT * H * 2 * I + 2.0 * T * H * 2 * Is,
                                    bytes=(kT + T) * H * 2 + (hit * I + Is) * 2 * H * 2 + kT * I * 2 + T * Is * 2),
        "gemm_down": dict(flops=2.0 * kT * I * H + 2.0 * T * Is * H,
                          bytes=kT * I * 2 + T * Is * 2 + (hit * I + Is) * H * 2 + (kT + T) * H * 2),
        "combine": dict(bound="hbm", bytes=(kT + T) * H * 2 + T * H * 2 + T * k * 8),
    }
    pk = peaks()
    for name in ("gemm_gate_up_swiglu", "gemm_down"):
        wk = work[name]
        t_hbm = wk["bytes"] / (pk["hbm"] * 1e9)
        t_tensor = wk["flops"] / (pk["bf16_sustained"] * 1e12)
        wk["bound"] = "hbm" if t_hbm > t_tensor else "tensor"
    return work


def workload_name(w0, dense=0, backward=False):
    if backward:
        return "backward of: " + workload_name_moe(w0)
    if dense:
        return "dense first-layer SwiGLU MLP, T=%d, H=%d, I=%d (size assumed)" % (w0.T, w0.H, dense)
    return workload_name_moe(w0)


def workload_name_moe(w0):
    if w0.wid in (4, 6):
        return "T=%d full-size layer, 16 hot experts (router rows x%g), expert_bias~N(0,0.05)" % (w0.T, w0.hot_scale)
    if w0.wid == 5:
        return ("%d-layer stack (x + moe(rmsnorm(x))), T=%d, full size, per-layer expert counts and balance loss"
                % (w0.layers, w0.T))
    return "%s (T=%d)" % (w0.name, w0.T)


def init_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value, device):
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- CPU oracle
class CpuSample:
    """The workload's inputs on the host (drawn once) and a timer of the CPU
    oracle -- router logits, routing and expert stage -- on its first n tokens."""

    def __init__(self, workload: int = WORKLOAD_ID, threads: int = 0):
        import oracle
        from group_limited_routing_gb300 import workloads as wl

        self.oracle = oracle
        if threads:
            oracle.set_threads(threads)
        w0 = wl.WORKLOADS[workload]
        self.layers = w0.layers     # a stack is timed on its first layer: rate / layers

        def u16(t):
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)

        self.x = u16(wl.hidden(w0))
        self.W = wl.router_weight(w0).numpy()
        self.b = wl.expert_bias(w0).numpy()
        Wgu, Wd = wl.expert_weights(w0)
        sgu, sd = wl.shared_weights(w0)
        self.gu, self.dn, self.sgu, self.sd = u16(Wgu), u16(Wd), u16(sgu), u16(sd)

    def run(self, n_tokens: int):
        """Returns (tokens/s, threads used, seconds)."""
        o = self.oracle
        xs = np.ascontiguousarray(self.x[:n_tokens])
        t0 = time.perf_counter()
        L = o.router_logits(xs, self.W)
        r = o.route(L, bias=self.b)
        o.experts(xs, self.gu, self.dn, self.sgu, self.sd, r["idx"], r["w"])
        dt = time.perf_counter() - t0
        return n_tokens / dt / self.layers, o.max_threads(), dt


def routing_parity(x, layer, tol=1e-5):
    """The bench batch's routing against the CPU oracle's, over every token
    (part of the CPU-oracle leg: the oracle recomputes the fp32 logits and the
    selection from the GPU run's own inputs).  Tokens whose oracle margin at
    the group (4th/5th) or expert (8th/9th) boundary is below tol are counted
    as near ties; tokens whose chosen set is clear but whose order inside it
    hangs on a gap below tol, as order ties; each class with how many of its
    tokens the GPU answered differently.  `exact_elsewhere` is whether every
    other token's indices are bit-identical."""
    import oracle

    def u16(t):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    if getattr(layer, "layers", None):
        layer = layer.layers[0]          # a stack: its first layer sees the bench input itself
    if getattr(layer, "routing", None) is None:
        return None
    t0 = time.perf_counter()
    bias = None if layer.expert_bias is None else layer.expert_bias.detach().cpu().numpy()
    L = oracle.router_logits(u16(x), layer.W_router.detach().cpu().numpy())
    c = layer.cfg
    ref = oracle.route(L, bias=bias, n_group=c.n_group, topk_group=c.topk_group, k=c.k, rsf=c.rsf, eps=c.eps)
    gi = layer.routing[0].cpu().numpy()
    gw = layer.routing[1].cpu().numpy().astype(np.float64)
    near = (ref["margin_group"] < tol) | (ref["margin_expert"] < tol)
    b = (ref["scores"] + (np.float32(0) if bias is None else bias.astype(np.float32))).astype(np.float32)
    bs = np.take_along_axis(b, ref["idx"].astype(np.int64), axis=1).astype(np.float64)
    order = (~near) & ((bs[:, :-1] - bs[:, 1:]).min(axis=1) < tol) if c.k > 1 else np.zeros_like(near)
    rest = ~near & ~order
    differs = (gi != ref["idx"]).any(axis=1)
    T = gi.shape[0]
    return {"tokens": int(T), "tol": tol,
            "near_tie_tokens": int(near.sum()), "near_tie_pct": round(100.0 * near.sum() / T, 4),
            "near_tie_differ": int((near & differs).sum()),
            "order_tie_tokens": int(order.sum()), "order_tie_pct": round(100.0 * order.sum() / T, 4),
            "order_tie_differ": int((order & differs).sum()),
            "exact_elsewhere": bool(not differs[rest].any()),
            "max_w_err_elsewhere": float(np.abs(gw[rest] - ref["w"][rest]).max()) if rest.any() else 0.0,
            "oracle_s": round(time.perf_counter() - t0, 1)}


# ------------------------------------------------------------------- ours
class BackwardStep:
    """The layer's backward as the timed step: routing and d_out fixed (one
    forward call routes the batch); __call__ runs moe_backward into
    preallocated gradients."""

    def __init__(self, layer, x, seed=99):
        self.layer = layer
        self.cfg = layer.cfg
        self.device = layer.device
        layer(x)
        g = torch.Generator(device=x.device)
        g.manual_seed(seed)
        self.d_out = torch.randn(x.shape, generator=g, device=x.device).to(torch.bfloat16)
        self.grads = layer.backward(self.d_out)
        self.last_launches = 0

    def __call__(self, x, out=None):
        from group_limited_routing_gb300 import moe
        if out is not None:
            self.grads["d_hidden"] = out
        L = self.layer
        moe.backward(L.cfg, x, L.W_gate_up, L.W_down, L.shared_gate_up, L.shared_down, L.routing[0], L.routing[1],
                     self.d_out, ws=L.ws_bwd, out=self.grads)
        self.last_launches = moe.last_launch_count()
        return self.grads["d_hidden"]

    def status(self):
        return self.layer.status()


def backward_work(T, H, E, I, k):
    """Algorithmic work per launch of the backward's kernels (weight-gradient
    GEMMs: the mean of its two launches, dW_down and dW_gate_up)."""
    R = (k + 1) * T
    return {
        "bwd_gate_up_recompute": dict(bound="tensor", flops=2.0 * R * H * 2 * I, bytes=R * H * 2 + 3 * E * I * H * 2),
        "bwd_dgrad_down_swiglu": dict(bound="tensor", flops=2.0 * R * H * I, bytes=R * H * 2 + E * I * H * 2),
        "bwd_dgrad_x": dict(bound="tensor", flops=2.0 * R * 2 * I * H, bytes=R * 2 * I * 2 + 2 * E * I * H * 2),
        "bwd_weight_grads": dict(bound="tensor", flops=3.0 * R * I * H, bytes=R * H * 2 + 3 * E * I * H * 2),
        "combine": dict(bound="hbm", bytes=R * H * 2 + T * H * 2 + T * k * 4),
    }


def build_model(w0, dev, dense_inter=0, fused_router=False, two_call=False):
    """The step's model: one MoE layer, the 19-layer stack of workload 5, or
    (dense_inter > 0) the dense first-layer MLP of that intermediate size.
    fused_router: one moe_layer call per step with the fused router (routing
    and bucketing inside the router kernel) instead of moe_route + moe_forward."""
    from group_limited_routing_gb300 import moe, workloads as wl

    if dense_inter:
        g = torch.Generator(device=dev)
        g.manual_seed(7000 + dense_inter)
        gu = (torch.randn(2 * dense_inter, w0.H, generator=g, device=dev) * 0.02).to(torch.bfloat16)
        dn = (torch.randn(dense_inter, w0.H, generator=g, device=dev) * 0.02).to(torch.bfloat16)
        return None, moe.DenseLayer(gu, dn, w0.T)

    cfg = moe.MoeConfig(T=w0.T, H=w0.H, E=w0.E, n_group=w0.n_group, topk_group=w0.topk_group, k=w0.k, I=w0.I,
                        Is=w0.Is)
    if fused_router:
        if w0.layers > 1:
            raise SystemExit("--fused-router runs single layers (the stack needs the balance loss)")
        from group_limited_routing_gb300 import _lib
        d = wl.layer_inputs(w0, dev)
        return cfg, moe.MoELayer(cfg, d["W_router"], d["expert_bias"], d["W_gate_up"], d["W_down"],
                                 d["shared_gate_up"], d["shared_down"], single_call=True,
                                 flags=_lib.MOE_LAYER_FUSED_ROUTER)
    # one moe_layer call per layer and step (two_call: moe_route + moe_forward)
    ws = dict(ws_route=moe.Workspace(cfg, 0, dev), ws_fwd=moe.Workspace(cfg, 1, dev)) if two_call else \
        dict(ws_layer=moe.Workspace(cfg, moe.WS_LAYER, dev))
    layers = []
    # the 19-layer stack workload also computes every layer's balance loss
    # (E * sum_i f_i P_i from the router scores) beside its expert counts
    for layer in range(w0.layers):
        d = wl.layer_inputs(w0, dev, layer=layer)
        layers.append(moe.MoELayer(cfg, d["W_router"], d["expert_bias"], d["W_gate_up"], d["W_down"],
                                   d["shared_gate_up"], d["shared_down"], aux=w0.layers > 1,
                                   single_call=not two_call, **ws))
    return cfg, (moe.MoEStack(layers) if w0.layers > 1 else layers[0])


def run_ours(args, world, rank, local):
    from group_limited_routing_gb300 import moe, workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w0 = wl.WORKLOADS[args.workload]
    if args.tokens:
        w0 = w0.with_T(args.tokens)
    T, H, E, I, k = w0.T, w0.H, w0.E, w0.I, w0.k
    cfg, layer = build_model(w0, dev, args.dense, args.fused_router, args.two_call)
    x = wl.hidden(w0, dev, layer=rank)      # each replica its own batch
    if args.backward:
        layer = BackwardStep(layer, x)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        layer(x, out=out)
    torch.cuda.synchronize(dev)
    if layer.status() != 0:
        raise RuntimeError("device status after warm-up: %d" % layer.status())

    # ---- timed region: K steps, inputs resident.  It follows ~0.5 s of untimed
    # steps so that clocks and power are in their loaded state and sampled.
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    layer(x, out=out)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    lead = max(1, min(2000, int(args.lead_in_ms / max(e0.elapsed_time(e1), 1e-3))))
    flush = args.flush_l2 or w0.wid == 1
    scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None
    launches = 0
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        time.sleep(0.25)
        clk.mark("load")
        for _ in range(lead):
            layer(x, out=out)
        if flush:
            # per-step events with a 256 MB scrub of L2 between steps (not timed)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            for a, b in evs:
                scrub.zero_()
                a.record(stream)
                layer(x, out=out)
                b.record(stream)
                launches += layer.last_launches
            torch.cuda.synchronize(dev)
            ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
        else:
            e0.record(stream)
            for _ in range(args.steps):
                layer(x, out=out)
                launches += layer.last_launches
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1) / args.steps
        clk.mark("end")
    barrier(world)
    ms_max = max_over_ranks(world, ms, dev)
    status = layer.status()
    if status != 0:
        raise RuntimeError("device status after the timed region: %d" % status)

    # ---- per-kernel durations (CUDA events around each launch, same stream)
    moe.profile_read(reset=True)
    moe.profile_enable(True)
    nprof = max(3, min(args.steps, 10))
    for _ in range(nprof):
        layer(x, out=out)
    torch.cuda.synchronize(dev)
    moe.profile_enable(False)
    prof = moe.profile_read(reset=True)
    # the same steps timed per stage: the routing and bucketing kernels as one
    # interval (their launches still overlap each other as in the timed loop)
    moe.profile_enable(True, stages=True)
    for _ in range(nprof):
        layer(x, out=out)
    torch.cuda.synchronize(dev)
    moe.profile_enable(False)
    sprof = moe.profile_read(reset=True)
    rp_stage = sprof.get("router_plus_permute", (0.0, 0))

    # ---- the same step replayed from a CUDA graph (no host work per step)
    graph_ms = None
    if not args.no_graph and not flush:
        g = moe.GraphedStep(layer, x)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        graph_ms = max_over_ranks(world, e0.elapsed_time(e1) / args.steps, dev)
        if g.status() != 0:
            raise RuntimeError("device status after the graph replays: %d" % g.status())
        del g

    # ---- end to end through the public API: pinned host in, pinned host out
    e2e_ms = None
    if not args.no_e2e and not args.backward:
        e2e_ms = time_e2e(args, world, layer, x, out, stream, dev)

    if rank != 0:
        return None
    hot = wl.hot_experts(w0)
    hot_share = None
    if hot.numel() and getattr(layer, "routing", None) is not None:
        counts = layer.routing[2].double().cpu()
        hot_share = float(counts[hot].sum() / counts.sum())
    # experts that received tokens (their weights are what the GEMMs stream), mean over layers
    moe_layers = getattr(layer, "layers", None) or [layer]
    hits = [int((l.routing[2] > 0).sum().item()) for l in moe_layers if getattr(l, "routing", None) is not None]
    hit = statistics.mean(hits) if hits else None
    line = report(args, world, w0, ms_max, prof, nprof * w0.layers, e2e_ms, launches, clk,
                  dict(flush=flush, lead=lead, hot_share=hot_share, graph_ms=graph_ms, dense=args.dense,
                       backward=args.backward, hit=hit,
                       rp_stage_ms=rp_stage[0] / rp_stage[1] if rp_stage[1] else None))
    if world == 1 and not args.no_cpu_baseline and not args.dense and not args.backward:
        # the CPU-oracle leg also checks the timed batch's routing, token by token
        line["parity"] = routing_parity(x, layer)
    return line


def time_e2e(args, world, layer, x, out, stream, dev):
    """Whole-job tokens/s through the public API with host buffers: every step
    uploads its batch from pinned host memory and downloads its output to
    pinned host memory; moe.HostPipeline overlaps those copies with the
    kernels of the neighbouring steps."""
    from group_limited_routing_gb300 import moe

    T, H = x.shape
    x_h = torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True)
    x_h.copy_(x)
    outs_h = [torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    pipe = moe.HostPipeline(layer)
    # warm-up of ~0.5 s: the first passes over freshly pinned host pages run
    # well below the steady copy rate, so they are kept out of the timing
    t_end = time.perf_counter() + 0.5
    while True:
        pipe.run([x_h] * 4, [outs_h[i % 2] for i in range(4)])
        torch.cuda.synchronize(dev)
        if time.perf_counter() > t_end:
            break
    barrier(world)
    # three timed passes of K steps, the median reported: the host <-> device
    # copy rate of this machine drops now and then by a third (host memory
    # shared with other jobs), which a single pass would report as ours
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    passes = []
    for _ in range(3):
        f0.record(stream)
        pipe.run([x_h] * args.steps, [outs_h[i % 2] for i in range(args.steps)])
        f1.record(stream)
        torch.cuda.synchronize(dev)
        passes.append(f0.elapsed_time(f1) / args.steps)
    e2e_ms = max_over_ranks(world, statistics.median(passes), dev)
    barrier(world)
    return e2e_ms


def report(args, world, w0, ms_max, prof, nprof, e2e_ms, launches, clk, extra):
    """nprof = layer-steps profiled (steps x layers): per-stage numbers are per layer."""
    T, H, E, I, k = w0.T, w0.H, w0.E, w0.I, w0.k
    pk = peaks()
    if extra["backward"]:
        work = backward_work(T, H, E, I, k)
    elif extra["dense"]:
        work = dense_work(T, H, extra["dense"])
    else:
        work = algorithmic_work(T, H, E, I, k, hit=extra.get("hit"), Is=w0.Is)
    stages = {}
    for name, (tot, n) in prof.items():
        if n == 0:
            continue
        avg = tot / n
        st = {"ms": round(avg, 4), "launches_per_step": round(n / nprof, 2)}
        if name in work:
            wk = work[name]
            st["bound"] = wk["bound"]
            if "flops" in wk:
                tf = wk["flops"] / (avg * 1e-3) / 1e12
                st["tflops"] = round(tf, 1)
            gb = wk["bytes"] / (avg * 1e-3) / 1e9
            st["gbs"] = round(gb, 1)
            st["frac"] = round(tf / pk["bf16_sustained"], 4) if wk["bound"] == "tensor" else round(gb / pk["hbm"], 4)
        stages[name] = st
    # router + permute as one HBM stage
    rp_names = ("split_router", "router_gemm", "route_select", "route_finalize", "bucket_hist", "bucket_scan",
                "bucket_scatter", "router_route_bucket", "bucket_tiles")
    rp_ms = sum(stages[n]["ms"] * stages[n]["launches_per_step"] for n in rp_names if n in stages)
    # the stage's algorithmic bytes per token (x read by the router, idx and w
    # written, the scores between the two kernels written and read, idx read
    # again by the bucketing, the two slot maps, x read by the gather and its
    # k copies written) plus the router weight once
    rp_bytes = (T * H * 2 + T * k * 8 + 2 * T * E * 4 + T * k * 4 + T * k * 4 * 2 + T * H * 2 + k * T * H * 2
                + E * H * 4)
    if extra["backward"]:
        # the backward's bucketing: x and d_out read, both permuted ((k+1)T rows each) written
        rp_bytes = 2 * T * H * 2 + T * k * 8 + 2 * (k + 1) * T * H * 2
    if rp_ms > 0:
        # timed as one interval when the stage pass ran (events only at its
        # ends, so its kernels overlap each other's launch and tail as in a
        # plain step); ms_kernel_sum adds the kernels' own event-bracketed times
        rp_one = extra.get("rp_stage_ms") or rp_ms
        stages["router_plus_permute"] = {"ms": round(rp_one, 4), "bound": "hbm",
                                         "gbs": round(rp_bytes / (rp_one * 1e-3) / 1e9, 1),
                                         "frac": round(rp_bytes / (rp_one * 1e-3) / 1e9 / pk["hbm"], 4),
                                         "ms_kernel_sum": round(rp_ms, 4),
                                         "timed": "one interval" if extra.get("rp_stage_ms") else "kernel sum"}
    # the same stage without the router GEMM, which is tensor-bound (fp32-accurate
    # logits take three bf16 products each): selection + bucketing + row scatter
    sp_names = ("route_select", "route_finalize", "bucket_hist", "bucket_scan", "bucket_scatter")
    sp_ms = sum(stages[n]["ms"] * stages[n]["launches_per_step"] for n in sp_names if n in stages)
    sp_bytes = T * E * 4 + T * k * 8 + T * k * 4 * 2 + T * H * 2 + k * T * H * 2
    if sp_ms > 0 and not extra["backward"] and not extra["dense"]:
        stages["select_plus_permute"] = {"ms": round(sp_ms, 4), "bound": "hbm",
                                         "gbs": round(sp_bytes / (sp_ms * 1e-3) / 1e9, 1),
                                         "frac": round(sp_bytes / (sp_ms * 1e-3) / 1e9 / pk["hbm"], 4)}
    # the roofline kernel: the tensor-core stage with the most time per step,
    # against the roofline that binds it at this size
    tensor_stages = [n for n in work if "flops" in work[n] and prof.get(n, (0, 0))[1] > 0]
    dom = max(tensor_stages, key=lambda n: prof[n][0])
    g1 = work[dom]
    g1_ms = prof[dom][0] / max(1, prof[dom][1])
    if g1["bound"] == "tensor":
        g1_ach, g1_peak, g1_unit = g1["flops"] / (g1_ms * 1e-3) / 1e12, pk["bf16_sustained"], "TFLOP/s"
        g1_kind = "%s bf16 dense, sustained" % pk["source"]
    else:
        g1_ach, g1_peak, g1_unit = g1["bytes"] / (g1_ms * 1e-3) / 1e9, pk["hbm"], "GB/s"
        g1_kind = "%s HBM copy bandwidth" % pk["source"]
    gemm_names = [n for n in tensor_stages if n != "router_gemm"]
    if not gemm_names:
        gemm_names = tensor_stages
    gemms_ms = sum(stages[n]["ms"] * stages[n]["launches_per_step"] for n in gemm_names)
    gemm_flops = sum(work[n]["flops"] * stages[n]["launches_per_step"] for n in gemm_names)
    gemm_bytes = sum(work[n]["bytes"] * stages[n]["launches_per_step"] for n in gemm_names)
    g_tf = gemm_flops / (gemms_ms * 1e-3) / 1e12
    g_gb = gemm_bytes / (gemms_ms * 1e-3) / 1e9
    g_bound = "hbm" if gemm_bytes / pk["hbm"] / 1e9 > gemm_flops / pk["bf16_sustained"] / 1e12 else "tensor"
    stages["expert_gemms"] = {"ms": round(gemms_ms, 4), "bound": g_bound, "tflops": round(g_tf, 1),
                              "gbs": round(g_gb, 1),
                              "frac": round(g_tf / pk["bf16_sustained"] if g_bound == "tensor" else g_gb / pk["hbm"],
                                            4)}

    value = world * T / (ms_max * 1e-3)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": workload_name(w0, extra["dense"], extra["backward"]),
                   "T_per_gpu": T, "hidden": H, "experts": E, "groups": w0.n_group, "topk_group": w0.topk_group,
                   "k": k, "inter": I, "shared_inter": w0.Is, "layers": w0.layers,
                   "parallelism": "replicas (dp%d)" % world,
                   "l2": ("L2 scrubbed (256 MB write) between timed steps, per-step CUDA events"
                          if extra["flush"] else
                          "expert weights (%.2f GB per layer) larger than L2, no flush" % (3 * E * I * H * 2 / 1e9)),
                   "untimed_lead_in_steps": extra["lead"],
                   "path": ("moe_layer with the fused router (routing and bucketing in the router kernel)"
                            if getattr(args, "fused_router", False) else
                            "moe_route + moe_forward" if getattr(args, "two_call", False) else
                            "moe_layer (routing and expert stage in one call)"),
                   "hot_expert_share": None if extra["hot_share"] is None else round(extra["hot_share"], 4)},
        "roofline": {"kernel": dom, "bound": g1["bound"], "achieved": round(g1_ach, 1),
                     "peak": g1_peak, "unit": g1_unit,
                     "frac": round(g1_ach / g1_peak, 4),
                     "traffic": gemm_traffic(dom) if T == 32768 and not (extra["dense"] or extra["backward"])
                     else None,
                     "traffic_unit": "bytes per launch (ncu dram read + write, profiles/gemm_dram_traffic_T32768.md)",
                     "peak_kind": g1_kind,
                     "algorithmic_flops_per_launch": g1["flops"],
                     "algorithmic_bytes_per_launch": g1["bytes"]},
        "stages": stages,
        "e2e": None if e2e_ms is None else
        {"value": round(world * T / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
         "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2,
         "how": "median of 3 passes of K steps, after ~0.5 s of untimed passes"},
        "graph": None if extra["graph_ms"] is None else
        {"ms_per_step": round(extra["graph_ms"], 4), "value": round(world * T / (extra["graph_ms"] * 1e-3), 1),
         "unit": "tokens/s", "what": "the same step captured once in a CUDA graph and replayed (inputs resident)"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_cpu_baseline and not extra["dense"] and not extra["backward"]:
        sample = CpuSample(args.workload)
        tps, thr, secs = sample.run(args.cpu_tokens)
        line["cpu_baseline"] = {"value": round(tps, 2), "unit": "tokens/s", "cores": thr, "kind": "oracle",
                                "sample": "first %d tokens of the workload: router logits, routing and expert "
                                          "stage (%.1f s)%s" % (
                                              args.cpu_tokens, secs,
                                              "" if w0.layers == 1 else
                                              ", layer 0 only, rate divided by %d layers" % w0.layers)}
        if args.cpu_tokens_1t:
            import oracle
            oracle.set_threads(1)
            tps1, _, secs1 = sample.run(args.cpu_tokens_1t)
            oracle.set_threads(thr)
            line["cpu_baseline"]["value_1thread"] = round(tps1, 2)
            line["cpu_baseline"]["sample_1thread"] = "first %d tokens, one thread (%.1f s)" % (
                args.cpu_tokens_1t, secs1)
    return line


def run_reference(args, world, rank):
    """The CPU oracle as it stands, on the host cores, one bounded sample per step."""
    if rank != 0:
        return None
    from group_limited_routing_gb300 import workloads as wl

    w0 = wl.WORKLOADS[args.workload]
    sample = CpuSample(args.workload)
    for _ in range(args.warmup):
        sample.run(args.ref_tokens)
    secs = 0.0
    thr = 0
    for _ in range(args.steps):
        _, thr, dt = sample.run(args.ref_tokens)
        secs += dt
    value = args.ref_tokens * args.steps / secs / sample.layers
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / args.steps, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": workload_name(w0), "sample_tokens_per_step": args.ref_tokens},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": thr, "kind": "oracle",
                         "sample": "first %d tokens per step: router logits, routing and expert stage%s"
                                   % (args.ref_tokens, "" if w0.layers == 1 else
                                      " (layer 0 only, rate divided by %d layers)" % w0.layers)},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-tokens", type=int, default=8192, help="oracle sample for cpu_baseline")
    ap.add_argument("--ref-tokens", type=int, default=128, help="oracle sample per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--backward", action="store_true",
                    help="time the layer's backward (moe_backward, routing fixed) instead of its forward")
    ap.add_argument("--dense", type=int, default=0, metavar="I",
                    help="time the dense first-layer MLP of intermediate size I instead of the MoE layer")
    ap.add_argument("--flush-l2", action="store_true",
                    help="scrub L2 between timed steps (always on for workload 1, whose weights fit in L2)")
    ap.add_argument("--cpu-tokens-1t", type=int, default=256,
                    help="oracle sample for the single-thread CPU figure (0 = skip)")
    ap.add_argument("--workload", type=int, default=WORKLOAD_ID, choices=(1, 2, 3, 4, 5, 6),
                    help="1 tiny, 2 decode T=16, 3 T=4096, 4 T=32768 skewed (the bench line), 5 19-layer stack, "
                         "6 T=32768 with ~half of all assignments on 16 hot experts")
    ap.add_argument("--lead-in-ms", type=float, default=500.0,
                    help="untimed loaded steps before the timed region (0: one step; for profiling captures)")
    ap.add_argument("--fused-router", action="store_true",
                    help="one moe_layer call per step with routing and bucketing fused into the router kernel")
    ap.add_argument("--two-call", action="store_true",
                    help="time the two calls moe_route + moe_forward per step instead of the one moe_layer call")
    ap.add_argument("--tokens", type=int, default=0,
                    help="tokens per step (default: the workload's 32768); smaller sizes for profiling captures")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        line = run_reference(args, world, rank)
    else:
        world, rank, local = init_dist()
        line = run_ours(args, world, rank, local)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
