#!/usr/bin/env python
"""Benchmark: routed MoE FFN decode on one GB300 (or N replicas).

Workload: the Q2_0 layer geometry (H=2560, 512 experts, top-10, F=640, blocks of
64 weights, 1,382,400 bytes per expert) as 48 distinct layers (24,576 experts,
33.97 GB resident in HBM), chained with RMSNorm and a residual add. A step is
one decode token (T=1, or a T-token verify window) through all 48 layers:
router GEMV, softmax top-k, bucketing, slot lookup, fused gate/up + SwiGLU,
down projection and combine, per layer. Each step streams ~0.66 GB of expert
weights plus 0.13 GB of router weights, far above the 129 MB L2, so nothing
is served from cache across steps.

metric: MoE-layer tokens/s (layers x tokens per second), with the expert-weight
HBM GB/s and its fraction of the measured copy bandwidth in "roofline".

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (one layer-token per step).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import configs as C  # noqa: E402

METRIC = "MoE-layer tokens/s (decode, Q2_0 layer H=2560 E=512 top-10 F=640)"
UNIT = "layer-tokens/s"
EPS = 1e-6


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--T", type=int, default=1, help="tokens per step (1 = decode, 4 = verify window)")
    ap.add_argument("--layers", type=int, default=48)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill (T=4096 Gemma-shaped layer) line")
    ap.add_argument("--no-residency", action="store_true", help="skip the residency-policy replay and load line")
    ap.add_argument("--no-verify", action="store_true",
                    help="skip the 48-layer chain at T=4 and the single Q2_0 layer at T=1 and T=4")
    ap.add_argument("--no-gemma-decode", action="store_true",
                    help="skip the Gemma-shaped layer's decode and verify windows (T = 1, 2, 8)")
    return ap.parse_args()


# DRAM traffic of k_decode per layer from one ncu capture of a 4-layer chain at T=1
# (dram__bytes_read.sum + dram__bytes_write.sum = 65,946,112 + 1,005,312 B);
# traffic grows in proportion to the layers. It holds only for the kernel sources it
# was taken on: any change to them makes the figure stale, and it is reported as null.
TRAFFIC_REF = {"T": 1, "bytes_per_layer": (66_007_296 + 1_505_792) / 4,
               "sources_sha256": "66ced7d4b55a6ddbc6a1ccdee5dfa84737029ea8e7e6c2068719c242ea5349ea"}
KERNEL_SOURCES = ["quantized_expert_ffn_gb300/csrc/decode_persistent.cu",
                  "quantized_expert_ffn_gb300/csrc/decode_persistent.cuh",
                  "quantized_expert_ffn_gb300/csrc/decode_common.cuh",
                  "quantized_expert_ffn_gb300/csrc/moe_internal.cuh"]


def measured_traffic(T: int, layers: int):
    """DRAM bytes per launch of the step kernel, or None if no capture matches."""
    import hashlib
    h = hashlib.sha256()
    root = os.path.dirname(os.path.abspath(__file__))
    for f in KERNEL_SOURCES:
        with open(os.path.join(root, f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != TRAFFIC_REF["sources_sha256"] or T != TRAFFIC_REF["T"]:
        return None
    return TRAFFIC_REF["bytes_per_layer"] * layers


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


def workload_config(args, n_gpus):
    return {"workload": f"q2_0 MoE decode: {args.layers} distinct layers of H=2560 E=512 top-10 F=640 "
                        f"chained (RMSNorm + residual), T={args.T} tokens per step",
            "T": args.T, "layers": args.layers, "H": 2560, "E": 512, "K": 10, "F": 640,
            "format": "Q2_0 (64 weights + fp16 scale per 18 bytes)",
            "global_batch": args.T * n_gpus, "parallelism": f"replicas x{n_gpus}",
            "l2": "inputs larger than L2: each step streams ~0.79 GB of distinct weights (L2 129 MB)"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.device), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.4)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [s.strip() for s in line.split(",")]))

    def mark(self):
        return time.time()

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [r for (t, r) in self.rows if t0 - 0.15 <= t <= t1 + 0.15] or [r for _, r in self.rows]
        sm = [float(r[0]) for r in rows if r and r[0].replace(".", "").isdigit()]
        smax = [float(r[1]) for r in rows if len(r) > 1 and r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, n in enumerate(names):
                if len(r) > 4 + i and r[4 + i].lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ our path

class Stack:
    """48 (or n) resident Q2_0 layers loaded through the slot table."""

    def __init__(self, L, torch, ctx, n_layers):
        import synth.device as sdev
        cfg = C.CONFIGS["q2_stack"]
        self.cfg, self.L, self.torch = cfg, L, torch
        self.eb = cfg.expert_bytes()
        self.arena = L.moe_arena_create(ctx, self.eb * cfg.E * n_layers + (1 << 20))
        self.slots = L.moe_slots_create(ctx, self.arena, n_layers, cfg.E, cfg.kind, cfg.zero_point,
                                        cfg.H, cfg.F, cfg.E * n_layers)
        staging = torch.empty(cfg.E * self.eb, dtype=torch.uint8, device="cuda")
        nb = 3 * cfg.matrix_blocks()
        self.Wr, self.bias, self.descs = [], [], []
        for l in range(n_layers):
            sdev.expert_blobs_into(staging, cfg.seed, cfg.tag_expert(l, 0), cfg.E, nb, cfg.d_lo, cfg.d_hi)
            base = staging.data_ptr()
            for e in range(cfg.E):
                L.moe_slot_load(self.slots, l, e, base + e * self.eb, self.eb)
            w = C.router_weights(cfg, l)
            self.Wr.append(torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).cuda())
            self.bias.append(torch.from_numpy(C.router_bias(cfg, l)).cuda())
            self.descs.append(L.layer_desc(self.slots, l, cfg.H, cfg.E, cfg.K, cfg.F, self.Wr[l], self.bias[l]))
        torch.cuda.synchronize()
        del staging


def run_residency(L, torch, ctx):
    """Replay of the residency policies on a sticky Zipf routing trace of the
    48-layer stack's shape (hit rates with 5, 10 and 20% of the (layer, expert)
    pairs resident, Belady's ceiling beside them; us_per_event is the host time of a
    token's 48 events routed in one moe_policy_route_token call, per event), and the
    rate at which moe_policy_apply makes experts resident from pinned host memory."""
    import time
    import synth.device as sdev
    from synth import traces
    E, Ln, K, T_prof, T_rep = 512, 48, 10, 32, 256
    tr = traces.routing_trace(T_prof + T_rep, Ln, E, K, seed=11)
    prof = traces.profile_ranking(tr[:T_prof])
    rep = np.ascontiguousarray(tr[T_prof:])
    n_ids = T_rep * Ln * K
    rows = []
    for frac in (0.05, 0.1, 0.2):
        cap = int(frac * Ln * E)
        row = {"capacity": cap, "resident_frac": round(frac, 3)}
        for name, kind in (("lru", L.POLICY_LRU), ("decayed_freq_hl32_guard2", L.POLICY_DECAYED_FREQ),
                           ("lfu_swap_0.7_1.5_2_every4_96", L.POLICY_LFU_SWAP)):
            pol = L.Policy(L.policy_params(kind, cap), Ln, E)
            pol.seed(*prof)
            hits = 0
            t0 = time.perf_counter()
            for t in range(T_rep):
                hits += int(pol.route_token(rep[t])[0].sum())
                pol.end_token()
            dt = time.perf_counter() - t0
            pol.close()
            row[name] = {"hit_rate": hits / n_ids, "misses_per_token": (n_ids - hits) / T_rep,
                         "us_per_event": dt / (T_rep * Ln) * 1e6}
        bel = L.moe_policy_belady(rep, E, cap, *prof)
        row["belady"] = {"hit_rate": bel / n_ids, "misses_per_token": (n_ids - bel) / T_rep}
        rows.append(row)
    # loads through moe_policy_apply: Q2_0 experts of the stack's shape from pinned host memory
    cfg = C.CONFIGS["q2_layer"]
    n = 32
    eb = cfg.expert_bytes()
    arena = L.moe_arena_create(ctx, n * ((eb + 255) // 256 * 256) + 4096)
    slots = L.moe_slots_create(ctx, arena, 1, cfg.E, cfg.kind, cfg.zero_point, cfg.H, cfg.F, n)
    staging = torch.empty(n * eb, dtype=torch.uint8, device="cuda")
    sdev.expert_blobs_into(staging, cfg.seed, cfg.tag_expert(0, 0), n, 3 * cfg.matrix_blocks(), cfg.d_lo, cfg.d_hi)
    host = staging.cpu().pin_memory()
    ptrs = np.zeros(cfg.E, dtype=np.uint64)
    ptrs[:n] = host.data_ptr() + np.arange(n, dtype=np.uint64) * np.uint64(eb)
    zero = np.zeros(n, np.int32)
    ex = np.arange(n, dtype=np.int32)
    none = np.full(n, -1, np.int32)
    stream = torch.cuda.current_stream()
    L.moe_policy_apply(slots, cfg.E, ptrs, eb, zero, ex, none, none, stream=stream)
    ms = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        L.moe_policy_apply(slots, cfg.E, ptrs, eb, zero, ex, zero, ex, stream=stream)  # evict + reload each
        e1.record(stream)
        stream.synchronize()
        ms.append(e0.elapsed_time(e1))
    L.moe_slots_destroy(slots)
    L.moe_arena_destroy(arena)
    del staging, host
    ms_med = float(np.median(ms))
    return {"trace": f"sticky Zipf(1.1) routing, {Ln} layers x {E} experts, top-{K}, {T_rep} tokens replayed "
                     f"after a {T_prof}-token profile seeds the pool; adjacent tokens share "
                     f"{traces.sharing(rep):.0%} of a layer's experts",
            "us_per_event": "host time per routing event, a token's 48 events routed in one "
                            "moe_policy_route_token call (swap rounds included)",
            "replay": rows,
            "load": {"what": f"{n} Q2_0 experts ({eb:,} B each) evicted and reloaded through moe_policy_apply "
                             "from pinned host memory (copy, repack, publish)",
                     "ms": ms_med, "gb_s": n * eb / (ms_med / 1e3) / 1e9}}


def run_prefill(L, torch, ctx, steps: int = 20, warmup: int = 3):
    """The prefill workload: one Gemma-shaped Q4 layer (H=2816, 128 experts, top-8,
    F=704, shared expert F=2112) on a 4096-token window, captured in a graph and
    replayed; bf16 N(0,1) activations, Zipf(1.2) router bias."""
    import synth.device as sdev
    cfg = C.CONFIGS["prefill"]
    T = 4096
    eb = cfg.expert_bytes()
    sh_bytes = cfg.expert_bytes(cfg.F_shared)
    arena = L.moe_arena_create(ctx, eb * cfg.E + sh_bytes + (1 << 20))
    slots = L.moe_slots_create(ctx, arena, 1, cfg.E, cfg.kind, cfg.zero_point, cfg.H, cfg.F, cfg.E)
    shared = L.moe_slots_create(ctx, arena, 1, 1, cfg.kind, cfg.zero_point, cfg.H, cfg.F_shared, 1)
    staging = torch.empty(cfg.E * eb, dtype=torch.uint8, device="cuda")
    sdev.expert_blobs_into(staging, cfg.seed, cfg.tag_expert(0, 0), cfg.E, 3 * cfg.matrix_blocks(), cfg.d_lo, cfg.d_hi)
    for e in range(cfg.E):
        L.moe_slot_load(slots, 0, e, staging.data_ptr() + e * eb, eb)
    L.moe_slot_load(shared, 0, 0, torch.from_numpy(C.shared_expert(cfg, 0)).cuda())
    Wr = torch.from_numpy(C.router_weights(cfg, 0).view(np.int16)).view(torch.bfloat16).cuda()
    bias = torch.from_numpy(C.router_bias(cfg, 0)).cuda()
    desc = L.layer_desc(slots, 0, cfg.H, cfg.E, cfg.K, cfg.F, Wr, bias, shared, cfg.F_shared)
    x = torch.from_numpy(C.activations(cfg, T, step=4096).view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.empty(T, cfg.H, device="cuda")
    ws = torch.empty(L.moe_layer_workspace(desc, T), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    del staging
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        L.moe_layer_forward(ctx, desc, x, y, ws, stream=stream)
    stream.synchronize()
    status = L.moe_status(ctx, stream)
    path = L.moe_ctx_get_option(ctx, L.OPT_LAST_PATH)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        L.moe_layer_forward(ctx, desc, x, y, ws, stream=stream)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    flops = T * (cfg.K * 2 * 3 * cfg.H * cfg.F + 2 * 3 * cfg.H * cfg.F_shared + 2 * cfg.H * cfg.E)
    del graph
    L.moe_slots_destroy(shared)
    L.moe_slots_destroy(slots)
    L.moe_arena_destroy(arena)
    return dict(ms=ms, flops=flops, status=status, path=path, T=T)


def max_over_ranks(values, device):
    """Element-wise maximum of `values` over every rank of the job (the slowest rank
    sets the time); the values themselves with one process."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist = torch.distributed
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_value(n_gpus: int, units_per_rank: float, max_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return n_gpus * units_per_rank / (max_ms / 1e3)


def run_gemma_decode(L, torch, ctx, Ts=(1, 2, 8), n_layers: int = 16, steps: int = 30, warmup: int = 3):
    """Decode and verify windows of the Gemma-shaped Q4 layer (H=2816, 128 experts,
    top-8, F=704, shared expert F=2112; Zipf(1.2) router bias): 16 distinct layers
    (~7 GB of weights, so every window's expert bytes come from HBM), each layer
    called through moe_layer_forward on the same T-token input, the 16 calls
    captured in a graph and replayed. Bytes per layer = distinct routed experts x
    3,345,408 + the shared expert 10,036,224 + the router 720,896."""
    import synth.device as sdev
    cfg = C.CONFIGS["gemma_layer"]
    eb, sh_bytes = cfg.expert_bytes(), cfg.expert_bytes(cfg.F_shared)
    arena = L.moe_arena_create(ctx, n_layers * (cfg.E * ((eb + 255) // 256 * 256) + sh_bytes + 4096) + (1 << 20))
    slots = L.moe_slots_create(ctx, arena, n_layers, cfg.E, cfg.kind, cfg.zero_point, cfg.H, cfg.F,
                               n_layers * cfg.E)
    shared = [L.moe_slots_create(ctx, arena, 1, 1, cfg.kind, cfg.zero_point, cfg.H, cfg.F_shared, 1)
              for _ in range(n_layers)]
    staging = torch.empty(cfg.E * eb, dtype=torch.uint8, device="cuda")
    sh_blob = torch.from_numpy(C.shared_expert(cfg, 0)).cuda()  # one blob, a copy per layer
    descs, keep = [], []
    for l in range(n_layers):
        sdev.expert_blobs_into(staging, cfg.seed, cfg.tag_expert(l, 0), cfg.E, 3 * cfg.matrix_blocks(), cfg.d_lo,
                               cfg.d_hi)
        for e in range(cfg.E):
            L.moe_slot_load(slots, l, e, staging.data_ptr() + e * eb, eb)
        L.moe_slot_load(shared[l], 0, 0, sh_blob)
        Wr = torch.from_numpy(C.router_weights(cfg, l).view(np.int16)).view(torch.bfloat16).cuda()
        bias = torch.from_numpy(C.router_bias(cfg, l)).cuda()
        keep += [Wr, bias]
        descs.append(L.layer_desc(slots, l, cfg.H, cfg.E, cfg.K, cfg.F, Wr, bias, shared[l], cfg.F_shared))
    torch.cuda.synchronize()
    del staging
    stream = torch.cuda.Stream()
    ws = torch.empty(L.moe_layer_workspace(descs[0], max(Ts)), dtype=torch.uint8, device="cuda")
    rows = []
    for T in Ts:
        x = torch.from_numpy(C.activations(cfg, T, step=7000 + T).view(np.int16)).view(torch.bfloat16).cuda()
        y = torch.empty(T, cfg.H, device="cuda")
        ids = torch.empty(n_layers, T, cfg.K, dtype=torch.int32, device="cuda")
        with torch.cuda.stream(stream):
            for l in range(n_layers):
                L.moe_layer_forward(ctx, descs[l], x, y, ws, ids=ids[l], stream=stream)
        stream.synchronize()
        status = L.moe_status(ctx, stream)
        path = L.moe_ctx_get_option(ctx, L.OPT_LAST_PATH)
        ids_h = ids.cpu().numpy()
        distinct = [len(np.unique(ids_h[l])) for l in range(n_layers)]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for l in range(n_layers):
                L.moe_layer_forward(ctx, descs[l], x, y, ws, stream=stream)
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(steps):
                graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms_layer = e0.elapsed_time(e1) / (steps * n_layers)
        layer_bytes = float(np.mean(distinct)) * eb + sh_bytes + cfg.E * cfg.H * 2
        rows.append(dict(T=T, ms_per_layer=ms_layer, layer_tokens_per_s=T / (ms_layer / 1e3),
                         distinct_experts=float(np.mean(distinct)), bytes_per_layer=layer_bytes,
                         gbs=layer_bytes / (ms_layer / 1e3) / 1e9, status=status,
                         path={1: "persistent", 2: "tcgen05 grouped GEMMs", 0: "mma.sync"}.get(path, str(path))))
        del graph
    for sh in shared:
        L.moe_slots_destroy(sh)
    L.moe_slots_destroy(slots)
    L.moe_arena_destroy(arena)
    return rows


def distinct_per_layer(lg, K):
    """Distinct experts chosen per layer from traced logits [layers][T][E] (larger
    logit first, ties to the lower index)."""
    out = []
    for ll in lg:
        chosen = set()
        for row in ll:
            order = np.lexsort((np.arange(row.size), -row))
            chosen.update(int(e) for e in order[:K])
        out.append(len(chosen))
    return out


def run_stack_window(L, torch, ctx, st, T: int, steps: int = 100, warmup: int = 5):
    """The 48-layer chain at a T-token verify window: graph replays of one
    moe_stack_forward per step; distinct experts per layer from a traced pass."""
    cfg = st.cfg
    n = len(st.descs)
    ws = torch.empty(L.moe_layer_workspace(st.descs[0], T) + T * cfg.H * 4 + 4096, dtype=torch.uint8, device="cuda")
    resid = torch.from_numpy(C.as_f64(C.activations(cfg, T, step=40 + T)).astype(np.float32)).cuda()
    stream = torch.cuda.Stream()
    tlg = torch.empty(n, T, cfg.E, dtype=torch.float32, device="cuda")
    tin = torch.empty(n, T, cfg.H, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(stream):
        L.moe_stack_forward(ctx, st.descs, resid.clone(), EPS, ws, tin, tlg)
    stream.synchronize()
    status = L.moe_status(ctx, stream)
    path = L.moe_ctx_get_option(ctx, L.OPT_LAST_PATH)
    distinct = distinct_per_layer(tlg.cpu().numpy(), cfg.K)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        L.moe_stack_forward(ctx, st.descs, resid, EPS, ws)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    del graph
    return dict(T=T, ms_per_step=ms, distinct=distinct, status=status, path=path)


def run_q2_single_layer(L, torch, ctx, st, Ts=(1, 4), steps: int = 30, warmup: int = 3):
    """The single Q2_0 layer (H=2560, 512 experts, top-10, F=640) in decode and verify
    windows: one moe_layer_forward per layer on each of the stack's 48 distinct layers
    (34 GB of experts, so every call's bytes come from HBM), the 48 calls captured in
    a graph and replayed, the same T-token input to every layer."""
    cfg = st.cfg
    n = len(st.descs)
    stream = torch.cuda.Stream()
    rows = []
    ws = torch.empty(L.moe_layer_workspace(st.descs[0], max(Ts)), dtype=torch.uint8, device="cuda")
    for T in Ts:
        x = torch.from_numpy(C.activations(cfg, T, step=8000 + T).view(np.int16)).view(torch.bfloat16).cuda()
        y = torch.empty(T, cfg.H, device="cuda")
        lg = torch.empty(n, T, cfg.E, dtype=torch.float32, device="cuda")
        with torch.cuda.stream(stream):
            for l in range(n):
                L.moe_layer_forward(ctx, st.descs[l], x, y, ws, logits=lg[l], stream=stream)
        stream.synchronize()
        status = L.moe_status(ctx, stream)
        path = L.moe_ctx_get_option(ctx, L.OPT_LAST_PATH)
        distinct = distinct_per_layer(lg.cpu().numpy(), cfg.K)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for l in range(n):
                L.moe_layer_forward(ctx, st.descs[l], x, y, ws, stream=stream)
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(steps):
                graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms_layer = e0.elapsed_time(e1) / (steps * n)
        del graph
        rows.append(dict(T=T, ms_per_layer=ms_layer, distinct=float(np.mean(distinct)), status=status, path=path))
    return rows


def run_ours(args, rank, world, local_rank):
    import torch
    from quantized_expert_ffn_gb300 import _lib as L

    torch.cuda.set_device(local_rank)
    ctx = L.moe_ctx_create(local_rank)
    st = Stack(L, torch, ctx, args.layers)
    cfg = st.cfg
    T = args.T
    ws = torch.empty(L.moe_layer_workspace(st.descs[0], T) + T * cfg.H * 4 + 4096, dtype=torch.uint8,
                     device="cuda")
    x0 = C.as_f64(C.activations(cfg, T, step=rank)).astype(np.float32)
    resid = torch.from_numpy(x0.copy()).cuda()
    stream = torch.cuda.Stream()
    # one eager pass (also checks status), then capture the whole step in a graph
    with torch.cuda.stream(stream):
        L.moe_stack_forward(ctx, st.descs, resid, EPS, ws)
    stream.synchronize()
    assert L.moe_status(ctx, stream) == 0
    path = "persistent" if L.moe_ctx_get_option(ctx, L.OPT_LAST_PATH) == 1 else "multi-kernel"
    # distinct experts per layer (the bytes a window really streams), from a traced pass
    tlg = torch.empty(args.layers, T, cfg.E, dtype=torch.float32, device="cuda")
    tin = torch.empty(args.layers, T, cfg.H, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(stream):
        L.moe_stack_forward(ctx, st.descs, resid.clone(), EPS, ws, tin, tlg)
    stream.synchronize()
    distinct = distinct_per_layer(tlg.cpu().numpy(), cfg.K)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        L.moe_stack_forward(ctx, st.descs, resid, EPS, ws)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    if rank == 0:
        sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    ms = ev0.elapsed_time(ev1)
    clocks = sampler.stop(t0, t1) if rank == 0 else None
    status = L.moe_status(ctx, stream)

    # per-layer roofline: eager layer-by-layer pass with events on the launching stream
    layer_ms = []
    with torch.cuda.stream(stream):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.layers + 1)]
        for rep in range(3):
            evs[0].record(stream)
            for l in range(args.layers):
                L.moe_stack_forward(ctx, [st.descs[l]], resid, EPS, ws)
                evs[l + 1].record(stream)
            stream.synchronize()
            layer_ms.append([evs[l].elapsed_time(evs[l + 1]) for l in range(args.layers)])
    layer_ms = float(np.mean(layer_ms))

    # end to end through the host-buffer entry point: H2D + 48 layers + D2H every step
    resid_h = torch.from_numpy(x0.copy()).pin_memory()
    e2e_steps = max(20, args.steps // 4)
    for _ in range(3):
        L.moe_stack_forward_host(ctx, st.descs, resid_h, EPS, ws, stream=stream)
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        L.moe_stack_forward_host(ctx, st.descs, resid_h, EPS, ws, stream=stream)
    e1.record(stream)
    stream.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    verify = None if args.no_verify else run_stack_window(L, torch, ctx, st, 4)
    single = None if args.no_verify else run_q2_single_layer(L, torch, ctx, st)
    pre = None if args.no_prefill else run_prefill(L, torch, ctx)
    gemma = None if args.no_gemma_decode else run_gemma_decode(L, torch, ctx)
    resid_line = None if (args.no_residency or rank != 0) else run_residency(L, torch, ctx)

    ms, e2e_ms_max = max_over_ranks([ms, e2e_ms], "cuda")
    return dict(ms=ms, e2e_ms=e2e_ms_max, layer_ms=layer_ms, clocks=clocks, status=status, cfg=cfg, path=path,
                distinct=distinct, prefill=pre, gemma=gemma, residency=resid_line, verify=verify, single=single)


# ------------------------------------------------------------------ oracle (CPU)

def oracle_sample_rate(seconds: float, T: int = 1, max_steps: int | None = None):
    """Time the fp64 oracle on layer-tokens of the same workload (one layer and
    one T-token window per sample), for about `seconds` of CPU work."""
    import oracle
    cfg = C.CONFIGS["q2_stack"]
    oracle.build()
    done, busy, l = 0, 0.0, 0
    while busy < seconds and (max_steps is None or done < max_steps):
        layer = l % cfg.layers
        Wr = C.as_f64(C.router_weights(cfg, layer))
        b = C.router_bias(cfg, layer).astype(np.float64)
        x = oracle.rmsnorm(C.as_f64(C.activations(cfg, T, step=1000 + l)), EPS)
        t0 = time.perf_counter()
        lg = oracle.router_logits(x, Wr, b)
        ids, _, _ = oracle.topk(lg, cfg.K)
        t1 = time.perf_counter()
        need = np.unique(ids)  # the inputs the oracle reads: generated outside the timing
        blobs = C.experts(cfg, layer, need)
        experts = [None] * cfg.E
        for i, e in enumerate(need):
            experts[int(e)] = blobs[i]
        t2 = time.perf_counter()
        oracle.layer_forward(cfg.kind, cfg.zero_point, cfg.H, cfg.E, cfg.K, cfg.F, None, None, experts, x,
                             logits_in=lg)
        t3 = time.perf_counter()
        busy += (t1 - t0) + (t3 - t2)
        done += 1
        l += 1
    return (done * T / busy if busy > 0 else 0.0), done, busy


def oracle_sample_rate_threads(seconds: float, T: int = 1, threads: int | None = None, rounds: int | None = None,
                               warmup_rounds: int = 0):
    """The same oracle work on every host core: one thread per core, each running
    layer-token samples (router, top-k, layer) for about `seconds` of wall time; the
    inputs are generated before the timed window (the oracle's C calls release the
    Python lock, so the threads run in parallel). With `rounds`, every thread runs
    exactly that many samples instead (after `warmup_rounds` untimed ones). Returns
    (layer-tokens/s, threads, samples done, wall seconds)."""
    import concurrent.futures as cf
    import oracle
    cfg = C.CONFIGS["q2_stack"]
    oracle.build()
    n = threads or os.cpu_count() or 1
    samples = []
    for i in range(n):
        layer = i % cfg.layers
        Wr = C.as_f64(C.router_weights(cfg, layer))
        b = C.router_bias(cfg, layer).astype(np.float64)
        x = oracle.rmsnorm(C.as_f64(C.activations(cfg, T, step=2000 + i)), EPS)
        lg = oracle.router_logits(x, Wr, b)
        ids, _, _ = oracle.topk(lg, cfg.K)
        need = np.unique(ids)
        blobs = C.experts(cfg, layer, need)
        experts = [None] * cfg.E
        for j, e in enumerate(need):
            experts[int(e)] = blobs[j]
        samples.append((Wr, b, x, experts))

    def work(i, deadline, rounds=None):
        Wr, b, x, experts = samples[i]
        done = 0
        while (time.perf_counter() < deadline) if rounds is None else (done < rounds):
            lg = oracle.router_logits(x, Wr, b)
            oracle.topk(lg, cfg.K)
            oracle.layer_forward(cfg.kind, cfg.zero_point, cfg.H, cfg.E, cfg.K, cfg.F, None, None, experts, x,
                                 logits_in=lg)
            done += 1
        return done

    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        if warmup_rounds:
            list(ex.map(lambda i: work(i, 0.0, warmup_rounds), range(n)))
        t0 = time.perf_counter()
        if rounds is not None:
            done = sum(ex.map(lambda i: work(i, 0.0, rounds), range(n)))
        else:
            done = sum(ex.map(lambda i: work(i, t0 + seconds), range(n)))
        wall = time.perf_counter() - t0
    return done * T / wall, n, done, wall


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for key in ("Model name", "BIOS Model name"):
            for line in out.splitlines():
                if line.startswith(key + ":"):
                    name = line.split(":", 1)[1].strip()
                    if name and name != "-":
                        return name
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


# ------------------------------------------------------------------ main

def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    n_gpus = max(world, 1)
    cfgj = workload_config(args, n_gpus)

    if args.impl == "reference":
        if rank != 0:
            return 0
        # a step: every host core runs one layer-step of the workload (W untimed steps
        # first); the oracle's C calls run in parallel threads
        rate, nthr, done, wall = oracle_sample_rate_threads(0.0, args.T, rounds=args.steps,
                                                            warmup_rounds=args.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": n_gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / max(args.steps, 1) * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": cfgj,
                "cpu_baseline": {"kind": "oracle", "value": rate, "unit": UNIT, "cores": nthr, "cpu": cpu_model(),
                                 "sample": f"{done} layer-steps of one {args.T}-token window each on {nthr} threads "
                                           f"(router, top-k, experts, combine; fp64)"},
                "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    r = run_ours(args, rank, world, local_rank)
    cfg = r["cfg"]
    T = args.T
    layer_tokens = args.layers * T
    value = job_value(n_gpus, layer_tokens * args.steps, r["ms"])
    e2e_value = job_value(n_gpus, layer_tokens, r["e2e_ms"])
    pk = peaks()
    hbm_peak = pk["hbm_gbs"] if pk else 6800.0
    expert_bytes = cfg.expert_bytes()
    router_bytes = cfg.E * cfg.H * 2
    # algorithmic bytes of one step (= one launch of the persistent kernel): per layer the
    # distinct experts of the window plus the router matrix
    step_expert_bytes = sum(r["distinct"]) * expert_bytes
    step_bytes = step_expert_bytes + args.layers * router_bytes
    step_s = r["ms"] / args.steps / 1e3
    achieved = step_bytes / step_s / 1e9
    step_expert_gbs = step_expert_bytes / step_s / 1e9
    # kernels of ours per step: the persistent path runs the whole 48-layer chain as
    # one cooperative kernel (plus a memset of its barrier words); the multi-kernel
    # path runs rmsnorm, router, top-k, bucket, plan, gate/up, down, combine per layer
    # the persistent kernel runs up to 48 layers per cooperative launch
    launches_per_step = -(-args.layers // 48) if r["path"] == "persistent" else 8 * args.layers
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": n_gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 mma / fp32 accumulate (Q2_0 weights)",
        "data": "synthetic", "config": cfgj,
        "stack_tokens_per_s": n_gpus * T * args.steps / (r["ms"] / 1e3),
        "expert_weight_gbs": step_expert_gbs,
        "expert_weight_frac_of_hbm": step_expert_gbs / hbm_peak,
        "distinct_experts_per_layer": float(np.mean(r["distinct"])),
        "eager_layer_ms": r["layer_ms"],
        "roofline": {"kernel": ("k_decode: one cooperative launch runs the whole chain of layers"
                                if r["path"] == "persistent"
                                else "the step's 8-kernel layer calls, in the captured step graph"),
                     "bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak,
                     "traffic": (measured_traffic(T, args.layers) if r["path"] == "persistent" else None),
                     "peak_source": "measured" if pk else "fallback",
                     "algorithmic_bytes_per_launch": step_bytes,
                     "algorithmic_bytes": "per layer: distinct experts x 1,382,400 B + router 2,621,440 B"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": T * cfg.H * 4,
                "d2h_bytes_per_step": T * cfg.H * 4},
        "gpu_launches": launches_per_step * args.steps,
        "path": r["path"],
        "clocks": r["clocks"],
        "device_status": r["status"],
    }
    if r["prefill"]:
        pre = r["prefill"]
        tf = pre["flops"] / (pre["ms"] / 1e3) / 1e12
        bf16_peak = pk["bf16_tflops"] if pk and "bf16_tflops" in pk else 1900.0
        line["prefill"] = {
            "workload": "Gemma-shaped Q4 layer H=2816 E=128 top-8 F=704 + shared F=2112, T=4096 "
                        "(router, top-k, bucket, plan, gate/up and down grouped GEMMs, combine)",
            "ms_per_layer": pre["ms"], "tflops": tf, "unit": "TFLOP/s", "flops_per_layer": pre["flops"],
            "peak": bf16_peak, "peak_source": "measured (bf16 burst; fp16 operands run at the same rate)" if pk
            else "fallback", "frac": tf / bf16_peak,
            "path": {2: "tcgen05 grouped GEMMs", 1: "persistent", 0: "mma.sync"}.get(pre["path"], str(pre["path"])),
            "device_status": pre["status"]}
    if r.get("gemma"):
        hbm = pk["hbm_gbs"] if pk and "hbm_gbs" in pk else 6800.0
        line["gemma_decode"] = {
            "workload": "Gemma-shaped Q4 layer H=2816 E=128 top-8 F=704 + shared F=2112, Zipf(1.2) router bias; "
                        "16 distinct layers (~7 GB) replayed, one moe_layer_forward per layer",
            "unit": "layer-tokens/s", "hbm_peak_gbs": hbm,
            "rows": [dict(row, frac_of_hbm=row["gbs"] / hbm) for row in r["gemma"]]}
    if r.get("verify"):
        v = r["verify"]
        vb = sum(v["distinct"]) * expert_bytes + args.layers * router_bytes
        gbs = vb / (v["ms_per_step"] / 1e3) / 1e9
        line["verify_window"] = {
            "workload": f"the same {args.layers}-layer Q2_0 chain at a {v['T']}-token verify window "
                        "(one moe_stack_forward per step, graph replays)",
            "T": v["T"], "ms_per_step": v["ms_per_step"],
            "layer_tokens_per_s": job_value(n_gpus, args.layers * v["T"], v["ms_per_step"]),
            "stack_tokens_per_s": job_value(n_gpus, v["T"], v["ms_per_step"]),
            "distinct_experts_per_layer": float(np.mean(v["distinct"])), "bytes_per_step": vb,
            "gbs": gbs, "frac_of_hbm": gbs / hbm_peak, "hbm_peak_gbs": hbm_peak,
            "path": {1: "persistent", 2: "tcgen05 grouped GEMMs", 0: "mma.sync"}.get(v["path"], str(v["path"])),
            "device_status": v["status"]}
    if r.get("single"):
        rows = []
        for row in r["single"]:
            b = row["distinct"] * expert_bytes + router_bytes
            gbs = b / (row["ms_per_layer"] / 1e3) / 1e9
            rows.append(dict(T=row["T"], ms_per_layer=row["ms_per_layer"],
                             layer_tokens_per_s=row["T"] / (row["ms_per_layer"] / 1e3),
                             distinct_experts=row["distinct"], bytes_per_layer=b, gbs=gbs, frac_of_hbm=gbs / hbm_peak,
                             path={1: "persistent", 2: "tcgen05 grouped GEMMs", 0: "mma.sync"}.get(row["path"],
                                                                                                 str(row["path"])),
                             status=row["status"]))
        line["q2_layer_decode"] = {
            "workload": "single Q2_0 layer H=2560 E=512 top-10 F=640 (Zipf(1.1) router bias), one moe_layer_forward "
                        f"per layer on each of the {args.layers} distinct layers of the chain (34 GB), graph replays",
            "unit": "layer-tokens/s", "hbm_peak_gbs": hbm_peak,
            "bytes": "per layer: distinct experts x 1,382,400 B + router 2,621,440 B", "rows": rows}
    if r.get("residency"):
        line["residency"] = r["residency"]
    if rank == 0 and not args.no_cpu_baseline:
        rate1, done1, busy1 = oracle_sample_rate(8.0, T)
        rate, nthr, done, wall = oracle_sample_rate_threads(8.0, T)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": nthr, "kind": "oracle",
                                "cpu": cpu_model(),
                                "sample": f"{done} layer-steps ({T}-token windows) of the chain's layers on {nthr} "
                                          f"threads, {wall:.1f} s wall (fp64; inputs generated outside the timing)",
                                "single_thread": {"value": rate1, "unit": UNIT, "cores": 1,
                                                  "sample": f"{done1} layer-steps, {busy1:.1f} s of one thread"}}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
