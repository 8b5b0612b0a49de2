"""GPU-side fixtures for the parity tests: resident layers built from the seeded
configurations through the C ABI, and the oracle run on the same inputs."""
from __future__ import annotations

import numpy as np

import oracle
import synth
import synth.device as sdev
from quantized_expert_ffn_gb300 import _lib as L
from synth import configs as C

TOL = 2e-3  # max over tokens of ||y - y_oracle||_inf / ||y_oracle||_inf


def torch():
    import torch as t
    return t


def to_dev(a, dtype=None):
    """numpy fp32 array or uint16 bf16 patterns -> CUDA tensor."""
    T = torch()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return T.from_numpy(a.view(np.int16).copy()).view(T.bfloat16).cuda()
    return T.from_numpy(a.copy()).cuda()


def rel_err(y, ref):
    """Per-token ||y - ref||_inf / ||ref||_inf, maximum over tokens."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.abs(y - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    return float((num / np.maximum(den, 1e-30)).max())


class GpuLayers:
    """`n_layers` layers of config `cfg`, all experts resident in one arena."""

    def __init__(self, ctx, cfg: C.Config, n_layers: int = 1, zero_point: int | None = None,
                 load: bool = True):
        T = torch()
        self.ctx, self.cfg, self.n_layers = ctx, cfg, n_layers
        self.zp = cfg.zero_point if zero_point is None else zero_point
        self.eb = cfg.expert_bytes()
        stride = (self.eb + 255) // 256 * 256
        cap = n_layers * cfg.E
        sh_bytes = 0
        if cfg.F_shared:
            sh_bytes = n_layers * ((cfg.expert_bytes(cfg.F_shared) + 255) // 256 * 256)
        self.arena = L.moe_arena_create(ctx, stride * cap + sh_bytes + 4096)
        self.slots = L.moe_slots_create(ctx, self.arena, n_layers, cfg.E, cfg.kind, self.zp, cfg.H,
                                        cfg.F, cap)
        self.shared = None
        if cfg.F_shared:
            self.shared = [L.moe_slots_create(ctx, self.arena, 1, 1, cfg.kind, self.zp, cfg.H,
                                              cfg.F_shared, 1) for _ in range(n_layers)]
        self.Wr, self.bias = [], []
        for l in range(n_layers):
            w = C.router_weights(cfg, l)
            self.Wr.append(to_dev(w))
            b = C.router_bias(cfg, l)
            self.bias.append(None if b is None else to_dev(b))
        if load:
            staging = T.empty(cfg.E * self.eb, dtype=T.uint8, device="cuda")
            nb = 3 * cfg.matrix_blocks()
            for l in range(n_layers):
                sdev.expert_blobs_into(staging, cfg.seed, cfg.tag_expert(l, 0), cfg.E, nb, cfg.d_lo,
                                       cfg.d_hi)
                for e in range(cfg.E):
                    L.moe_slot_load(self.slots, l, e, staging.data_ptr() + e * self.eb, self.eb)
                if self.shared:
                    sh = T.from_numpy(C.shared_expert(cfg, l)).cuda()
                    L.moe_slot_load(self.shared[l], 0, 0, sh)
            T.cuda.synchronize()
            del staging

    # optional layer_desc fields (act, router_scale, down_scale, router_kind, drop policy)
    opts: dict = {}

    def desc(self, l: int = 0):
        cfg = self.cfg
        return L.layer_desc(self.slots, l, cfg.H, cfg.E, cfg.K, cfg.F, self.Wr[l], self.bias[l],
                            self.shared[l] if self.shared else None, cfg.F_shared, **self.opts)

    def workspace(self, T_tokens: int, extra: int = 0):
        T = torch()
        n = L.moe_layer_workspace(self.desc(0), T_tokens) + extra
        return T.empty(n, dtype=T.uint8, device="cuda")

    def forward(self, x, l: int = 0):
        T = torch()
        Tn = x.shape[0]
        y = T.empty(Tn, self.cfg.H, dtype=T.float32, device="cuda")
        logits = T.empty(Tn, self.cfg.E, dtype=T.float32, device="cuda")
        ids = T.empty(Tn, self.cfg.K, dtype=T.int32, device="cuda")
        ws = self.workspace(Tn)
        L.moe_layer_forward(self.ctx, self.desc(l), x, y, ws, logits=logits, ids=ids)
        T.cuda.synchronize()
        return y, logits, ids

    def close(self):
        T = torch()
        T.cuda.synchronize()
        if self.shared:
            for s in self.shared:
                L.moe_slots_destroy(s)
        L.moe_slots_destroy(self.slots)
        L.moe_arena_destroy(self.arena)


def oracle_layer(cfg: C.Config, l: int, x64, logits_gpu, zero_point=None, tokens=None):
    """Oracle output for the given tokens, routed with the GPU's fp32 logits.

    x64: [T][H] fp64 values the GPU saw; logits_gpu: [T][E] fp32. Returns the
    oracle dict for the selected rows (all rows when tokens is None)."""
    zp = cfg.zero_point if zero_point is None else zero_point
    rows = np.arange(x64.shape[0]) if tokens is None else np.asarray(tokens)
    lg = np.asarray(logits_gpu, dtype=np.float64)[rows]
    ids, _, _ = oracle.topk(lg, cfg.K)
    need = np.unique(ids)
    blobs = C.experts(cfg, l, need)
    experts = [None] * cfg.E
    for i, e in enumerate(need):
        experts[int(e)] = blobs[i]
    shared = C.shared_expert(cfg, l)
    return oracle.layer_forward(cfg.kind, zp, cfg.H, cfg.E, cfg.K, cfg.F, None, None, experts,
                                np.ascontiguousarray(x64[rows]), shared=shared,
                                F_shared=cfg.F_shared, logits_in=lg)


def oracle_layer_by_bucket(cfg: C.Config, l: int, x64, logits_gpu, threads: int | None = None):
    """Oracle output for EVERY token of a wide window, routed with the GPU's fp32
    logits: the same definition as oracle.layer_forward (top-k and weights from
    oracle.topk, each selected expert's FFN from oracle.expert_ffn, the combine in
    k order in fp64, then the shared expert), evaluated one expert bucket at a time
    so that each expert's weights are dequantised once. The oracle's C calls run on
    a thread pool (ctypes releases the GIL during them).

    Returns dict(y [T][H] fp64, ids [T][K], counts [E])."""
    import concurrent.futures as cf
    import os
    T = x64.shape[0]
    lg = np.asarray(logits_gpu, dtype=np.float64)
    ids, w, _ = oracle.topk(lg, cfg.K)
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    need = np.flatnonzero(counts)
    blobs = C.experts(cfg, l, need)
    x64 = np.ascontiguousarray(x64, dtype=np.float64)
    ye = {}

    def run(i):
        e = int(need[i])
        rows = np.flatnonzero((ids == e).any(axis=1))
        return e, rows, oracle.expert_ffn(cfg.kind, cfg.zero_point, blobs[i], cfg.H, cfg.F, x64[rows])

    shared = C.shared_expert(cfg, l)
    chunks = [np.arange(s, min(s + 64, T)) for s in range(0, T, 64)] if shared is not None else []

    def run_shared(rows):
        return rows, oracle.expert_ffn(cfg.kind, cfg.zero_point, shared, cfg.H, cfg.F_shared, x64[rows])

    y_sh = np.zeros((T, cfg.H))
    with cf.ThreadPoolExecutor(max_workers=threads or os.cpu_count() or 4) as ex:
        futs = [ex.submit(run, i) for i in range(len(need))]
        sfuts = [ex.submit(run_shared, r) for r in chunks]
        for f in futs:
            e, rows, y = f.result()
            ye[e] = (rows, y)
        for f in sfuts:
            rows, y = f.result()
            y_sh[rows] = y
    # row of token t in its expert's bucket output
    pos = {e: {int(t): j for j, t in enumerate(rows)} for e, (rows, _) in ye.items()}
    y = np.zeros((T, cfg.H))
    for t in range(T):
        acc = np.zeros(cfg.H)
        for k in range(cfg.K):
            e = int(ids[t, k])
            acc += w[t, k] * ye[e][1][pos[e][t]]
        y[t] = acc + y_sh[t]
    return dict(y=y, ids=ids, counts=counts)
