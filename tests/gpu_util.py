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
