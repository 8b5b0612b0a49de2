"""A serving loop with a residency policy driving the slot pool: per token, route on
the GPU, hand the ids to the policy, apply its loads and evictions to the pool
(each table entry published after its copy lands), then run the layer. With a
demand policy every routed expert is resident when the layer runs, so the output
matches the oracle; the pool's table always equals the policy's residency."""
import numpy as np
import pytest

import oracle
from quantized_expert_ffn_gb300 import _lib as L
from synth import configs as C

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch
    torch.cuda.init()
    return torch


@pytest.fixture(scope="module")
def ctx(torch):
    c = L.moe_ctx_create(0)
    yield c
    L.moe_ctx_destroy(c)


def _pool(torch, ctx, cfg, capacity):
    eb = cfg.expert_bytes()
    arena = L.moe_arena_create(ctx, capacity * ((eb + 255) // 256 * 256) + 4096)
    slots = L.moe_slots_create(ctx, arena, 1, cfg.E, cfg.kind, cfg.zero_point, cfg.H, cfg.F, capacity)
    blobs = C.experts(cfg, 0, range(cfg.E))
    pinned = [torch.from_numpy(b).pin_memory() for b in blobs]
    ptrs = np.array([t.data_ptr() for t in pinned], dtype=np.uint64)
    return arena, slots, blobs, pinned, ptrs, eb


def _table(slots, E):
    return [L.moe_slot_lookup(slots, 0, e) >= 0 for e in range(E)]


@pytest.mark.parametrize("kind", [L.POLICY_LRU, L.POLICY_DECAYED_FREQ])
def test_demand_policy_serves_every_token(torch, ctx, kind):
    cfg = C.CONFIGS["tiny"]
    cap = 5
    arena, slots, blobs, pinned, ptrs, eb = _pool(torch, ctx, cfg, cap)
    pol = L.Policy(L.policy_params(kind, cap), 1, cfg.E)
    try:
        Wr = torch.from_numpy(C.router_weights(cfg, 0)).cuda()
        desc = L.layer_desc(slots, 0, cfg.H, cfg.E, cfg.K, cfg.F, Wr)
        ws = torch.empty(L.moe_layer_workspace(desc, 1), dtype=torch.uint8, device="cuda")
        x_all = C.activations(cfg, 24, step=77)
        loads = 0
        for t in range(24):
            x = torch.from_numpy(x_all[t:t + 1].copy()).cuda()
            lg = torch.empty(1, cfg.E, device="cuda")
            ids = torch.empty(1, cfg.K, dtype=torch.int32, device="cuda")
            w = torch.empty(1, cfg.K, device="cuda")
            L.moe_router_topk(ctx, x, Wr, None, cfg.K, lg, ids, w)
            ids_h = ids.cpu().numpy()[0]
            hit, le, el, ee = pol.route(0, ids_h)
            loads += le.size
            L.moe_policy_apply(slots, cfg.E, ptrs, eb, np.zeros(le.size, np.int32), le, el, ee)
            pol.end_token()
            assert _table(slots, cfg.E) == [pol.resident(0, e) for e in range(cfg.E)]
            y = torch.empty(1, cfg.H, device="cuda")
            lg2 = torch.empty(1, cfg.E, device="cuda")
            ids2 = torch.empty(1, cfg.K, dtype=torch.int32, device="cuda")
            L.moe_layer_forward(ctx, desc, x, y, ws, logits=lg2, ids=ids2)
            assert L.moe_status(ctx) == 0  # every routed expert was resident
            assert torch.equal(ids2, ids)
            r = oracle.layer_forward(cfg.kind, cfg.zero_point, cfg.H, cfg.E, cfg.K, cfg.F, None, None, list(blobs),
                                     x_all[t:t + 1].astype(np.float64),
                                     logits_in=lg2.cpu().numpy().astype(np.float64))
            yy = y.cpu().numpy().astype(np.float64)
            assert np.abs(yy - r["y"]).max() <= 2e-3 * np.abs(r["y"]).max()
        assert loads > cap  # the pool turned over
    finally:
        pol.close()
        torch.cuda.synchronize()
        L.moe_slots_destroy(slots)
        L.moe_arena_destroy(arena)


def test_swap_policy_applies_its_rounds_and_misses_are_flagged(torch, ctx):
    cfg = C.CONFIGS["tiny"]
    cap = 4
    arena, slots, blobs, pinned, ptrs, eb = _pool(torch, ctx, cfg, cap)
    pol = L.Policy(L.policy_params(L.POLICY_LFU_SWAP, cap, swap_every=2, max_swaps=2), 1, cfg.E)
    try:
        # seed experts 12..15; route to 0 and 1 every token: they swap in
        seed = np.arange(12, 16, dtype=np.int32)
        assert pol.seed(np.zeros(4, np.int32), seed) == 4
        L.moe_policy_apply(slots, cfg.E, ptrs, eb, np.zeros(4, np.int32), seed, np.full(4, -1, np.int32),
                           np.full(4, -1, np.int32))
        swapped = 0
        for t in range(6):
            hit, le, el, ee = pol.route(0, np.array([0, 1], dtype=np.int32))
            assert le.size == 0
            sl, se, vl, ve = pol.end_token()
            L.moe_policy_apply(slots, cfg.E, ptrs, eb, sl, se, vl, ve)
            swapped += sl.size
            assert _table(slots, cfg.E) == [pol.resident(0, e) for e in range(cfg.E)]
        assert swapped == 2 and pol.resident(0, 0) and pol.resident(0, 1)
        # an expert the policy does not hold is absent on the GPU: flagged, adds nothing
        Wr = torch.zeros(cfg.E, cfg.H, device="cuda")
        bias = torch.zeros(cfg.E, device="cuda")
        absent = [e for e in range(cfg.E) if not pol.resident(0, e)]
        bias[absent[0]] = 5.0
        bias[0] = 4.0
        desc = L.layer_desc(slots, 0, cfg.H, cfg.E, cfg.K, cfg.F, Wr, bias)
        ws = torch.empty(L.moe_layer_workspace(desc, 1), dtype=torch.uint8, device="cuda")
        x = torch.from_numpy(C.activations(cfg, 1, step=78)).cuda()
        y = torch.empty(1, cfg.H, device="cuda")
        L.moe_layer_forward(ctx, desc, x, y, ws)
        assert L.moe_status(ctx) & L.STATUS_EXPERT_ABSENT
    finally:
        pol.close()
        torch.cuda.synchronize()
        L.moe_slots_destroy(slots)
        L.moe_arena_destroy(arena)


def test_pinned_pageable_and_device_blobs_load_the_same_bytes(torch, ctx):
    # pinned (asynchronous copy) and pageable (synchronous copy) host blobs go through
    # the pool's staging buffer, device blobs are read directly: same layer bits
    cfg = C.CONFIGS["tiny"]
    blobs = C.experts(cfg, 0, range(cfg.E))
    Wr = torch.from_numpy(C.router_weights(cfg, 0)).cuda()
    x = torch.from_numpy(C.activations(cfg, 4, step=79)).cuda()
    eb = cfg.expert_bytes()
    outs = []
    for how in ("pinned", "pageable", "device"):
        arena = L.moe_arena_create(ctx, cfg.E * ((eb + 255) // 256 * 256) + 4096)
        slots = L.moe_slots_create(ctx, arena, 1, cfg.E, cfg.kind, cfg.zero_point, cfg.H, cfg.F, cfg.E)
        keep = []
        for e in range(cfg.E):
            t = torch.from_numpy(blobs[e])
            t = t.pin_memory() if how == "pinned" else (t.cuda() if how == "device" else t)
            keep.append(t)
            L.moe_slot_load(slots, 0, e, t)
        desc = L.layer_desc(slots, 0, cfg.H, cfg.E, cfg.K, cfg.F, Wr)
        ws = torch.empty(L.moe_layer_workspace(desc, 4), dtype=torch.uint8, device="cuda")
        y = torch.empty(4, cfg.H, device="cuda")
        L.moe_layer_forward(ctx, desc, x, y, ws)
        assert L.moe_status(ctx) == 0
        outs.append(y.clone())
        torch.cuda.synchronize()
        L.moe_slots_destroy(slots)
        L.moe_arena_destroy(arena)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
