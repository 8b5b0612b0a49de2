"""The persistent decode kernel (one cooperative launch per layer call or per
chain of layers) against the multi-kernel path: same bits, so every parity
result of one path holds for the other."""
import numpy as np
import pytest

from quantized_expert_ffn_gb300 import _lib as L
from synth import configs as C
from tests.gpu_util import TOL, GpuLayers, oracle_layer, rel_err, to_dev

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


def _both_paths(ctx, g, x):
    L.moe_ctx_set_option(ctx, L.OPT_PERSISTENT_DECODE, 1)
    a = g.forward(x)
    # the comparison means something only if the persistent kernel really ran
    assert L.moe_ctx_get_option(ctx, L.OPT_LAST_PATH) == 1
    L.moe_ctx_set_option(ctx, L.OPT_PERSISTENT_DECODE, 0)
    try:
        b = g.forward(x)
        assert L.moe_ctx_get_option(ctx, L.OPT_LAST_PATH) == 0
    finally:
        L.moe_ctx_set_option(ctx, L.OPT_PERSISTENT_DECODE, 1)
    return a, b


@pytest.mark.parametrize("name,Ts", [("tiny", (1, 3, 4)), ("q2_layer", (1, 2, 4, 8)),
                                     ("gemma_layer", (1, 2, 5, 8))])
def test_persistent_equals_multikernel_bitwise(torch, ctx, name, Ts):
    cfg = C.CONFIGS[name]
    g = GpuLayers(ctx, cfg)
    try:
        for T in Ts:
            x = to_dev(C.activations(cfg, T, step=300 + T))
            (y1, l1, i1), (y2, l2, i2) = _both_paths(ctx, g, x)
            assert L.moe_status(ctx) == 0
            assert torch.equal(l1, l2), (name, T)
            assert torch.equal(i1, i2), (name, T)
            assert torch.equal(y1, y2), (name, T, (y1 - y2).abs().max().item())
        # and the persistent result against the oracle
        T = Ts[-1]
        xn = C.activations(cfg, T, step=300 + T)
        y, lg, ids = g.forward(to_dev(xn))
        r = oracle_layer(cfg, 0, C.as_f64(xn), lg.cpu().numpy())
        assert np.array_equal(ids.cpu().numpy(), r["ids"])
        assert rel_err(y.cpu().numpy(), r["y"]) <= TOL
    finally:
        g.close()


def test_t_invariance_across_the_path_boundary(torch, ctx):
    # T = 9 runs the multi-kernel path, T = 1 the persistent kernel: same bits per token
    cfg = C.CONFIGS["q2_layer"]
    g = GpuLayers(ctx, cfg)
    try:
        x = to_dev(C.activations(cfg, 9, step=333))
        y9, l9, i9 = g.forward(x)
        assert L.moe_ctx_get_option(ctx, L.OPT_LAST_PATH) == 0
        for t in (0, 4, 8):
            y1, l1, i1 = g.forward(x[t:t + 1].contiguous())
            assert L.moe_ctx_get_option(ctx, L.OPT_LAST_PATH) == 1
            assert torch.equal(y1[0], y9[t]) and torch.equal(l1[0], l9[t]) and torch.equal(i1[0], i9[t])
    finally:
        g.close()


@pytest.mark.parametrize("T", [1, 4])
def test_persistent_stack_equals_layer_by_layer(torch, ctx, T):
    cfg = C.CONFIGS["q2_stack"]
    n = 3
    g = GpuLayers(ctx, cfg, n_layers=n)
    try:
        descs = [g.desc(l) for l in range(n)]
        ws = g.workspace(T)
        r0 = torch.from_numpy(C.as_f64(C.activations(cfg, T, step=400 + T)).astype(np.float32)).cuda()
        # persistent: the whole chain in one launch
        ra = r0.clone()
        tin = torch.empty(n, T, cfg.H, dtype=torch.bfloat16, device="cuda")
        tlg = torch.empty(n, T, cfg.E, device="cuda")
        L.moe_stack_forward(g.ctx, descs, ra, 1e-6, ws, tin, tlg)
        assert L.moe_ctx_get_option(ctx, L.OPT_LAST_PATH) == 1
        assert L.moe_status(ctx) == 0
        # multi-kernel path
        L.moe_ctx_set_option(ctx, L.OPT_PERSISTENT_DECODE, 0)
        try:
            rb = r0.clone()
            tin2 = torch.empty_like(tin)
            tlg2 = torch.empty_like(tlg)
            L.moe_stack_forward(g.ctx, descs, rb, 1e-6, ws, tin2, tlg2)
        finally:
            L.moe_ctx_set_option(ctx, L.OPT_PERSISTENT_DECODE, 1)
        torch.cuda.synchronize()
        assert torch.equal(tin, tin2)
        assert torch.equal(tlg, tlg2)
        assert torch.equal(ra, rb)
    finally:
        g.close()


def test_persistent_absent_expert(torch, ctx):
    cfg = C.CONFIGS["q2_layer"]
    g = GpuLayers(ctx, cfg)
    try:
        x = to_dev(C.activations(cfg, 2, step=500))
        y, lg, ids = g.forward(x)
        e = int(ids.cpu()[1, 3])
        L.moe_slot_evict(g.slots, 0, e)
        (y1, _, _), (y2, _, _) = _both_paths(ctx, g, x)
        assert L.moe_status(ctx) & L.STATUS_EXPERT_ABSENT
        assert torch.equal(y1, y2)
        assert not torch.equal(y1, y)
    finally:
        g.close()


def test_option_query(torch, ctx):
    assert L.moe_ctx_get_option(ctx, L.OPT_PERSISTENT_DECODE) == 1
    L.moe_ctx_set_option(ctx, L.OPT_PERSISTENT_DECODE, 0)
    try:
        assert L.moe_ctx_get_option(ctx, L.OPT_PERSISTENT_DECODE) == 0
    finally:
        L.moe_ctx_set_option(ctx, L.OPT_PERSISTENT_DECODE, 1)
    with pytest.raises(L.MoeError):
        L.moe_ctx_set_option(ctx, L.OPT_LAST_PATH, 1)
    with pytest.raises(L.MoeError):
        L.moe_ctx_get_option(ctx, 99)


def test_bounded_wait_gives_up_and_the_context_recovers(torch, ctx):
    # a grid-barrier arrival that never comes (test hook): every wait runs into its
    # time limit, the kernel returns with MOE_STATUS_TIMEOUT, and the next call on
    # the same context runs normally
    import time
    cfg = C.CONFIGS["q2_stack"]
    n = 3
    g = GpuLayers(ctx, cfg, n_layers=n)
    try:
        descs = [g.desc(l) for l in range(n)]
        ws = g.workspace(1)
        r0 = torch.from_numpy(C.as_f64(C.activations(cfg, 1, step=450)).astype(np.float32)).cuda()
        good = r0.clone()
        L.moe_stack_forward(g.ctx, descs, good, 1e-6, ws)
        assert L.moe_status(ctx) == 0
        for layer in (0, 2):
            L.moe_ctx_set_option(ctx, L.OPT_TEST_SKIP_ARRIVAL, layer)
            assert L.moe_ctx_get_option(ctx, L.OPT_TEST_SKIP_ARRIVAL) == layer
            try:
                r = r0.clone()
                t0 = time.time()
                L.moe_stack_forward(g.ctx, descs, r, 1e-6, ws)
                bits = L.moe_status(ctx)
                dt = time.time() - t0
            finally:
                L.moe_ctx_set_option(ctx, L.OPT_TEST_SKIP_ARRIVAL, -1)
            assert bits & L.STATUS_TIMEOUT
            assert L.moe_ctx_get_option(ctx, L.OPT_LAST_PATH) == 1
            assert 0.2 < dt < 30.0  # gave up after about a second, did not hang
            again = r0.clone()
            L.moe_stack_forward(g.ctx, descs, again, 1e-6, ws)
            assert L.moe_status(ctx) == 0
            assert torch.equal(again, good)
        with pytest.raises(L.MoeError):
            L.moe_ctx_set_option(ctx, L.OPT_TEST_SKIP_ARRIVAL, -2)
    finally:
        g.close()
