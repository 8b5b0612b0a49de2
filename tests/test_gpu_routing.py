"""Routing forms beyond the softmax top-k layer, on every path (persistent decode
kernel, multi-kernel, tensor-core prefill), against the oracle:
  - GeGLU-tanh experts;
  - the router input scaled per input dimension and the per-expert down scale
    (kairos README, "The MoE forward");
  - sigmoid top-k routers, plain and normalised (Krasis white paper sec. 5.3);
  - the P/M route-drop rule without renormalisation (Krasis white paper sec. 7.2-7.3).
The oracle routes with the GPU's fp32 logits; the drop rule is decided, as on the
GPU, in fp32 on the GPU's fp32 route weights."""
import numpy as np
import pytest

import oracle
from quantized_expert_ffn_gb300 import _lib as L
from synth import configs as C
from tests.gpu_util import TOL, GpuLayers, rel_err, to_dev

pytestmark = pytest.mark.gpu

# T: 1 and 4 run the persistent kernel, 12 the multi-kernel path, 100 (Gemma, Q4)
# the tensor-core prefill path
CASES = [("q2_layer", 1), ("q2_layer", 4), ("q2_layer", 12), ("gemma_layer", 2), ("gemma_layer", 100)]


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


@pytest.fixture(scope="module")
def layers(ctx):
    made = {name: GpuLayers(ctx, C.CONFIGS[name]) for name in ("q2_layer", "gemma_layer")}
    yield made
    for g in made.values():
        g.close()


def _experts(cfg, ids):
    need = np.unique(ids)
    blobs = C.experts(cfg, 0, need)
    ex = [None] * cfg.E
    for i, e in enumerate(need):
        ex[int(e)] = blobs[i]
    return ex


def _run(g, x, **opts):
    g.opts = opts
    try:
        y, lg, ids = g.forward(x)
        path = L.moe_ctx_get_option(g.ctx, L.OPT_LAST_PATH)
        assert L.moe_status(g.ctx) == 0
    finally:
        g.opts = {}
    return y, lg, ids, path


def _expect_path(cfg, T, path):
    if T >= 64:
        assert path == 2
    elif T <= 8:
        assert path == 1
    else:
        assert path == 0


def _oracle(cfg, x64, lg, **kw):
    lg64 = np.asarray(lg, dtype=np.float64)
    ids, _, _ = oracle.topk(lg64, cfg.K)
    return oracle.layer_forward_routed(cfg.kind, cfg.zero_point, cfg.H, cfg.E, cfg.K, cfg.F, None, None,
                                       _experts(cfg, ids), x64, shared=C.shared_expert(cfg, 0),
                                       F_shared=cfg.F_shared, logits_in=lg64, **kw)


@pytest.mark.parametrize("name,T", CASES)
def test_geglu_tanh_experts(layers, name, T):
    g = layers[name]
    cfg = g.cfg
    x = C.activations(cfg, T, step=1200 + T)
    y, lg, ids, path = _run(g, to_dev(x), act=L.ACT_GEGLU_TANH)
    _expect_path(cfg, T, path)
    r = _oracle(cfg, C.as_f64(x), lg.cpu().numpy(), act=oracle.ACT_GEGLU_TANH)
    assert np.array_equal(ids.cpu().numpy(), r["ids"])
    assert rel_err(y.cpu().numpy(), r["y"]) <= TOL


@pytest.mark.parametrize("name,T", CASES)
def test_router_scale_and_down_scale(torch, layers, name, T):
    g = layers[name]
    cfg = g.cfg
    rng = np.random.default_rng(1300 + T)
    rs = rng.uniform(0.5, 1.5, cfg.H).astype(np.float32)
    ds = rng.uniform(0.5, 2.0, cfg.E).astype(np.float32)
    ds[rng.choice(cfg.E, cfg.E // 8, replace=False)] = 0.0  # zero-scale experts add nothing
    x = C.activations(cfg, T, step=1300 + T)
    y, lg, ids, path = _run(g, to_dev(x), router_scale=to_dev(rs), down_scale=to_dev(ds))
    _expect_path(cfg, T, path)
    # logits of the scaled router input (the GPU accumulates in fp32)
    x64 = C.as_f64(x)
    Wr = C.as_f64(C.router_weights(cfg, 0))
    b = C.router_bias(cfg, 0)
    want_lg = oracle.router_logits_scaled(x64, Wr, rs.astype(np.float64), None if b is None else C.as_f64(b))
    err = np.abs(lg.cpu().numpy() - want_lg).max() / np.abs(want_lg).max()
    assert err <= 1e-5, err
    r = _oracle(cfg, x64, lg.cpu().numpy(), down_scale=ds.astype(np.float64))
    assert np.array_equal(ids.cpu().numpy(), r["ids"])
    assert rel_err(y.cpu().numpy(), r["y"]) <= TOL


@pytest.mark.parametrize("kind", [L.ROUTER_SIGMOID, L.ROUTER_SIGMOID_NORM])
@pytest.mark.parametrize("name,T", CASES)
def test_sigmoid_routers(layers, name, T, kind):
    g = layers[name]
    cfg = g.cfg
    x = C.activations(cfg, T, step=1400 + T)
    y, lg, ids, path = _run(g, to_dev(x), router_kind=kind)
    _expect_path(cfg, T, path)
    r = _oracle(cfg, C.as_f64(x), lg.cpu().numpy(), router_kind=kind)
    assert np.array_equal(ids.cpu().numpy(), r["ids"])
    assert rel_err(y.cpu().numpy(), r["y"]) <= TOL


@pytest.mark.parametrize("name,T", CASES)
def test_route_drop_policy(torch, layers, name, T):
    g = layers[name]
    cfg = g.cfg
    rng = np.random.default_rng(1500 + T)
    el = (rng.random(cfg.E) < 0.6).astype(np.uint8)
    P, M = 50, 15
    x = C.activations(cfg, T, step=1500 + T)
    xd = to_dev(x)
    omitted = torch.full((T,), -1.0, device="cuda")
    y, lg, ids, path = _run(g, xd, drop_eligible=to_dev(el), drop_protect_pct=P, drop_mass_pct=M,
                            omitted_out=omitted)
    _expect_path(cfg, T, path)
    # the GPU's fp32 route weights before the drop (the same arithmetic as the layer's)
    lg2 = torch.empty(T, cfg.E, device="cuda")
    ids2 = torch.empty(T, cfg.K, dtype=torch.int32, device="cuda")
    w2 = torch.empty(T, cfg.K, device="cuda")
    L.moe_router_topk(g.ctx, xd, g.Wr[0], g.bias[0], cfg.K, lg2, ids2, w2)
    torch.cuda.synchronize()
    assert torch.equal(ids2, ids)
    if path != 2:  # the tensor-core router sums in another order; the others agree bitwise
        assert torch.equal(lg2, lg)
    r = _oracle(cfg, C.as_f64(x), lg.cpu().numpy(), drop_eligible=el, drop_protect_pct=P, drop_mass_pct=M,
                drop_w32=w2.cpu().numpy())
    sure = r["margin"] > 1e-5  # decisions not within rounding of flipping
    assert sure.mean() > 0.9
    om = omitted.cpu().numpy()
    assert np.array_equal(om[sure], r["omitted"][sure])
    assert (r["omitted"] > 0).any()  # the policy did drop routes
    yg = y.cpu().numpy()
    assert rel_err(yg[sure], r["y"][sure]) <= TOL
    # without the policy nothing is omitted and the output changes
    omitted.fill_(-1.0)
    y0, _, _, _ = _run(g, xd, omitted_out=omitted)
    assert (omitted == 0).all()
    assert not torch.equal(y0, y)


def test_persistent_and_multikernel_agree_bitwise_with_routing_forms(torch, layers):
    g = layers["q2_layer"]
    cfg = g.cfg
    rng = np.random.default_rng(1600)
    opts = dict(router_scale=to_dev(rng.uniform(0.5, 1.5, cfg.H).astype(np.float32)),
                down_scale=to_dev(rng.uniform(0.5, 2.0, cfg.E).astype(np.float32)),
                router_kind=L.ROUTER_SIGMOID_NORM, act=L.ACT_GEGLU_TANH,
                drop_eligible=to_dev((rng.random(cfg.E) < 0.5).astype(np.uint8)), drop_protect_pct=60,
                drop_mass_pct=20)
    x = to_dev(C.activations(cfg, 4, step=1600))
    ya, la, ia, pa = _run(g, x, **opts)
    L.moe_ctx_set_option(g.ctx, L.OPT_PERSISTENT_DECODE, 0)
    try:
        yb, lb, ib, pb = _run(g, x, **opts)
    finally:
        L.moe_ctx_set_option(g.ctx, L.OPT_PERSISTENT_DECODE, 1)
    assert (pa, pb) == (1, 0)
    assert torch.equal(la, lb) and torch.equal(ia, ib) and torch.equal(ya, yb)


def test_routing_option_checks(layers):
    g = layers["q2_layer"]
    x = to_dev(C.activations(g.cfg, 1, step=1700))
    for bad in (dict(router_kind=3), dict(drop_eligible=to_dev(np.ones(g.cfg.E, np.uint8)), drop_mass_pct=101)):
        with pytest.raises(L.MoeError):
            _run(g, x, **bad)
