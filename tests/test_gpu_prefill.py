"""Prefill-sized windows: Q4 experts run as tcgen05 grouped GEMMs (fp16 operands,
fp32 accumulation in tensor memory). Parity against the oracle on sampled rows,
against the mma.sync path on every row, and the path really taken."""
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


@pytest.fixture(scope="module")
def gemma(ctx):
    g = GpuLayers(ctx, C.CONFIGS["gemma_layer"])
    yield g
    g.close()


def _x(cfg, T, step):
    return C.activations(cfg, T, step=step)


def _forward(g, x):
    y, lg, ids = g.forward(x)
    path = L.moe_ctx_get_option(g.ctx, L.OPT_LAST_PATH)
    assert L.moe_status(g.ctx) == 0
    return y, lg, ids, path


@pytest.mark.parametrize("T,n_rows", [(64, 12), (100, 12), (1000, 10)])
def test_prefill_matches_oracle_on_sampled_rows(gemma, T, n_rows):
    cfg = gemma.cfg
    x = _x(cfg, T, step=900 + T)
    y, lg, ids, path = _forward(gemma, to_dev(x))
    assert path == 2  # tensor-core grouped GEMMs
    rows = np.sort(np.random.default_rng(T).choice(T, size=n_rows, replace=False))
    r = oracle_layer(cfg, 0, C.as_f64(x), lg.cpu().numpy(), tokens=rows)
    assert np.array_equal(ids.cpu().numpy()[rows], r["ids"])
    err = rel_err(y.cpu().numpy()[rows], r["y"])
    assert err <= TOL, err


def test_prefill_fp32_activations(gemma):
    # fp32 x (the bf16 values, exactly) through the tensor-core path: the gather
    # converts it to fp16 rows; the router runs on CUDA cores (its GEMM wants bf16)
    cfg = gemma.cfg
    T = 300
    x = _x(cfg, T, step=940)
    x32 = C.as_f64(x).astype(np.float32)
    y, lg, ids, path = _forward(gemma, to_dev(x32))
    assert path == 2
    rows = np.array([0, 1, 77, 150, 299])
    r = oracle_layer(cfg, 0, C.as_f64(x), lg.cpu().numpy(), tokens=rows)
    assert np.array_equal(ids.cpu().numpy()[rows], r["ids"])
    assert rel_err(y.cpu().numpy()[rows], r["y"]) <= TOL


def test_prefill_close_to_mma_sync_path_on_every_row(gemma):
    cfg = gemma.cfg
    T = 256
    x = to_dev(_x(cfg, T, step=950))
    ya, la, ia, pa = _forward(gemma, x)
    L.moe_ctx_set_option(gemma.ctx, L.OPT_PREFILL_MIN_T, 1 << 20)
    try:
        yb, lb, ib, pb = _forward(gemma, x)
    finally:
        L.moe_ctx_set_option(gemma.ctx, L.OPT_PREFILL_MIN_T, 64)
    assert (pa, pb) == (2, 0)
    # the routers differ only in fp32 summation order (tensor-core GEMM vs per-row
    # CUDA-core order): logits agree to ~1e-6, routing agrees except on exact
    # near-ties, and the outputs of tokens routed alike agree within the tolerance
    assert float((la - lb).abs().max()) <= 1e-4
    same = (ia == ib).all(dim=1).cpu().numpy()
    assert same.mean() >= 0.99
    assert rel_err(ya.cpu().numpy()[same], yb.cpu().numpy()[same]) <= TOL


def test_prefill_deterministic(gemma):
    x = to_dev(_x(gemma.cfg, 300, step=960))
    a, _, _, _ = _forward(gemma, x)
    b, _, _, _ = _forward(gemma, x)
    import torch
    assert torch.equal(a, b)


def test_prefill_threshold_option(gemma):
    assert L.moe_ctx_get_option(gemma.ctx, L.OPT_PREFILL_MIN_T) == 64
    with pytest.raises(L.MoeError):
        L.moe_ctx_set_option(gemma.ctx, L.OPT_PREFILL_MIN_T, 0)
    x = to_dev(_x(gemma.cfg, 63, step=970))
    _, _, _, path = _forward(gemma, x)
    assert path == 0  # below the threshold: mma.sync kernels


def test_q2_stays_on_mma_sync(ctx):
    cfg = C.CONFIGS["q2_layer"]
    g = GpuLayers(ctx, cfg)
    try:
        x = _x(cfg, 80, step=980)
        y, lg, ids, path = _forward(g, to_dev(x))
        assert path == 0
        rows = np.array([0, 41, 79])
        r = oracle_layer(cfg, 0, C.as_f64(x), lg.cpu().numpy(), tokens=rows)
        assert rel_err(y.cpu().numpy()[rows], r["y"]) <= TOL
    finally:
        g.close()
