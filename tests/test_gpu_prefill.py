"""Prefill-sized windows: Q4 experts run as tcgen05 grouped GEMMs (fp16 operands,
fp32 accumulation in tensor memory). Parity against the oracle on every row (the
bench's 4,096-token window included), against the mma.sync path, and the path
really taken."""
import numpy as np
import pytest

from quantized_expert_ffn_gb300 import _lib as L
from synth import configs as C
from tests.gpu_util import TOL, GpuLayers, oracle_layer, oracle_layer_by_bucket, rel_err, to_dev

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


def _coverage(counts, nc=256):
    """Column groups of <= nc live pairs per expert (the plan's split) and the B box
    height each group's tile loads (round-up(n, 16) to the next of 16..256)."""
    sizes = []
    for c in counts[counts > 0]:
        sizes += [nc] * (int(c) // nc) + ([int(c) % nc] if c % nc else [])
    sizes = np.array(sizes)
    r16 = (sizes + 15) // 16 * 16
    boxes = np.select([r16 <= 16, r16 <= 32, r16 <= 64, r16 <= 128], [16, 32, 64, 128], 256)
    return sizes, {int(b): int((boxes == b).sum()) for b in (16, 32, 64, 128, 256)}


def _check_every_row(g, cfg, T, step):
    x = _x(cfg, T, step=step)
    y, lg, ids, path = _forward(g, to_dev(x))
    assert path == 2  # tensor-core grouped GEMMs
    r = oracle_layer_by_bucket(cfg, 0, C.as_f64(x), lg.cpu().numpy())
    assert np.array_equal(ids.cpu().numpy(), r["ids"])
    err = rel_err(y.cpu().numpy(), r["y"])
    sizes, boxes = _coverage(r["counts"])
    print(f"\nT={T}: {len(sizes)} routed column groups, sizes {sizes.min()}..{sizes.max()}, "
          f"{int((sizes <= 16).sum())} of <= 16 columns, partial last groups "
          f"{int(((sizes % 256) != 0).sum())}; B boxes {boxes}; max rel err {err:.2e}")
    assert err <= TOL, err
    return boxes


@pytest.mark.parametrize("T", [64, 100, 1000])
def test_prefill_matches_oracle_on_every_row(gemma, T):
    _check_every_row(gemma, gemma.cfg, T, 900 + T)


def test_prefill_full_window_matches_oracle_on_every_row(ctx):
    # the 4,096-token window the bench times (same configuration, same inputs): every
    # row against the oracle; with 128 experts and the calibrated Zipf skew it takes
    # every B box height, groups of <= 16 columns, partial last groups of the large
    # buckets, and both experts' last M-tiles (704 = 11 x 64 gate/up rows, 2,816 =
    # 22 x 128 down rows; the shared expert's 2,112 = 33 x 64)
    cfg = C.CONFIGS["prefill"]
    g = GpuLayers(ctx, cfg)
    try:
        boxes = _check_every_row(g, cfg, 4096, 4096)
        assert all(v > 0 for v in boxes.values()), boxes
    finally:
        g.close()


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
