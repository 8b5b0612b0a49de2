"""moe_layer_forward_static: the layer entry point for callers that cannot
allocate device memory (it runs on the library's fixed 4 MiB scratch array).

Checked against moe_layer_forward with a caller workspace on the same inputs,
on two calls in a row (the second call finds the first call's leftovers in the
shared scratch): both run the same kernels, so ids, logits and outputs must be
the same bits. This file is collected last on purpose."""
import pytest

from quantized_expert_ffn_gb300 import _lib as L
from synth import configs as C
from tests.gpu_util import GpuLayers, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import torch
    torch.cuda.init()
    c = L.moe_ctx_create(0)
    yield c
    L.moe_ctx_destroy(c)


@pytest.mark.parametrize("name,T", [("q2_layer", 4), ("gemma_layer", 8)])
def test_static_scratch_matches_workspace_entry_point(ctx, name, T):
    import torch
    cfg = C.CONFIGS[name]
    g = GpuLayers(ctx, cfg)
    try:
        desc = g.desc()
        for step in (0, 1):
            x = to_dev(C.activations(cfg, T, step=900 + step))
            y_ref, logits_ref, ids_ref = g.forward(x)
            outs = []
            for _ in range(2):  # two calls in a row on the shared scratch
                y = torch.full((T, cfg.H), float("nan"), device="cuda")
                logits = torch.empty(T, cfg.E, device="cuda")
                ids = torch.empty(T, cfg.K, dtype=torch.int32, device="cuda")
                L.moe_layer_forward_static(ctx, desc, x, y, logits=logits, ids=ids)
                torch.cuda.synchronize()
                assert L.moe_status(ctx) == 0
                # the same kernels on the same inputs: the same bits, whatever the
                # previous call left in the shared scratch
                assert torch.equal(ids, ids_ref)
                assert torch.equal(logits, logits_ref)
                assert torch.equal(y, y_ref)
                outs.append(y)
            assert torch.equal(outs[1], outs[0])
    finally:
        g.close()


def test_static_scratch_allocates_nothing(ctx):
    # after a first call (which looks up the array's address), further calls leave
    # the device's free memory unchanged
    import torch
    cfg = C.CONFIGS["q2_layer"]
    g = GpuLayers(ctx, cfg)
    try:
        desc = g.desc()
        x = to_dev(C.activations(cfg, 4, step=950))
        y = torch.empty(4, cfg.H, device="cuda")
        L.moe_layer_forward_static(ctx, desc, x, y)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for _ in range(5):
            L.moe_layer_forward_static(ctx, desc, x, y)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert L.moe_status(ctx) == 0
    finally:
        g.close()


def test_static_scratch_rejects_windows_that_do_not_fit(ctx):
    import torch
    cfg = C.CONFIGS["tiny"]
    g = GpuLayers(ctx, cfg)
    try:
        desc = g.desc()
        assert L.moe_layer_workspace(desc, 4096) > 4 * 1024 * 1024
        x = to_dev(C.activations(cfg, 4096))
        y = torch.empty(4096, cfg.H, device="cuda")
        with pytest.raises(L.MoeError) as e:
            L.moe_layer_forward_static(ctx, desc, x, y)
        assert e.value.code == -10
        assert "static scratch" in str(e.value)
    finally:
        g.close()
