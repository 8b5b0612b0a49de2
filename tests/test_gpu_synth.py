"""The CUDA twin of the input generator writes the same bytes as the host one."""
import numpy as np
import pytest

import synth
import synth.device as sdev
from synth import configs as C

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "q2_layer", "gemma_layer"])
def test_device_blobs_equal_host_blobs(name):
    import torch
    cfg = C.CONFIGS[name]
    nb = 3 * cfg.matrix_blocks()
    n = 3
    first = cfg.tag_expert(0, 5)
    dst = torch.empty(n * nb * 18, dtype=torch.uint8, device="cuda")
    sdev.expert_blobs_into(dst, cfg.seed, first, n, nb, cfg.d_lo, cfg.d_hi)
    host = synth.expert_blobs(cfg.seed, range(first, first + n), nb, cfg.d_lo, cfg.d_hi)
    assert np.array_equal(dst.cpu().numpy(), host.reshape(-1))
