"""Build and call the CUDA twin of synth.expert_blobs (synth_dev.cu)."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_dev.cu")
LIB = os.path.join(_HERE, "_build", "libmoe_synth.so")
_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(_SRC):
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = LIB + f".{os.getpid()}.tmp"
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                           "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", "-shared",
                           "-o", tmp, _SRC])
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_expert_blobs.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_longlong,
                                           ctypes.c_ulonglong, ctypes.c_longlong, ctypes.c_double,
                                           ctypes.c_double, ctypes.c_void_p]
        lib.synth_expert_blobs.restype = ctypes.c_int
        _lib = lib
    return _lib


def expert_blobs_into(dst, seed: int, first_tag: int, n_experts: int, n_blocks: int, d_lo: float,
                      d_hi: float, stream=None):
    """Fill the device uint8 tensor dst[n_experts * n_blocks * 18] with the same bytes as
    synth.expert_blobs(seed, range(first_tag, first_tag + n_experts), n_blocks, d_lo, d_hi)."""
    import torch
    assert dst.is_cuda and dst.dtype == torch.uint8 and dst.numel() >= n_experts * n_blocks * 18
    s = (stream or torch.cuda.current_stream()).cuda_stream
    rc = _load().synth_expert_blobs(dst.data_ptr(), n_experts, n_blocks, seed, first_tag, d_lo,
                                    d_hi - d_lo, s)
    if rc != 0:
        raise RuntimeError(f"synth_expert_blobs failed ({rc})")
