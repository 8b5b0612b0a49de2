"""Host-side checks of the C ABI: the library builds, loads and exports every
function include/moe.h declares; argument errors come back as codes."""
import os
import re

import pytest

import quantized_expert_ffn_gb300 as q
from quantized_expert_ffn_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src, flags=re.M))
    return names


def test_library_exports_every_declared_function():
    lib = q.load()
    names = _declared()
    assert len(names) >= 20
    for n in sorted(names):
        assert hasattr(lib, n), n
    # and the binding wraps each compute/handle call under the same name
    for n in names - {"moe_last_error"}:
        assert hasattr(L, n), n


def test_expert_bytes_and_argument_errors():
    assert L.moe_expert_bytes(L.Q2_64, 1, 2560, 640) == 1_382_400
    assert L.moe_expert_bytes(L.Q4_32, 8, 2816, 704) == 3_345_408
    assert L.moe_expert_bytes(L.Q4_32, 8, 2816, 2112) == 10_036_224
    with pytest.raises(L.MoeError) as e:
        L.moe_expert_bytes(L.Q2_64, 4, 2560, 640)  # zero point out of range
    assert e.value.code == -1
    with pytest.raises(L.MoeError) as e:
        L.moe_expert_bytes(L.Q2_64, 1, 2560, 600)  # F not a multiple of 64
    assert e.value.code == -2
    with pytest.raises(L.MoeError) as e:
        L.moe_expert_bytes(7, 1, 2560, 640)
    assert e.value.code == -1


def test_context_without_a_device_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(L.MoeError) as e:
        L.moe_ctx_create(0)
    assert e.value.code == -4
    assert "device" in str(e.value)


def test_header_is_plain_c_without_cuda_headers():
    # the boundary is a C ABI: include/moe.h compiles as strict C99 and as C++ with no
    # CUDA or torch header on the include path
    import shutil
    import subprocess
    import tempfile
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = '#include "moe.h"\nint main(void) { moe_ctx *c = 0; (void)c; return (int)sizeof(moe_layer_desc) > 0 ? 0 : 1; }\n'
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "use.c")
        with open(path, "w") as f:
            f.write(src)
        for cc, flags in (("gcc", ["-std=c99", "-pedantic"]), ("g++", ["-std=c++17", "-x", "c++"])):
            if shutil.which(cc) is None:
                continue
            r = subprocess.run([cc, *flags, "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I",
                                os.path.join(root, "include"), path], capture_output=True, text=True)
            assert r.returncode == 0, r.stderr
