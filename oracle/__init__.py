"""fp64 CPU oracle for the routed mixture-of-experts FFN layer.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers. The CUDA library never imports,
links or executes anything here, and nothing here imports the CUDA library.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64, index-order loops). This
module compiles it with gcc and wraps it with ctypes over numpy arrays.

Functions and the passages they follow:
  f16_to_f64, dequant, expert_bytes -- Strata article, "The byte budget, in code"
      (Q2_0 block = 64 weights, 16 bytes of 2-bit codes + an fp16 scale; expert =
      gate, up, down) and "The CPU kernels" (codes {0,1,2,3} = {-1,0,1,2} x scale,
      2-bit unpack order); Q4 blocks of 32 with w = d*(q-8) as the tiny layer's
      configuration states.
  router_logits, topk -- kairos-engine README, "The MoE forward" (router GEMM to
      per-expert logits, top-k); Krasis white paper sec. 5.3 (select top-k ids and
      weights); softmax over all experts renormalised over the K selected.
  bucket -- kairos-engine README, "The MoE forward" (expert-major buckets).
  expert_ffn -- Krasis white paper sec. 5.3 and 16.8 (bias-free SwiGLU experts).
  layer_forward -- Krasis white paper sec. 5.3 (weighted reduce), Finding 2 (one
      fixed reduction order), sec. 7.5 (zero-weight slots add nothing); kairos
      README (shared and routed branches summed).
  rmsnorm -- kairos-engine README, "The MoE forward" ("normalise" before routing).

Every function here is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

Q4 = 0
Q2 = 1
ACT_SWIGLU = 0
ACT_GEGLU_TANH = 1
STATUS_ABSENT = 1
STATUS_NONFINITE = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libmoe_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/libmoe_oracle.so (gcc, -O2, no fp contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-std=c11", "-D_DEFAULT_SOURCE", "-O2", "-ffp-contract=off",
                           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    d, i, i64 = ctypes.c_double, ctypes.c_int, ctypes.c_int64
    p = ctypes.c_void_p
    lib.orc_f16_to_f64.restype = d
    lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.orc_expert_bytes.restype = i64
    lib.orc_expert_bytes.argtypes = [i, i, i]
    lib.orc_dequant.restype = None
    lib.orc_dequant.argtypes = [i, i, p, i64, p]
    lib.orc_router_logits.restype = None
    lib.orc_router_logits.argtypes = [p, i, i, p, i, p, p]
    lib.orc_topk.restype = i
    lib.orc_topk.argtypes = [p, i, i, i, p, p]
    lib.orc_bucket.restype = None
    lib.orc_bucket.argtypes = [p, i, i, i, p, p, p, p, p]
    lib.orc_expert_ffn.restype = None
    lib.orc_expert_ffn.argtypes = [i, i, i, p, i, i, p, i, p]
    lib.orc_layer_forward.restype = i
    lib.orc_layer_forward.argtypes = [i, i, i, i, i, i, i, p, p, p, p, i, p, i, p, p, p, p, p]
    lib.orc_rmsnorm.restype = None
    lib.orc_rmsnorm.argtypes = [p, i, i, d, p]
    lib.orc_router_logits_scaled.restype = None
    lib.orc_router_logits_scaled.argtypes = [p, i, i, p, i, p, p, p]
    lib.orc_route_weights.restype = None
    lib.orc_route_weights.argtypes = [i, p, i, p]
    lib.orc_route_drop.restype = i
    lib.orc_route_drop.argtypes = [p, p, i, i, i, p, p, p]
    lib.orc_layer_forward_routed.restype = i
    lib.orc_layer_forward_routed.argtypes = [i, i, i, i, i, i, i, p, p, p, i, p, p, i, i, p, p, p, i, p, i, p,
                                             p, p, p, p, p]
    _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint8)


def f16_to_f64(bits: int) -> float:
    return _load().orc_f16_to_f64(int(bits) & 0xFFFF)


def block_weights(kind: int) -> int:
    return 64 if kind == Q2 else 32


def expert_bytes(kind: int, H: int, F: int) -> int:
    return int(_load().orc_expert_bytes(kind, H, F))


def dequant(kind: int, zero_point: int, blocks, n_weights: int) -> np.ndarray:
    blocks = _u8(blocks)
    assert n_weights % block_weights(kind) == 0
    assert blocks.size >= n_weights // block_weights(kind) * 18
    out = np.empty(n_weights, dtype=np.float64)
    _load().orc_dequant(kind, zero_point, _ptr(blocks), n_weights, _ptr(out))
    return out


def router_logits(x, Wr, bias=None) -> np.ndarray:
    x = _f64(x)
    Wr = _f64(Wr)
    T, H = x.shape
    E = Wr.shape[0]
    assert Wr.shape == (E, H)
    b = None if bias is None else _f64(bias)
    out = np.empty((T, E), dtype=np.float64)
    _load().orc_router_logits(_ptr(x), T, H, _ptr(Wr), E, _ptr(b), _ptr(out))
    return out


def topk(logits, K: int):
    """Returns (ids [T][K] int32, w [T][K] f64, nonfinite flag)."""
    logits = _f64(logits)
    T, E = logits.shape
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    bad = _load().orc_topk(_ptr(logits), T, E, K, _ptr(ids), _ptr(w))
    return ids, w, bool(bad)


def bucket(ids, E: int):
    """Returns dict(counts [E], offsets [E+1], perm [T*K], active [n_active])."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, K = ids.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(max(T * K, 1), dtype=np.int32)
    active = np.empty(max(E, 1), dtype=np.int32)
    na = np.zeros(1, dtype=np.int32)
    _load().orc_bucket(_ptr(ids), T, K, E, _ptr(counts), _ptr(offsets), _ptr(perm),
                       _ptr(active), _ptr(na))
    return dict(counts=counts, offsets=offsets, perm=perm[:T * K], active=active[:int(na[0])])


def expert_ffn(kind: int, zero_point: int, blob, H: int, F: int, x, act: int = ACT_SWIGLU):
    blob = _u8(blob)
    assert blob.size >= expert_bytes(kind, H, F)
    x = _f64(x)
    x2 = x.reshape(-1, H)
    y = np.empty_like(x2)
    _load().orc_expert_ffn(kind, zero_point, act, _ptr(blob), H, F, _ptr(x2), x2.shape[0], _ptr(y))
    return y.reshape(x.shape)


def layer_forward(kind: int, zero_point: int, H: int, E: int, K: int, F: int, Wr, bias,
                  experts, x, shared=None, F_shared: int = 0, logits_in=None,
                  act: int = ACT_SWIGLU):
    """experts: list of E uint8 blobs (None = absent). Returns dict(y, ids, w, logits, status)."""
    x = _f64(x)
    T = x.shape[0]
    assert x.shape == (T, H) and len(experts) == E
    Wr_ = None if Wr is None else _f64(Wr)
    b = None if bias is None else _f64(bias)
    blobs = [None if e is None else _u8(e) for e in experts]
    table = (ctypes.c_void_p * E)(*[None if e is None else e.ctypes.data for e in blobs])
    sh = None if shared is None else _u8(shared)
    li = None if logits_in is None else _f64(logits_in)
    if li is None:
        assert Wr_ is not None and Wr_.shape == (E, H)
    y = np.empty((T, H), dtype=np.float64)
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    logits = np.empty((T, E), dtype=np.float64)
    status = _load().orc_layer_forward(kind, zero_point, act, H, E, K, F, _ptr(Wr_), _ptr(b),
                                       ctypes.cast(table, ctypes.c_void_p), _ptr(sh), F_shared,
                                       _ptr(x), T, _ptr(li), _ptr(y), _ptr(ids), _ptr(w),
                                       _ptr(logits))
    return dict(y=y, ids=ids, w=w, logits=logits, status=int(status))


ROUTER_SOFTMAX, ROUTER_SIGMOID, ROUTER_SIGMOID_NORM = 0, 1, 2


def router_logits_scaled(x, Wr, scale, bias=None) -> np.ndarray:
    """logits = Wr (x * scale) (+ bias), the router input scaled per input dimension."""
    x = _f64(x)
    Wr = _f64(Wr)
    T, H = x.shape
    E = Wr.shape[0]
    sc = _f64(scale)
    assert Wr.shape == (E, H) and sc.shape == (H,)
    b = None if bias is None else _f64(bias)
    out = np.empty((T, E), dtype=np.float64)
    _load().orc_router_logits_scaled(_ptr(x), T, H, _ptr(Wr), E, _ptr(b), _ptr(sc), _ptr(out))
    return out


def route_weights(kind: int, sel_logits) -> np.ndarray:
    """Route weights of the K chosen logits (rank order) for a router kind."""
    l = _f64(sel_logits)
    w = np.empty_like(l)
    _load().orc_route_weights(kind, _ptr(l), l.size, _ptr(w))
    return w


def route_drop(w32, eligible, P: int, M: int):
    """The P/M drop rule on one token's fp32 route weights; returns (weights after the
    drop (f32), dropped count, dropped share (f32), decision margin)."""
    w = np.ascontiguousarray(w32, dtype=np.float32)
    el = _u8(eligible)
    K = w.size
    assert el.size == K and K <= 64
    out = np.empty_like(w)
    share = np.zeros(1, dtype=np.float32)
    margin = np.zeros(1, dtype=np.float64)
    n = _load().orc_route_drop(_ptr(w), _ptr(el), K, P, M, _ptr(out), _ptr(share), _ptr(margin))
    return out, int(n), float(share[0]), float(margin[0])


def layer_forward_routed(kind: int, zero_point: int, H: int, E: int, K: int, F: int, Wr, bias, experts, x,
                         shared=None, F_shared: int = 0, logits_in=None, act: int = ACT_SWIGLU,
                         router_scale=None, router_kind: int = ROUTER_SOFTMAX, down_scale=None,
                         drop_eligible=None, drop_protect_pct: int = 0, drop_mass_pct: int = 0, drop_w32=None):
    """layer_forward with a scaled router input, a router kind, the drop rule and a
    per-expert down scale. Returns dict(y, ids, w, omitted, margin, status)."""
    x = _f64(x)
    T = x.shape[0]
    assert x.shape == (T, H) and len(experts) == E
    Wr_ = None if Wr is None else _f64(Wr)
    b = None if bias is None else _f64(bias)
    rs = None if router_scale is None else _f64(router_scale)
    ds = None if down_scale is None else _f64(down_scale)
    de = None if drop_eligible is None else _u8(drop_eligible)
    dw = None if drop_w32 is None else np.ascontiguousarray(drop_w32, dtype=np.float32)
    blobs = [None if e is None else _u8(e) for e in experts]
    table = (ctypes.c_void_p * E)(*[None if e is None else e.ctypes.data for e in blobs])
    sh = None if shared is None else _u8(shared)
    li = None if logits_in is None else _f64(logits_in)
    if li is None:
        assert Wr_ is not None and Wr_.shape == (E, H)
    y = np.empty((T, H), dtype=np.float64)
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    omitted = np.zeros(T, dtype=np.float32)
    margin = np.ones(T, dtype=np.float64)
    status = _load().orc_layer_forward_routed(kind, zero_point, act, H, E, K, F, _ptr(Wr_), _ptr(b), _ptr(rs),
                                              router_kind, _ptr(ds), _ptr(de), drop_protect_pct, drop_mass_pct,
                                              _ptr(dw), ctypes.cast(table, ctypes.c_void_p), _ptr(sh), F_shared,
                                              _ptr(x), T, _ptr(li), _ptr(y), _ptr(ids), _ptr(w), _ptr(omitted),
                                              _ptr(margin))
    return dict(y=y, ids=ids, w=w, omitted=omitted, margin=margin, status=int(status))


def rmsnorm(x, eps: float = 1e-6) -> np.ndarray:
    x = _f64(x)
    T, H = x.shape
    out = np.empty_like(x)
    _load().orc_rmsnorm(_ptr(x), T, H, float(eps), _ptr(out))
    return out
