"""ctypes binding of libmoe.so (include/moe.h): argument marshalling only.

Every function keeps its C name. Tensors are torch tensors on the context's GPU
(their data_ptr() is passed); streams default to torch's current stream. No
computation happens here: a missing or unloadable library raises, there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

MOE_OK = 0
ERRORS = {-1: "MOE_ERR_ARG", -2: "MOE_ERR_SHAPE", -3: "MOE_ERR_UNSUPPORTED", -4: "MOE_ERR_CUDA",
          -5: "MOE_ERR_NOMEM", -6: "MOE_ERR_EXPERT_ABSENT", -7: "MOE_ERR_NONFINITE",
          -8: "MOE_ERR_TIMEOUT", -9: "MOE_ERR_BOUNDS", -10: "MOE_ERR_WORKSPACE"}
STATUS_EXPERT_ABSENT, STATUS_NONFINITE, STATUS_TIMEOUT, STATUS_BOUNDS = 1, 2, 4, 8
F32, BF16 = 0, 1
Q4_32, Q2_64 = 0, 1
ACT_SWIGLU, ACT_GEGLU_TANH = 0, 1
ROUTER_SOFTMAX, ROUTER_SIGMOID, ROUTER_SIGMOID_NORM = 0, 1, 2


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class Format(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("zero_point", ctypes.c_int)]


class LayerDesc(ctypes.Structure):
    _fields_ = [("slots", ctypes.c_void_p), ("layer", ctypes.c_int), ("H", ctypes.c_int),
                ("E", ctypes.c_int), ("K", ctypes.c_int), ("F", ctypes.c_int),
                ("Wr", ctypes.c_void_p), ("wr_dtype", ctypes.c_int), ("bias", ctypes.c_void_p),
                ("shared", ctypes.c_void_p), ("F_shared", ctypes.c_int), ("act", ctypes.c_int),
                ("router_scale", ctypes.c_void_p), ("down_scale", ctypes.c_void_p), ("router_kind", ctypes.c_int),
                ("drop_eligible", ctypes.c_void_p), ("drop_protect_pct", ctypes.c_int),
                ("drop_mass_pct", ctypes.c_int), ("omitted_out", ctypes.c_void_p)]


class PolicyParams(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("capacity", ctypes.c_int), ("half_life", ctypes.c_double),
                ("recency_guard", ctypes.c_int), ("decay", ctypes.c_float), ("margin", ctypes.c_float),
                ("min_count", ctypes.c_float), ("swap_every", ctypes.c_int), ("max_swaps", ctypes.c_int)]


POLICY_LRU, POLICY_DECAYED_FREQ, POLICY_LFU_SWAP = 0, 1, 2

_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t

_SIGS = {
    "moe_ctx_create": [_I, ctypes.POINTER(_P)],
    "moe_ctx_destroy": [_P],
    "moe_status": [_P, _P, ctypes.POINTER(ctypes.c_uint32)],
    "moe_ctx_set_option": [_P, _I, _I],
    "moe_ctx_get_option": [_P, _I, ctypes.POINTER(_I)],
    "moe_expert_bytes": [Format, _I, _I, ctypes.POINTER(_SZ)],
    "moe_arena_create": [_P, _SZ, ctypes.POINTER(_P)],
    "moe_arena_destroy": [_P],
    "moe_slots_create": [_P, _P, _I, _I, Format, _I, _I, _I, ctypes.POINTER(_P)],
    "moe_slots_destroy": [_P],
    "moe_slot_load": [_P, _I, _I, _P, _SZ, _P],
    "moe_slot_evict": [_P, _I, _I, _P],
    "moe_slot_lookup": [_P, _I, _I, ctypes.POINTER(ctypes.c_int32)],
    "moe_router_topk": [_P, _P, _I, _I, _I, _P, _I, _P, _I, _I, _P, _P, _P, _P],
    "moe_bucket": [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P],
    "moe_layer_workspace": [ctypes.POINTER(LayerDesc), _I, ctypes.POINTER(_SZ)],
    "moe_expert_ffn": [_P, ctypes.POINTER(LayerDesc), _P, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "moe_layer_forward": [_P, ctypes.POINTER(LayerDesc), _P, _I, _I, _P, _P, _P, _P, _SZ, _P],
    "moe_layer_forward_static": [_P, ctypes.POINTER(LayerDesc), _P, _I, _I, _P, _P, _P, _P],
    "moe_layer_forward_host": [_P, ctypes.POINTER(LayerDesc), _P, _I, _I, _P, _P, _SZ, _P],
    "moe_stack_forward": [_P, ctypes.POINTER(LayerDesc), _I, _P, _I, ctypes.c_float, _P, _P, _P, _SZ,
                          _P],
    "moe_stack_forward_host": [_P, ctypes.POINTER(LayerDesc), _I, _P, _I, ctypes.c_float, _P, _SZ, _P],
    "moe_rmsnorm_bf16": [_P, _P, _I, _I, ctypes.c_float, _P, _P],
    "moe_policy_create": [ctypes.POINTER(PolicyParams), _I, _I, ctypes.POINTER(_P)],
    "moe_policy_destroy": [_P],
    "moe_policy_seed": [_P, _P, _P, _I, ctypes.POINTER(_I)],
    "moe_policy_route": [_P, _I, _P, _I, _P, _P, _P, _P, ctypes.POINTER(_I)],
    "moe_policy_route_token": [_P, _P, _I, _I, _P, _P, _P, _P, _P, _I, ctypes.POINTER(_I)],
    "moe_policy_end_token": [_P, _P, _P, _P, _P, _I, ctypes.POINTER(_I)],
    "moe_policy_resident": [_P, _I, _I, ctypes.POINTER(_I)],
    "moe_policy_count": [_P, ctypes.POINTER(_I)],
    "moe_policy_apply": [_P, _I, _P, _SZ, _P, _P, _P, _P, _I, _P],
    "moe_policy_belady": [_P, _I, _I, _I, _I, _I, _P, _P, _I, ctypes.POINTER(ctypes.c_longlong)],
}


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libmoe.so (building it with nvcc first when missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build_if_missing else _build.LIB
    if not os.path.exists(path):
        raise MoeError(-4, f"CUDA library not built: {path}")
    lib = ctypes.CDLL(path)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = _I
    lib.moe_last_error.argtypes = []
    lib.moe_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(rc: int):
    if rc != MOE_OK:
        raise MoeError(rc, _lib.moe_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise MoeError(-1, f"unsupported dtype {t.dtype}")


# ---------------------------------------------------------------- handles

def moe_ctx_create(device: int = 0) -> int:
    out = _P()
    _check(load().moe_ctx_create(device, ctypes.byref(out)))
    return out.value


def moe_ctx_destroy(ctx: int):
    _check(load().moe_ctx_destroy(ctx))


OPT_PERSISTENT_DECODE = 1
OPT_LAST_PATH = 2
OPT_PREFILL_MIN_T = 3
OPT_TEST_SKIP_ARRIVAL = 4


def moe_ctx_set_option(ctx: int, option: int, value: int):
    _check(load().moe_ctx_set_option(ctx, option, value))


def moe_ctx_get_option(ctx: int, option: int) -> int:
    out = _I()
    _check(load().moe_ctx_get_option(ctx, option, ctypes.byref(out)))
    return out.value


def moe_status(ctx: int, stream=None) -> int:
    bits = ctypes.c_uint32()
    _check(load().moe_status(ctx, _stream(stream), ctypes.byref(bits)))
    return bits.value


def moe_expert_bytes(kind: int, zero_point: int, H: int, F: int) -> int:
    out = _SZ()
    _check(load().moe_expert_bytes(Format(kind, zero_point), H, F, ctypes.byref(out)))
    return out.value


def moe_arena_create(ctx: int, nbytes: int) -> int:
    out = _P()
    _check(load().moe_arena_create(ctx, nbytes, ctypes.byref(out)))
    return out.value


def moe_arena_destroy(arena: int):
    _check(load().moe_arena_destroy(arena))


def moe_slots_create(ctx: int, arena: int, n_layers: int, n_experts: int, kind: int, zero_point: int,
                     H: int, F: int, capacity: int) -> int:
    out = _P()
    _check(load().moe_slots_create(ctx, arena, n_layers, n_experts, Format(kind, zero_point), H, F,
                                   capacity, ctypes.byref(out)))
    return out.value


def moe_slots_destroy(slots: int):
    _check(load().moe_slots_destroy(slots))


def moe_slot_load(slots: int, layer: int, expert: int, blob, nbytes: int | None = None, stream=None):
    """blob: torch uint8 tensor (host or device) or a raw pointer with nbytes."""
    if nbytes is None:
        nbytes = blob.numel() * blob.element_size()
    _check(load().moe_slot_load(slots, layer, expert, _ptr(blob), nbytes, _stream(stream)))


def moe_slot_evict(slots: int, layer: int, expert: int, stream=None):
    _check(load().moe_slot_evict(slots, layer, expert, _stream(stream)))


def moe_slot_lookup(slots: int, layer: int, expert: int) -> int:
    out = ctypes.c_int32()
    _check(load().moe_slot_lookup(slots, layer, expert, ctypes.byref(out)))
    return out.value


# ---------------------------------------------------------------- steps

def moe_router_topk(ctx: int, x, Wr, bias, K: int, logits, ids, w, stream=None):
    T, H = x.shape
    E = Wr.shape[0]
    _check(load().moe_router_topk(ctx, _ptr(x), dtype_code(x), T, H, _ptr(Wr), dtype_code(Wr),
                                  _ptr(bias), E, K, _ptr(logits), _ptr(ids), _ptr(w), _stream(stream)))


def moe_bucket(ctx: int, ids, E: int, counts, offsets, perm, active, n_active, stream=None):
    T, K = ids.shape
    _check(load().moe_bucket(ctx, _ptr(ids), T, K, E, _ptr(counts), _ptr(offsets), _ptr(perm),
                             _ptr(active), _ptr(n_active), _stream(stream)))


def layer_desc(slots: int, layer: int, H: int, E: int, K: int, F: int, Wr=None, bias=None,
               shared: int | None = None, F_shared: int = 0, act: int = ACT_SWIGLU, router_scale=None,
               down_scale=None, router_kind: int = ROUTER_SOFTMAX, drop_eligible=None, drop_protect_pct: int = 0,
               drop_mass_pct: int = 0, omitted_out=None) -> LayerDesc:
    wr_dtype = dtype_code(Wr) if Wr is not None else BF16
    return LayerDesc(slots, layer, H, E, K, F, _ptr(Wr), wr_dtype, _ptr(bias), shared, F_shared, act,
                     _ptr(router_scale), _ptr(down_scale), router_kind, _ptr(drop_eligible), drop_protect_pct,
                     drop_mass_pct, _ptr(omitted_out))


def moe_layer_workspace(desc: LayerDesc, T_max: int) -> int:
    out = _SZ()
    _check(load().moe_layer_workspace(ctypes.byref(desc), T_max, ctypes.byref(out)))
    return out.value


def moe_expert_ffn(ctx: int, desc: LayerDesc, x, ids, w, offsets, perm, y, ws, stream=None):
    T = x.shape[0]
    _check(load().moe_expert_ffn(ctx, ctypes.byref(desc), _ptr(x), dtype_code(x), T, _ptr(ids), _ptr(w),
                                 _ptr(offsets), _ptr(perm), _ptr(y), _ptr(ws), ws.numel(),
                                 _stream(stream)))


def moe_layer_forward(ctx: int, desc: LayerDesc, x, y, ws, logits=None, ids=None, stream=None):
    T = x.shape[0]
    _check(load().moe_layer_forward(ctx, ctypes.byref(desc), _ptr(x), dtype_code(x), T, _ptr(y),
                                    _ptr(logits), _ptr(ids), _ptr(ws), ws.numel(), _stream(stream)))


def moe_layer_forward_static(ctx: int, desc: LayerDesc, x, y, logits=None, ids=None, stream=None):
    """moe_layer_forward with the library's fixed scratch (no workspace, no allocation)."""
    T = x.shape[0]
    _check(load().moe_layer_forward_static(ctx, ctypes.byref(desc), _ptr(x), dtype_code(x), T, _ptr(y),
                                           _ptr(logits), _ptr(ids), _stream(stream)))


def moe_layer_forward_host(ctx: int, desc: LayerDesc, x_host, y_host, ws, stream=None):
    T = x_host.shape[0]
    _check(load().moe_layer_forward_host(ctx, ctypes.byref(desc), _ptr(x_host), dtype_code(x_host), T,
                                         _ptr(y_host), _ptr(ws), ws.numel(), _stream(stream)))


def moe_stack_forward(ctx: int, descs, resid, eps: float, ws, trace_in=None, trace_logits=None,
                      stream=None):
    arr = (LayerDesc * len(descs))(*descs)
    T = resid.shape[0]
    _check(load().moe_stack_forward(ctx, arr, len(descs), _ptr(resid), T, eps, _ptr(trace_in),
                                    _ptr(trace_logits), _ptr(ws), ws.numel(), _stream(stream)))


def moe_stack_forward_host(ctx: int, descs, resid_host, eps: float, ws, stream=None):
    arr = (LayerDesc * len(descs))(*descs)
    T = resid_host.shape[0]
    _check(load().moe_stack_forward_host(ctx, arr, len(descs), _ptr(resid_host), T, eps, _ptr(ws),
                                         ws.numel(), _stream(stream)))


def moe_rmsnorm_bf16(ctx: int, x, eps: float, out, stream=None):
    T, H = x.shape
    _check(load().moe_rmsnorm_bf16(ctx, _ptr(x), T, H, eps, _ptr(out), _stream(stream)))


# ------------------------------------------------------------ residency policies
# (host arrays: numpy; marshalling only)

def policy_params(kind: int, capacity: int, half_life: float = 32.0, recency_guard: int = 2, decay: float = 0.7,
                  margin: float = 1.5, min_count: float = 2.0, swap_every: int = 4,
                  max_swaps: int = 96) -> PolicyParams:
    return PolicyParams(kind, capacity, half_life, recency_guard, decay, margin, min_count, swap_every, max_swaps)


def _np_ptr(a):
    return None if a is None else a.ctypes.data


class Policy:
    """A moe_policy handle over n_layers x n_experts pairs."""

    def __init__(self, params: PolicyParams, n_layers: int, n_experts: int):
        import numpy as np
        self._np = np
        h = _P()
        _check(load().moe_policy_create(ctypes.byref(params), n_layers, n_experts, ctypes.byref(h)))
        self.h = h.value
        self.n_layers, self.n_experts = n_layers, n_experts
        self.cap = max(params.max_swaps, 1)

    def seed(self, layers, experts) -> int:
        np = self._np
        l = np.ascontiguousarray(layers, dtype=np.int32)
        e = np.ascontiguousarray(experts, dtype=np.int32)
        out = _I()
        _check(load().moe_policy_seed(self.h, _np_ptr(l), _np_ptr(e), l.size, ctypes.byref(out)))
        return out.value

    def route(self, layer: int, ids):
        """Returns (hit [n] uint8, loads [m] int32, evict_layer [m], evict_expert [m])."""
        np = self._np
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        n = ids.size
        hit = np.zeros(n, dtype=np.uint8)
        le = np.zeros(max(n, 1), dtype=np.int32)
        el = np.zeros(max(n, 1), dtype=np.int32)
        ee = np.zeros(max(n, 1), dtype=np.int32)
        m = _I()
        _check(load().moe_policy_route(self.h, layer, _np_ptr(ids), n, _np_ptr(hit), _np_ptr(le), _np_ptr(el),
                                       _np_ptr(ee), ctypes.byref(m)))
        k = m.value
        return hit, le[:k].copy(), el[:k].copy(), ee[:k].copy()

    def route_token(self, ids):
        """ids [n_layers][K]: one token's events for layers 0 .. n_layers - 1, in order.
        Returns (hit [n_layers][K] uint8, load_layer [m], load_expert [m],
        evict_layer [m], evict_expert [m])."""
        np = self._np
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        nl, K = ids.shape
        hit = np.zeros((nl, K), dtype=np.uint8)
        cap = max(nl * K, 1)
        bufs = [np.zeros(cap, dtype=np.int32) for _ in range(4)]
        m = _I()
        _check(load().moe_policy_route_token(self.h, _np_ptr(ids), nl, K, _np_ptr(hit), *[_np_ptr(b) for b in bufs],
                                             cap, ctypes.byref(m)))
        return (hit,) + tuple(b[:m.value].copy() for b in bufs)

    def end_token(self, plan: bool = True):
        """Returns (load_layer, load_expert, evict_layer, evict_expert) of the swaps made."""
        np = self._np
        bufs = [np.zeros(self.cap, dtype=np.int32) for _ in range(4)] if plan else [None] * 4
        m = _I()
        _check(load().moe_policy_end_token(self.h, *[_np_ptr(b) for b in bufs], self.cap, ctypes.byref(m)))
        if not plan:
            return None
        return tuple(b[:m.value].copy() for b in bufs)

    def resident(self, layer: int, expert: int) -> bool:
        out = _I()
        _check(load().moe_policy_resident(self.h, layer, expert, ctypes.byref(out)))
        return bool(out.value)

    def count(self) -> int:
        out = _I()
        _check(load().moe_policy_count(self.h, ctypes.byref(out)))
        return out.value

    def close(self):
        if self.h:
            load().moe_policy_destroy(self.h)
            self.h = None


def moe_policy_apply(slots: int, n_experts: int, blob_ptrs, nbytes: int, load_layer, load_expert, evict_layer,
                     evict_expert, stream=None):
    import numpy as np
    bp = np.ascontiguousarray(blob_ptrs, dtype=np.uint64)
    arrs = [np.ascontiguousarray(a, dtype=np.int32) for a in (load_layer, load_expert, evict_layer, evict_expert)]
    _check(load().moe_policy_apply(slots, n_experts, _np_ptr(bp), nbytes, *[_np_ptr(a) for a in arrs],
                                   arrs[0].size, _stream(stream)))


# the C names, for callers that hold the handle themselves (Policy wraps these)
def moe_policy_create(params: PolicyParams, n_layers: int, n_experts: int) -> int:
    h = _P()
    _check(load().moe_policy_create(ctypes.byref(params), n_layers, n_experts, ctypes.byref(h)))
    return h.value


def moe_policy_destroy(h: int):
    _check(load().moe_policy_destroy(h))


def moe_policy_seed(h: int, layers, experts) -> int:
    import numpy as np
    l = np.ascontiguousarray(layers, dtype=np.int32)
    e = np.ascontiguousarray(experts, dtype=np.int32)
    out = _I()
    _check(load().moe_policy_seed(h, _np_ptr(l), _np_ptr(e), l.size, ctypes.byref(out)))
    return out.value


def moe_policy_route(h: int, layer: int, ids, hit, load_expert, evict_layer, evict_expert) -> int:
    n = _I()
    _check(load().moe_policy_route(h, layer, _np_ptr(ids), ids.size, _np_ptr(hit), _np_ptr(load_expert),
                                   _np_ptr(evict_layer), _np_ptr(evict_expert), ctypes.byref(n)))
    return n.value


def moe_policy_route_token(h: int, ids, hit, load_layer, load_expert, evict_layer, evict_expert, cap: int) -> int:
    n = _I()
    _check(load().moe_policy_route_token(h, _np_ptr(ids), ids.shape[0], ids.shape[1], _np_ptr(hit),
                                         _np_ptr(load_layer), _np_ptr(load_expert), _np_ptr(evict_layer),
                                         _np_ptr(evict_expert), cap, ctypes.byref(n)))
    return n.value


def moe_policy_end_token(h: int, load_layer, load_expert, evict_layer, evict_expert, cap: int) -> int:
    n = _I()
    _check(load().moe_policy_end_token(h, _np_ptr(load_layer), _np_ptr(load_expert), _np_ptr(evict_layer),
                                       _np_ptr(evict_expert), cap, ctypes.byref(n)))
    return n.value


def moe_policy_resident(h: int, layer: int, expert: int) -> bool:
    out = _I()
    _check(load().moe_policy_resident(h, layer, expert, ctypes.byref(out)))
    return bool(out.value)


def moe_policy_count(h: int) -> int:
    out = _I()
    _check(load().moe_policy_count(h, ctypes.byref(out)))
    return out.value


def moe_policy_belady(trace, n_experts: int, capacity: int, seed_layers=None, seed_experts=None) -> int:
    """trace: int32 [T][n_layers][K] (host). Belady's hits with the pool seeded."""
    import numpy as np
    tr = np.ascontiguousarray(trace, dtype=np.int32)
    T, Ln, K = tr.shape
    sl = None if seed_layers is None else np.ascontiguousarray(seed_layers, dtype=np.int32)
    se = None if seed_experts is None else np.ascontiguousarray(seed_experts, dtype=np.int32)
    out = ctypes.c_longlong()
    _check(load().moe_policy_belady(_np_ptr(tr), T, Ln, K, n_experts, capacity, _np_ptr(sl), _np_ptr(se),
                                    0 if sl is None else sl.size, ctypes.byref(out)))
    return out.value
