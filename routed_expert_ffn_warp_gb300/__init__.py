"""Routed-expert FFN (MoE layer) for NVIDIA GB300 -- Python binding of ``libmoe_gb300.so``.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels (``csrc/``). The functions keep the C ABI's names (``include/moe.h``):
``moe_create``, ``moe_load_router``, ``moe_load_experts``, ``moe_forward``,
``moe_forward_host``, ``moe_get_routing``, ``moe_get_logits``,
``moe_get_status``, ``moe_weight_bytes``, ``moe_last_error``, ``moe_destroy``.
Pointers may come from numpy arrays (host) or torch tensors (host or device);
PyTorch is used for device memory and streams only.

There is no fallback: if the compiled library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_T_TOO_LARGE = -2
MOE_ERR_NOT_LOADED = -3
MOE_ERR_CUDA = -4
MOE_ERR_TIMEOUT = -5
MOE_ERR_NAN_SCALE = -6
MOE_ERR_NOMEM = -7
MOE_OUT_BF16 = 0
MOE_OUT_F32 = 1
MOE_FLAG_TEST_FORCE_TIMEOUT = 1
MOE_FLAG_GENERAL_PATH = 2
MOE_FLAG_TC_GATEUP = 4
MOE_FLAG_NO_TC = 8
MOE_FORMAT_MXFP4 = 0
MOE_FORMAT_AFFINE64 = 1

EXPORTED = ["moe_create", "moe_load_router", "moe_load_shared_gate", "moe_load_experts", "moe_load_experts_affine",
            "moe_forward", "moe_forward_host",
            "moe_get_routing", "moe_get_logits", "moe_get_status", "moe_profile_events", "moe_forward_phases",
            "moe_launches_per_forward", "moe_route_static", "moe_route_static_error", "moe_probe_mma_rate",
            "moe_probe_error", "moe_weight_bytes", "moe_last_error", "moe_destroy"]


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} (code {code})")
        self.code = code


class moe_config(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("ffn", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("shared_ffn", ctypes.c_int), ("t_max", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("flags", ctypes.c_uint), ("expert_begin", ctypes.c_int), ("expert_end", ctypes.c_int),
                ("weight_format", ctypes.c_int), ("weight_bits", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the compiled library (build it with ``routed_expert_ffn_warp_gb300.build``)."""
    global _lib
    if _lib is not None:  # every forward call comes through here: no lock once loaded
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: run `python -m routed_expert_ffn_warp_gb300.build` "
                                   "(there is no CPU fallback)")
            lib = ctypes.CDLL(path)
            vp, i32, P = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER
            lib.moe_create.argtypes = [P(moe_config), i32, P(vp)]
            lib.moe_load_router.argtypes = [vp, vp, vp]
            lib.moe_load_experts.argtypes = [vp, vp, vp]
            lib.moe_load_experts_affine.argtypes = [vp, vp]
            lib.moe_load_experts_affine.restype = i32
            lib.moe_load_shared_gate.argtypes = [vp, vp]
            lib.moe_load_shared_gate.restype = i32
            lib.moe_forward.argtypes = [vp, vp, i32, vp, vp]
            lib.moe_forward_host.argtypes = [vp, vp, i32, vp, vp, i32]
            lib.moe_profile_events.argtypes = [vp, P(vp), i32]
            lib.moe_forward_phases.argtypes = [vp, i32, P(ctypes.c_char_p)]
            lib.moe_launches_per_forward.argtypes = [vp, i32]
            lib.moe_get_routing.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
            lib.moe_get_logits.argtypes = [vp, vp, vp, vp]
            lib.moe_get_status.argtypes = [vp, i32]
            lib.moe_route_static.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp]
            lib.moe_route_static.restype = i32
            lib.moe_route_static_error.argtypes = []
            lib.moe_route_static_error.restype = ctypes.c_char_p
            lib.moe_probe_mma_rate.argtypes = [i32, i32, i32, P(ctypes.c_double), P(ctypes.c_double)]
            lib.moe_probe_mma_rate.restype = i32
            lib.moe_probe_error.argtypes = []
            lib.moe_probe_error.restype = ctypes.c_char_p
            lib.moe_weight_bytes.argtypes = [vp]
            lib.moe_weight_bytes.restype = ctypes.c_size_t
            lib.moe_last_error.argtypes = [vp]
            lib.moe_last_error.restype = ctypes.c_char_p
            lib.moe_destroy.argtypes = [vp]
            lib.moe_destroy.restype = None
            for name in ("moe_create", "moe_load_router", "moe_load_experts", "moe_forward", "moe_forward_host",
                         "moe_get_routing", "moe_get_logits", "moe_get_status", "moe_profile_events",
                         "moe_forward_phases", "moe_launches_per_forward"):
                getattr(lib, name).restype = i32
            _lib = lib
    return _lib


def ptr(a) -> int | None:
    """Address of a numpy array or torch tensor (None stays None)."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        assert a.is_contiguous(), "tensor must be contiguous"
        return a.data_ptr()
    assert a.flags["C_CONTIGUOUS"], "array must be C-contiguous"
    return a.ctypes.data


def stream_handle(stream) -> int | None:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(ctx, rc: int, what: str) -> int:
    if rc < 0:
        msg = load_library().moe_last_error(ctx).decode(errors="replace")
        raise MoeError(rc, f"{what}: {msg}")
    return rc


# ---------------------------------------------------------------- C ABI, same names

def moe_create(cfg: moe_config, device: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(None, load_library().moe_create(ctypes.byref(cfg), device, ctypes.byref(h)), "moe_create")
    return h.value


def moe_load_router(ctx: int, w, bias=None) -> None:
    _check(ctx, load_library().moe_load_router(ctx, ptr(w), ptr(bias)), "moe_load_router")


def moe_load_shared_gate(ctx: int, w=None) -> None:
    _check(ctx, load_library().moe_load_shared_gate(ctx, ptr(w)), "moe_load_shared_gate")


def moe_load_experts(ctx: int, codes, scales) -> None:
    _check(ctx, load_library().moe_load_experts(ctx, ptr(codes), ptr(scales)), "moe_load_experts")


def moe_load_experts_affine(ctx: int, experts) -> None:
    _check(ctx, load_library().moe_load_experts_affine(ctx, ptr(experts)), "moe_load_experts_affine")


def moe_forward(ctx: int, x, T: int, out, stream=None) -> None:
    _check(ctx, load_library().moe_forward(ctx, ptr(x), T, ptr(out), stream_handle(stream)), "moe_forward")


def moe_forward_host(ctx: int, x_host, T: int, out_host, stream=None, synchronize: bool = True) -> None:
    _check(ctx, load_library().moe_forward_host(ctx, ptr(x_host), T, ptr(out_host), stream_handle(stream),
                                                1 if synchronize else 0), "moe_forward_host")


def moe_get_routing(ctx: int, ids=None, gates=None, counts=None, offsets=None, perm=None, stream=None,
                    inv=None) -> None:
    _check(ctx, load_library().moe_get_routing(ctx, ptr(ids), ptr(gates), ptr(counts), ptr(offsets), ptr(perm),
                                               ptr(inv), stream_handle(stream)), "moe_get_routing")


def moe_get_logits(ctx: int, hi=None, lo=None, stream=None) -> None:
    _check(ctx, load_library().moe_get_logits(ctx, ptr(hi), ptr(lo), stream_handle(stream)), "moe_get_logits")


def moe_get_status(ctx: int, clear: bool = False) -> int:
    return load_library().moe_get_status(ctx, 1 if clear else 0)


def moe_profile_events(ctx: int, events=None) -> None:
    """events: list of torch.cuda.Event (created with enable_timing=True) or None to stop."""
    if not events:
        _check(ctx, load_library().moe_profile_events(ctx, None, 0), "moe_profile_events")
        return
    arr = (ctypes.c_void_p * len(events))(*[ev.cuda_event if hasattr(ev, "cuda_event") else ev for ev in events])
    _check(ctx, load_library().moe_profile_events(ctx, arr, len(events)), "moe_profile_events")


def moe_forward_phases(ctx: int, T: int = 1) -> list[str]:
    names = ctypes.c_char_p()
    n = load_library().moe_forward_phases(ctx, T, ctypes.byref(names))
    out = names.value.decode().split(",")
    assert len(out) == n
    return out


def moe_launches_per_forward(ctx: int, T: int) -> int:
    return load_library().moe_launches_per_forward(ctx, T)


def moe_route_static(x, T: int, d: int, w_router, bias, n_experts: int, top_k: int, ids, gates, counts, offsets,
                     perm, stream=None) -> None:
    """Routing without allocation (static device scratch); device pointers throughout."""
    lib = load_library()
    rc = lib.moe_route_static(ptr(x), T, d, ptr(w_router), ptr(bias), n_experts, top_k, ptr(ids), ptr(gates),
                              ptr(counts), ptr(offsets), ptr(perm), stream_handle(stream))
    if rc < 0:
        raise MoeError(rc, "moe_route_static: " + lib.moe_route_static_error().decode(errors="replace"))


def moe_probe_mma_rate(device: int = 0, mmas_per_sm: int = 200000, n: int = 192) -> tuple[float, float]:
    """(TFLOP/s, ms) of the block-scaled MMA kind the expert GEMMs use (M=128, K=32, N=n), measured on `device`."""
    lib = load_library()
    tf, ms = ctypes.c_double(), ctypes.c_double()
    rc = lib.moe_probe_mma_rate(device, mmas_per_sm, n, ctypes.byref(tf), ctypes.byref(ms))
    if rc < 0:
        raise MoeError(rc, lib.moe_probe_error().decode(errors="replace"))
    return tf.value, ms.value


def moe_weight_bytes(ctx: int) -> int:
    return load_library().moe_weight_bytes(ctx)


def moe_last_error(ctx: int | None) -> str:
    return load_library().moe_last_error(ctx).decode(errors="replace")


def moe_destroy(ctx: int | None) -> None:
    if ctx:
        load_library().moe_destroy(ctx)


# ---------------------------------------------------------------- convenience wrapper

@dataclass
class LayerShape:
    d: int
    ffn: int
    n_experts: int
    top_k: int
    shared_ffn: int = 0
    t_max: int = 16
    out_dtype: int = MOE_OUT_BF16
    flags: int = 0
    expert_begin: int = 0  # an expert-parallel shard [expert_begin, expert_end); 0, 0 = every expert
    expert_end: int = 0
    weight_format: int = MOE_FORMAT_MXFP4  # or MOE_FORMAT_AFFINE64 with weight_bits 2, 3, 4 or 8
    weight_bits: int = 0

    def config(self) -> moe_config:
        return moe_config(self.d, self.ffn, self.n_experts, self.top_k, self.shared_ffn, self.t_max,
                          self.out_dtype, self.flags, self.expert_begin, self.expert_end, self.weight_format,
                          self.weight_bits)


class MoeLayer:
    """Owns one context (one layer's weights and workspace) on one device."""

    def __init__(self, shape: LayerShape, device: int = 0):
        self.shape = shape
        self.device = device
        self.ctx = moe_create(shape.config(), device)

    def load(self, w_router, bias, codes, scales, w_shared_gate=None) -> "MoeLayer":
        moe_load_router(self.ctx, w_router, bias)
        moe_load_experts(self.ctx, codes, scales)
        if w_shared_gate is not None:
            moe_load_shared_gate(self.ctx, w_shared_gate)
        return self

    def load_affine(self, w_router, bias, experts, w_shared_gate=None) -> "MoeLayer":
        """Router and affine group-64 experts (canonical affine bytes of every expert, in order)."""
        moe_load_router(self.ctx, w_router, bias)
        moe_load_experts_affine(self.ctx, experts)
        if w_shared_gate is not None:
            moe_load_shared_gate(self.ctx, w_shared_gate)
        return self

    def forward(self, x, T: int, out, stream=None) -> None:
        moe_forward(self.ctx, x, T, out, stream)

    def forward_host(self, x_host, T: int, out_host, stream=None, synchronize: bool = True) -> None:
        moe_forward_host(self.ctx, x_host, T, out_host, stream, synchronize)

    def routing(self, ids=None, gates=None, counts=None, offsets=None, perm=None, stream=None, inv=None) -> None:
        moe_get_routing(self.ctx, ids, gates, counts, offsets, perm, stream, inv)

    def logits(self, hi=None, lo=None, stream=None) -> None:
        moe_get_logits(self.ctx, hi, lo, stream)

    def status(self, clear: bool = False) -> int:
        return moe_get_status(self.ctx, clear)

    def weight_bytes(self) -> int:
        return moe_weight_bytes(self.ctx)

    def close(self) -> None:
        if self.ctx:
            moe_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
