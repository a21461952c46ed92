"""Seeded synthetic inputs for the routed-expert FFN layer (both sides use these bytes).

This package draws the random inputs and nothing else: no dequantisation, no
routing, no FFN arithmetic. The CPU oracle and the CUDA library both consume
what it returns. The generator itself is C (``synth.c``) so that the tens of
gigabytes of expert weights a 36-layer decode stack needs come out in seconds.

Workloads (shapes and distributions of the layers the pages run):

* ``tiny``    T=4, d=256, ffn=512, E=8, k=2, no shared expert, one layer, seed 0.
* ``decode``  T=1, d=ffn=2880, E=128, k=4: a gpt-oss-120B-shaped MoE layer
              ("Neural Server" technical page, section "What it runs on and what
              it runs": hidden 2880, 128 experts, four active per token), 36 layers.
* ``verify``  T=16, same shapes, router bias = Zipf(1.1) log-probabilities over a
              random permutation of the experts (skewed buckets), 36 layers.
* ``small``   T=8, d=2048, ffn=512, E=256, k=8, shared expert ffn=2048, 48 layers.
* ``prefill`` T=1024, d=ffn=2880, E=128, k=4, no bias, 4 layers.

* ``prefill16k`` T=16384, same shapes, one layer: a ridge-crossing prompt chunk
              (512 tokens per expert on average).
* ``affine3`` T=1, d=2560, ffn=640, E=512, k=10, shared expert ffn=640, 48 layers,
              3-bit affine group-64 experts ("Running Qwen3.8-Flash-Next on a
              32 GB Mac with Transformers", architecture and the table of where
              every weight lives; the shared expert's ffn is not printed there
              and is taken equal to the routed one).
Layer ``l`` of workload number ``c`` (tiny=1, decode=2, verify=3, small=4,
prefill=5, prefill16k=6, affine3=7) uses seed ``1000*c + l``; the tiny layer uses seed 0.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsynth.so")
_lock = threading.Lock()
_lib = None


@dataclass(frozen=True)
class Workload:
    name: str
    number: int
    T: int
    d: int
    ffn: int
    E: int
    k: int
    shared_ffn: int
    layers: int
    zipf_bias: float  # 0.0 = no router bias
    scale_lo: int = 120
    scale_hi: int = 124
    affine_bits: int = 0  # 0: MXFP4 experts; else affine group-64 experts with codes of this width

    def seed(self, layer: int) -> int:
        return 0 if self.name == "tiny" else 1000 * self.number + layer

    @property
    def n_experts_stored(self) -> int:
        return self.E + (1 if self.shared_ffn > 0 else 0)

    def code_bytes(self, f: int | None = None) -> int:
        f = self.ffn if f is None else f
        return 3 * f * self.d // 2

    def scale_bytes(self, f: int | None = None) -> int:
        f = self.ffn if f is None else f
        return 3 * f * self.d // 32

    def expert_bytes(self, f: int | None = None) -> int:
        return self.code_bytes(f) + self.scale_bytes(f)

    @property
    def total_code_bytes(self) -> int:
        return self.E * self.code_bytes() + (self.code_bytes(self.shared_ffn) if self.shared_ffn else 0)

    @property
    def total_scale_bytes(self) -> int:
        return self.E * self.scale_bytes() + (self.scale_bytes(self.shared_ffn) if self.shared_ffn else 0)

    def affine_bytes(self, f: int | None = None) -> int:
        """Bytes of one affine expert: codes of its 3 f d weights, a bf16 scale and bias per 64."""
        f = self.ffn if f is None else f
        n = 3 * f * self.d
        return n * self.affine_bits // 8 + n // 16

    @property
    def total_affine_bytes(self) -> int:
        return self.E * self.affine_bytes() + (self.affine_bytes(self.shared_ffn) if self.shared_ffn else 0)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS: dict[str, Workload] = {
    "tiny": Workload("tiny", 1, T=4, d=256, ffn=512, E=8, k=2, shared_ffn=0, layers=1, zipf_bias=0.0),
    "decode": Workload("decode", 2, T=1, d=2880, ffn=2880, E=128, k=4, shared_ffn=0, layers=36, zipf_bias=0.0),
    "verify": Workload("verify", 3, T=16, d=2880, ffn=2880, E=128, k=4, shared_ffn=0, layers=36, zipf_bias=1.1),
    "small": Workload("small", 4, T=8, d=2048, ffn=512, E=256, k=8, shared_ffn=2048, layers=48, zipf_bias=0.0),
    "prefill": Workload("prefill", 5, T=1024, d=2880, ffn=2880, E=128, k=4, shared_ffn=0, layers=4, zipf_bias=0.0),
    # a ridge-crossing prompt chunk: 512 tokens per expert on average, where the expert GEMMs reuse every
    # weight tile across many token blocks and the tensor cores, not HBM, bind
    "prefill16k": Workload("prefill16k", 6, T=16384, d=2880, ffn=2880, E=128, k=4, shared_ffn=0, layers=1,
                           zipf_bias=0.0),
    # decode of the affine-expert model: 512 routed experts of ffn 640 (top 10) and one shared expert per layer,
    # 3-bit codes with a bf16 scale and bias per 64 weights
    "affine3": Workload("affine3", 7, T=1, d=2560, ffn=640, E=512, k=10, shared_ffn=640, layers=48, zipf_bias=0.0,
                        affine_bits=3),
}


def build(force: bool = False) -> str:
    """Compile the generator (plain C, no contraction so x86-64 and AArch64 agree)."""
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
                               "-o", tmp, src, "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i32, vp, sz = ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
            lib.synth_u64.argtypes = [u64, u64, u64]
            lib.synth_u64.restype = u64
            lib.synth_x.argtypes = [u64, i32, i32, vp]
            lib.synth_router.argtypes = [u64, i32, i32, vp]
            lib.synth_bias_zipf.argtypes = [u64, i32, ctypes.c_double, vp]
            lib.synth_shared_gate.argtypes = [u64, i32, vp]
            lib.synth_code_bytes.argtypes = [u64, u64, sz, vp]
            lib.synth_scale_bytes.argtypes = [u64, u64, sz, i32, i32, vp]
            lib.synth_experts.argtypes = [u64, i32, i32, i32, i32, i32, i32, vp, vp, i32]
            lib.synth_experts.restype = i32
            lib.synth_experts_affine.argtypes = [u64, i32, i32, i32, i32, i32, vp, i32]
            lib.synth_experts_affine.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def gen_x(seed: int, T: int, d: int) -> np.ndarray:
    """bf16 bit patterns, shape [T, d], dtype uint16."""
    x = np.empty((T, d), dtype=np.uint16)
    if x.size:
        _load().synth_x(seed, T, d, _ptr(x))
    return x


def gen_router(seed: int, E: int, d: int) -> np.ndarray:
    w = np.empty((E, d), dtype=np.float32)
    _load().synth_router(seed, E, d, _ptr(w))
    return w


def gen_shared_gate(seed: int, d: int) -> np.ndarray:
    """Shared-expert gate row w_sg [d] fp32, N(0, 1/d), from a stream of its own."""
    w = np.empty((d,), dtype=np.float32)
    _load().synth_shared_gate(seed, d, _ptr(w))
    return w


def gen_bias(seed: int, E: int, s: float) -> np.ndarray:
    b = np.empty((E,), dtype=np.float32)
    _load().synth_bias_zipf(seed, E, s, _ptr(b))
    return b


def gen_experts(wl: Workload, seed: int, codes: np.ndarray | None = None, scales: np.ndarray | None = None,
                nthreads: int | None = None):
    """Codes and scales of all experts of a layer (canonical expert-major layout)."""
    if codes is None:
        codes = np.empty((wl.total_code_bytes,), dtype=np.uint8)
    if scales is None:
        scales = np.empty((wl.total_scale_bytes,), dtype=np.uint8)
    assert codes.nbytes >= wl.total_code_bytes and scales.nbytes >= wl.total_scale_bytes
    if nthreads is None:
        nthreads = max(1, min(32, len(os.sched_getaffinity(0))))
    rc = _load().synth_experts(seed, wl.d, wl.ffn, wl.shared_ffn, wl.E, wl.scale_lo, wl.scale_hi,
                               _ptr(codes), _ptr(scales), nthreads)
    if rc != 0:
        raise RuntimeError("synth_experts failed")
    return codes, scales


def gen_experts_affine(wl: Workload, seed: int, out: np.ndarray | None = None, bits: int | None = None,
                       nthreads: int | None = None) -> np.ndarray:
    """All affine experts of a layer (canonical affine layout, expert-major; shared expert last)."""
    bits = wl.affine_bits if bits is None else bits
    w = wl.with_(affine_bits=bits)
    if out is None:
        out = np.empty((w.total_affine_bytes,), dtype=np.uint8)
    assert out.nbytes >= w.total_affine_bytes
    if nthreads is None:
        nthreads = max(1, min(32, len(os.sched_getaffinity(0))))
    if _load().synth_experts_affine(seed, wl.d, wl.ffn, wl.shared_ffn, wl.E, bits, _ptr(out), nthreads) != 0:
        raise RuntimeError("synth_experts_affine failed")
    return out


def gen_layer(wl: Workload, layer: int = 0, T: int | None = None, with_experts: bool = True) -> dict:
    """All inputs of one layer: x (bf16 bits), router weights, optional bias, expert codes/scales."""
    seed = wl.seed(layer)
    T = wl.T if T is None else T
    out = {
        "seed": seed,
        "x": gen_x(seed, T, wl.d),
        "w_router": gen_router(seed, wl.E, wl.d),
        "bias": gen_bias(seed, wl.E, wl.zipf_bias) if wl.zipf_bias > 0 else None,
    }
    if with_experts and wl.affine_bits:
        out["experts"] = gen_experts_affine(wl, seed)
    elif with_experts:
        out["codes"], out["scales"] = gen_experts(wl, seed)
    return out


def bf16_bits_to_f32(x: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (x.astype(np.uint32) << 16).view(np.float32)
