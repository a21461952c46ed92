"""CPU oracle for the routed-expert FFN layer -- TEST INFRASTRUCTURE ONLY.

Python bindings (ctypes) over ``moe_oracle.c``, a plain fp64 C statement of the
layer. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the CUDA library never does, and the
oracle never imports the library. The only inputs the two sides share come
from ``synth`` (seeded random bytes, no arithmetic of the method).

What pins it (tests/test_oracle_*.py): exhaustive E2M1/E8M0 tables against
their bit-field definitions, the 13,219,200-byte expert of the "Neural Server"
technical page, hand-computed closed-form layers, brute-force top-k over all
subsets, exact ties, gate and bucketing invariants, exact power-of-two scaling,
expert-relabel equivariance, and an independent dense float64 PyTorch
restatement on tiny layers. The optional sigmoid-gated shared expert
(tests/test_oracle_shared_gate.py) and the affine group-64 expert format
(tests/test_oracle_affine.py) have pins of their own.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, ENAN_SCALE, ENOMEM = 0, -1, -2, -3


def build(force: bool = False) -> str:
    """Compile the oracle with plain flags (no fast-math, no contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_HERE, "moe_oracle.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, vp, dbl, u8, u16 = ctypes.c_int, ctypes.c_void_p, ctypes.c_double, ctypes.c_uint8, ctypes.c_uint16
            lib.oracle_e2m1.argtypes = [i32]
            lib.oracle_e2m1.restype = dbl
            lib.oracle_e8m0.argtypes = [i32]
            lib.oracle_e8m0.restype = dbl
            lib.oracle_bf16.argtypes = [u16]
            lib.oracle_bf16.restype = dbl
            lib.oracle_mx_element.argtypes = [vp, vp, i32, i32, i32]
            lib.oracle_mx_element.restype = dbl
            lib.oracle_expert_code_bytes.argtypes = [i32, i32]
            lib.oracle_expert_code_bytes.restype = ctypes.c_size_t
            lib.oracle_expert_scale_bytes.argtypes = [i32, i32]
            lib.oracle_expert_scale_bytes.restype = ctypes.c_size_t
            lib.oracle_logits_token.argtypes = [vp, i32, vp, vp, i32, vp]
            lib.oracle_topk_token.argtypes = [vp, i32, i32, vp, vp]
            lib.oracle_bucket.argtypes = [vp, i32, i32, vp, vp, vp, vp]
            lib.oracle_expert_ffn.argtypes = [vp, vp, i32, i32, vp, vp, vp]
            lib.oracle_expert_ffn.restype = i32
            lib.oracle_route.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp]
            lib.oracle_route.restype = i32
            lib.oracle_layer_tokens.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp,
                                                vp]
            lib.oracle_shared_gate_token.argtypes = [vp, i32, vp]
            lib.oracle_shared_gate_token.restype = dbl
            lib.oracle_layer_tokens_shard.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                                      i32, vp, vp]
            lib.oracle_layer_tokens_shard.restype = i32
            lib.oracle_affine_code.argtypes = [vp, i32, i32, i32, i32]
            lib.oracle_affine_code.restype = i32
            lib.oracle_affine_element.argtypes = [vp, vp, vp, i32, i32, i32, i32]
            lib.oracle_affine_element.restype = dbl
            lib.oracle_affine_expert_bytes.argtypes = [i32, i32, i32]
            lib.oracle_affine_expert_bytes.restype = ctypes.c_size_t
            lib.oracle_expert_ffn_affine.argtypes = [vp, i32, i32, i32, vp, vp]
            lib.oracle_expert_ffn_affine.restype = i32
            lib.oracle_layer_tokens_affine.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, i32, vp,
                                                       vp, vp, vp]
            lib.oracle_layer_tokens_affine.restype = i32
            lib.oracle_layer_tokens.restype = i32
            _lib = lib
    return _lib


def _p(a):
    """Address of a C-contiguous array. The caller must hold a reference to `a`
    until the C call returns: never pass a temporary made in the call's own
    argument list (it may be freed before the call runs)."""
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "need a C-contiguous numpy array"
    return a.ctypes.data


def _check(rc: int, what: str):
    if rc != OK:
        raise ValueError(f"oracle {what} failed with code {rc}")


def e2m1(code: int) -> float:
    return _load().oracle_e2m1(code)


def e8m0(e: int) -> float:
    return _load().oracle_e8m0(e)


def bf16(bits: int) -> float:
    return _load().oracle_bf16(bits)


def mx_element(codes: np.ndarray, scales: np.ndarray, K: int, r: int, c: int) -> float:
    return _load().oracle_mx_element(_p(codes), _p(scales), K, r, c)


def expert_code_bytes(d: int, f: int) -> int:
    return _load().oracle_expert_code_bytes(d, f)


def expert_scale_bytes(d: int, f: int) -> int:
    return _load().oracle_expert_scale_bytes(d, f)


def logits_token(x_row: np.ndarray, w_router: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    x_row = np.ascontiguousarray(x_row, dtype=np.uint16)
    w_router = np.ascontiguousarray(w_router, dtype=np.float32)
    E, d = w_router.shape
    out = np.empty((E,), dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    _load().oracle_logits_token(_p(x_row), d, _p(w_router), _p(b), E, _p(out))
    return out


def topk_token(logits: np.ndarray, k: int):
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    ids = np.empty((k,), dtype=np.int32)
    gates = np.empty((k,), dtype=np.float64)
    _load().oracle_topk_token(_p(logits), logits.shape[0], k, _p(ids), _p(gates))
    return ids, gates


def bucket(ids: np.ndarray, E: int):
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    P = ids.shape[0]
    counts = np.empty((E,), dtype=np.int32)
    offsets = np.empty((E + 1,), dtype=np.int32)
    perm = np.empty((P,), dtype=np.int32)
    inv = np.empty((P,), dtype=np.int32)
    _load().oracle_bucket(_p(ids), P, E, _p(counts), _p(offsets), _p(perm), _p(inv))
    return counts, offsets, perm, inv


def expert_ffn(codes_e: np.ndarray, scales_e: np.ndarray, d: int, f: int, x: np.ndarray):
    """One expert on one fp64 input vector; returns (h[f], out[d])."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    h = np.empty((f,), dtype=np.float64)
    out = np.empty((d,), dtype=np.float64)
    codes_e = np.ascontiguousarray(codes_e)
    scales_e = np.ascontiguousarray(scales_e)
    _check(_load().oracle_expert_ffn(_p(codes_e), _p(scales_e),
                                     d, f, _p(x), _p(h), _p(out)), "expert_ffn")
    return h, out


def route(x: np.ndarray, w_router: np.ndarray, bias: np.ndarray | None, k: int) -> dict:
    """Routing of all tokens: logits, ids, gates, counts, offsets, perm, inv."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    w_router = np.ascontiguousarray(w_router, dtype=np.float32)
    T, d = x.shape
    E = w_router.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = {
        "logits": np.empty((T, E), dtype=np.float64),
        "ids": np.empty((T, k), dtype=np.int32),
        "gates": np.empty((T, k), dtype=np.float64),
        "counts": np.empty((E,), dtype=np.int32),
        "offsets": np.empty((E + 1,), dtype=np.int32),
        "perm": np.empty((T * k,), dtype=np.int32),
        "inv": np.empty((T * k,), dtype=np.int32),
    }
    _check(_load().oracle_route(_p(x), T, d, _p(w_router), _p(b), E, k, _p(out["logits"]), _p(out["ids"]),
                                _p(out["gates"]), _p(out["counts"]), _p(out["offsets"]), _p(out["perm"]),
                                _p(out["inv"])), "route")
    return out


def shared_gate_token(x_row: np.ndarray, w_sg: np.ndarray) -> float:
    """sigmoid(w_sg . x_t) of one token (fp64)."""
    x_row = np.ascontiguousarray(x_row, dtype=np.uint16)
    w_sg = np.ascontiguousarray(w_sg, dtype=np.float32)
    return _load().oracle_shared_gate_token(_p(x_row), x_row.shape[0], _p(w_sg))


def layer_tokens(d: int, F: int, E: int, k: int, S: int, x: np.ndarray, w_router: np.ndarray,
                 bias: np.ndarray | None, codes: np.ndarray, scales: np.ndarray, tokens=None,
                 want_h: bool = False, w_shared_gate: np.ndarray | None = None) -> dict:
    """fp64 layer output of the listed tokens (default: all): y [n][d], ids, gates, optional h [n][k][F].
    With w_shared_gate [d] the shared expert's output is scaled by sigmoid(w_shared_gate . x_t)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T = x.shape[0]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = tokens.shape[0]
    y = np.empty((n, d), dtype=np.float64)
    h = np.empty((n, k, F), dtype=np.float64) if want_h else None
    ids = np.empty((n, k), dtype=np.int32)
    gates = np.empty((n, k), dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    sg = None if w_shared_gate is None else np.ascontiguousarray(w_shared_gate, dtype=np.float32)
    w_router = np.ascontiguousarray(w_router, dtype=np.float32)
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    _check(_load().oracle_layer_tokens(d, F, E, k, S, _p(x), _p(w_router),
                                       _p(b), _p(codes), _p(scales),
                                       _p(tokens), n, _p(y), _p(h), _p(ids), _p(gates), _p(sg)), "layer_tokens")
    return {"y": y, "h": h, "ids": ids, "gates": gates, "tokens": tokens}


def host_threads() -> int:
    """Host cores this process may run on (its CPU affinity)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def layer_tokens_parallel(d: int, F: int, E: int, k: int, S: int, x: np.ndarray, w_router: np.ndarray,
                          bias: np.ndarray | None, codes: np.ndarray, scales: np.ndarray, tokens=None,
                          threads: int | None = None, w_shared_gate: np.ndarray | None = None) -> dict:
    """layer_tokens for many tokens on several host threads.

    The token list is cut into contiguous chunks, one oracle_layer_tokens call
    per chunk on a thread pool (ctypes releases the GIL for the duration of the
    C call). Every token is still evaluated alone by the same fp64 code in the
    same order, so the results are bit-identical to one single-threaded call;
    only the wall time changes. Returns the layer_tokens dict plus "threads"."""
    from concurrent.futures import ThreadPoolExecutor

    x = np.ascontiguousarray(x, dtype=np.uint16)
    T = x.shape[0]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = tokens.shape[0]
    threads = host_threads() if threads is None else max(1, int(threads))
    threads = min(threads, max(1, n))
    w_router = np.ascontiguousarray(w_router, dtype=np.float32)
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    _load()  # load and declare the library once, before the threads start
    bounds = [(i * n) // threads for i in range(threads + 1)]

    def run(i):
        return layer_tokens(d, F, E, k, S, x, w_router, bias, codes, scales,
                            tokens=tokens[bounds[i]:bounds[i + 1]], w_shared_gate=w_shared_gate)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(run, range(threads)))
    out = {key: np.concatenate([pt[key] for pt in parts]) for key in ("y", "ids", "gates")}
    out["tokens"] = tokens
    out["h"] = None
    out["threads"] = threads
    return out


def layer_tokens_shard(d: int, F: int, E: int, k: int, S: int, x: np.ndarray, w_router: np.ndarray,
                       bias: np.ndarray | None, codes: np.ndarray, scales: np.ndarray, e_begin: int, e_end: int,
                       with_shared: bool, tokens=None, w_shared_gate: np.ndarray | None = None) -> np.ndarray:
    """One expert shard's part of the layer output [n][d]: global routing, only experts in
    [e_begin, e_end) contribute, the shared expert only when with_shared."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T = x.shape[0]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    y = np.empty((tokens.shape[0], d), dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    sg = None if w_shared_gate is None else np.ascontiguousarray(w_shared_gate, dtype=np.float32)
    w_router = np.ascontiguousarray(w_router, dtype=np.float32)
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    _check(_load().oracle_layer_tokens_shard(d, F, E, k, S, _p(x), _p(w_router), _p(b), _p(codes), _p(scales),
                                             _p(tokens), tokens.shape[0], e_begin, e_end, 1 if with_shared else 0,
                                             _p(sg), _p(y)), "layer_tokens_shard")
    return y


# ---------------------------------------------------------------- affine group-64 experts

def affine_code(packed: np.ndarray, K: int, bits: int, r: int, c: int) -> int:
    packed = np.ascontiguousarray(packed)
    return _load().oracle_affine_code(_p(packed), K, bits, r, c)


def affine_element(packed: np.ndarray, scales: np.ndarray, biases: np.ndarray, K: int, bits: int, r: int,
                   c: int) -> float:
    packed, scales, biases = (np.ascontiguousarray(a) for a in (packed, scales, biases))
    return _load().oracle_affine_element(_p(packed), _p(scales), _p(biases), K, bits, r, c)


def affine_expert_bytes(d: int, f: int, bits: int) -> int:
    return _load().oracle_affine_expert_bytes(d, f, bits)


def expert_ffn_affine(expert: np.ndarray, d: int, f: int, bits: int, x: np.ndarray) -> np.ndarray:
    """One affine group-64 expert (codes, bf16 scales, bf16 biases in one byte range) on one fp64 vector."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty((d,), dtype=np.float64)
    expert = np.ascontiguousarray(expert)
    _check(_load().oracle_expert_ffn_affine(_p(expert), d, f, bits, _p(x), _p(out)),
           "expert_ffn_affine")
    return out


def layer_tokens_affine(d: int, F: int, E: int, k: int, S: int, bits: int, x: np.ndarray, w_router: np.ndarray,
                        bias: np.ndarray | None, experts: np.ndarray, tokens=None,
                        w_shared_gate: np.ndarray | None = None) -> dict:
    """fp64 layer output of the listed tokens with affine group-64 experts: y [n][d], ids, gates."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T = x.shape[0]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = tokens.shape[0]
    y = np.empty((n, d), dtype=np.float64)
    ids = np.empty((n, k), dtype=np.int32)
    gates = np.empty((n, k), dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    sg = None if w_shared_gate is None else np.ascontiguousarray(w_shared_gate, dtype=np.float32)
    w_router = np.ascontiguousarray(w_router, dtype=np.float32)
    experts = np.ascontiguousarray(experts)
    _check(_load().oracle_layer_tokens_affine(d, F, E, k, S, bits, _p(x), _p(w_router), _p(b),
                                              _p(experts), _p(tokens), n, _p(y), _p(ids),
                                              _p(gates), _p(sg)), "layer_tokens_affine")
    return {"y": y, "ids": ids, "gates": gates, "tokens": tokens}


def layer_tokens_affine_parallel(d: int, F: int, E: int, k: int, S: int, bits: int, x: np.ndarray,
                                 w_router: np.ndarray, bias: np.ndarray | None, experts: np.ndarray, tokens=None,
                                 threads: int | None = None, w_shared_gate: np.ndarray | None = None) -> dict:
    """layer_tokens_affine over a thread pool, one contiguous chunk of tokens per call (bit-identical)."""
    from concurrent.futures import ThreadPoolExecutor

    x = np.ascontiguousarray(x, dtype=np.uint16)
    T = x.shape[0]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = tokens.shape[0]
    threads = host_threads() if threads is None else max(1, int(threads))
    threads = min(threads, max(1, n))
    experts = np.ascontiguousarray(experts)
    _load()
    bounds = [(i * n) // threads for i in range(threads + 1)]

    def run(i):
        return layer_tokens_affine(d, F, E, k, S, bits, x, w_router, bias, experts,
                                   tokens=tokens[bounds[i]:bounds[i + 1]], w_shared_gate=w_shared_gate)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(run, range(threads)))
    out = {key: np.concatenate([pt[key] for pt in parts]) for key in ("y", "ids", "gates")}
    out["tokens"] = tokens
    out["threads"] = threads
    return out
