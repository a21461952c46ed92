"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Routing (ids, counts, offsets, perm) must match bit for bit; gates within
1e-6; outputs within 2e-2 * ||ref||_inf for bf16 and 1e-4 * ||ref||_inf for
fp32 outputs. Sizes span several tiles and ragged tails; the full-size
workloads are checked on every token (the oracle runs on all host cores).
"""
import numpy as np
import pytest

import oracle
import synth
from moe_testlib import (BF16_TOL, F32_TOL, bf16_bits_to_f64, build_lib, check_output, check_routing, make_layer, oracle_layer,
                         oracle_route, run_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU not available for a gpu-marked test")
    return build_lib()


def _parity(m, wl, L, out_f32=False, tokens=None, t_max=None, flags=0):
    layer = make_layer(m, wl, L, t_max=t_max, out_f32=out_f32, flags=flags)
    g = run_gpu(m, layer, L["x"], out_f32=out_f32)
    assert g["status"] == 0
    rr = oracle_route(wl, L)
    check_routing(g, rr, wl.E)
    ref = oracle_layer(wl, L, tokens=tokens)
    y = g["y"] if tokens is None else g["y"][np.asarray(tokens)]
    rel = check_output(y, ref["y"], F32_TOL if out_f32 else BF16_TOL)
    layer.close()
    return g, ref, rel


@pytest.mark.parametrize("out_f32", [False, True])
def test_tiny_layer(m, out_f32):
    wl = synth.WORKLOADS["tiny"]
    _parity(m, wl, synth.gen_layer(wl, 0), out_f32=out_f32)


SMALL_SHAPES = [
    # (T, d, ffn, E, k, shared, zipf)
    (1, 96, 160, 8, 1, 0, 0.0),
    (3, 224, 96, 16, 2, 0, 1.1),
    (5, 160, 224, 128, 4, 64, 0.0),
    (7, 64, 64, 256, 8, 96, 1.1),
    (9, 128, 32, 8, 8, 0, 0.0),
    (13, 288, 320, 32, 4, 0, 0.0),
    (16, 352, 96, 16, 4, 128, 1.1),
]


@pytest.mark.parametrize("shape", SMALL_SHAPES)
@pytest.mark.parametrize("out_f32", [False, True])
@pytest.mark.parametrize("path", ["fused-tc", "fused", "general", "general-tc"])
def test_small_shapes(m, shape, out_f32, path):
    """fused-tc: the single-launch tcgen05 kernel (MOE_FLAG_TC_GATEUP); fused: the single-launch
    mma.sync kernel (MOE_FLAG_NO_TC); general / general-tc: the multi-kernel path with either GEMM."""
    T, d, F, E, k, S, z = shape
    wl = synth.WORKLOADS["tiny"].with_(name="shape", number=9, T=T, d=d, ffn=F, E=E, k=k, shared_ffn=S, zipf_bias=z)
    flags = {"fused-tc": m.MOE_FLAG_TC_GATEUP, "fused": m.MOE_FLAG_NO_TC,
             "general": m.MOE_FLAG_GENERAL_PATH | m.MOE_FLAG_NO_TC,
             "general-tc": m.MOE_FLAG_GENERAL_PATH | m.MOE_FLAG_TC_GATEUP}[path]
    if path.startswith("fused"):
        lay = make_layer(m, wl, synth.gen_layer(wl, 17), flags=flags)
        assert m.moe_launches_per_forward(lay.ctx, T) == 1, "expected the single-launch path"
        lay.close()
    _parity(m, wl, synth.gen_layer(wl, 17), out_f32=out_f32, flags=flags)


@pytest.mark.parametrize("flags", [0, 2])
def test_wide_scale_exponent_range(m, flags):
    """E8M0 exponents over [96, 150] (2^-31 .. 2^23): the scale decode is exact across the range."""
    wl = synth.WORKLOADS["tiny"].with_(name="wide", T=5, d=128, ffn=96, E=8, k=2, scale_lo=96, scale_hi=150)
    _parity(m, wl, synth.gen_layer(wl, 21), out_f32=True, flags=flags)


def test_path_selection(m):
    """Contexts whose calls can exceed 16 (token, expert) pairs: one launch (the fused tcgen05 kernel) up to
    16 tokens, the multi-kernel tcgen05 path above; MOE_FLAG_NO_TC: the fused mma.sync kernel up to 16
    tokens, register-decode GEMMs above; a decode context (t_max * k <= 16): the fused mma.sync kernel."""
    wl = synth.WORKLOADS["decode"]  # k = 4
    lay = m.MoeLayer(m.LayerShape(wl.d, wl.ffn, wl.E, wl.k, t_max=1024))
    assert m.moe_launches_per_forward(lay.ctx, 1) == 1 and m.moe_forward_phases(lay.ctx, 1) == ["layer"]
    assert m.moe_launches_per_forward(lay.ctx, 4) == 1
    assert m.moe_launches_per_forward(lay.ctx, 16) == 1
    # router (one launch up to 32 tokens, fp32 pass + top-k above), bucket, x planes, x panels, 2 GEMMs, combine
    assert m.moe_launches_per_forward(lay.ctx, 17) == 7
    assert m.moe_launches_per_forward(lay.ctx, 32) == 7
    assert m.moe_launches_per_forward(lay.ctx, 33) == 8
    assert m.moe_forward_phases(lay.ctx, 33) == ["route", "panels", "gateup", "down", "combine"]
    lay.close()
    lay = m.MoeLayer(m.LayerShape(wl.d, wl.ffn, wl.E, wl.k, t_max=1024, flags=m.MOE_FLAG_NO_TC))
    assert m.moe_launches_per_forward(lay.ctx, 16) == 1
    assert m.moe_launches_per_forward(lay.ctx, 17) == 5  # up to 32 tokens the router launch prepares the f16 x
    assert m.moe_launches_per_forward(lay.ctx, 33) == 7
    lay.close()
    lay = m.MoeLayer(m.LayerShape(wl.d, wl.ffn, wl.E, wl.k, t_max=4))
    assert m.moe_launches_per_forward(lay.ctx, 4) == 1 and lay.weight_bytes() == wl.E * wl.expert_bytes()
    lay.close()


def test_forced_timeout_is_reported_and_context_survives(m):
    """A device-side wait that cannot be satisfied gives up within its bound,
    the status word says MOE_ERR_TIMEOUT, and the GPU stays usable."""
    wl = synth.WORKLOADS["tiny"]
    L = synth.gen_layer(wl, 0)
    layer = make_layer(m, wl, L, flags=m.MOE_FLAG_TEST_FORCE_TIMEOUT)
    run_gpu(m, layer, L["x"])  # run_gpu synchronises; the kernel returned
    assert layer.status(clear=True) == m.MOE_ERR_TIMEOUT
    assert layer.status() == 0
    layer.close()
    _parity(m, wl, L)  # a normal context on the same GPU still matches the oracle


@pytest.mark.parametrize("flags", [0, 2])
def test_every_token_count_up_to_16(m, flags):
    """Row counts 1..16 (ragged n8 tiles) through one context sized t_max = 16."""
    wl = synth.WORKLOADS["tiny"].with_(T=16, E=16, k=4, shared_ffn=64)
    L = synth.gen_layer(wl, 3)
    layer = make_layer(m, wl, L, t_max=16, out_f32=True, flags=flags)
    full_ref = oracle_layer(wl, L)
    for T in range(1, 17):
        g = run_gpu(m, layer, L["x"][:T], out_f32=True)
        check_output(g["y"], full_ref["y"][:T], F32_TOL)
        assert np.array_equal(g["ids"], full_ref["ids"][:T])
    layer.close()


@pytest.mark.parametrize("cls", ["single", "batch", "mma.sync"])
def test_batch_invariance(m, cls):
    """Within a path, a token's output bits do not depend on the other tokens of its call: the fused
    tcgen05 kernel with a batch of 4 vs single tokens ("single") and a batch of 16 vs sub-batches of 5
    and 11 ("batch"); the fused mma.sync kernel (MOE_FLAG_NO_TC) with a batch of 4 vs single tokens."""
    wl = synth.WORKLOADS["tiny"].with_(T=16, E=32, k=4)
    L = synth.gen_layer(wl, 5)
    layer = make_layer(m, wl, L, t_max=16, out_f32=True, flags=m.MOE_FLAG_NO_TC if cls == "mma.sync" else 0)
    if cls != "batch":
        full = run_gpu(m, layer, L["x"][:4].copy(), out_f32=True)
        for t in (0, 3):
            one = run_gpu(m, layer, L["x"][t:t + 1].copy(), out_f32=True)
            assert np.array_equal(one["y"][0], full["y"][t])
    else:
        full = run_gpu(m, layer, L["x"], out_f32=True)
        a = run_gpu(m, layer, L["x"][:5].copy(), out_f32=True)
        b = run_gpu(m, layer, L["x"][5:].copy(), out_f32=True)
        assert np.array_equal(a["y"], full["y"][:5])
        assert np.array_equal(b["y"], full["y"][5:])
    layer.close()


def test_down_scale_plus_one_doubles_exactly(m):
    wl = synth.WORKLOADS["tiny"].with_(T=6)
    L = synth.gen_layer(wl, 0)
    layer = make_layer(m, wl, L, out_f32=True)
    g1 = run_gpu(m, layer, L["x"], out_f32=True)
    sc = L["scales"].copy()
    per, gu = wl.scale_bytes(), 2 * wl.ffn * wl.d // 32
    for e in range(wl.E):
        sc[e * per + gu:(e + 1) * per] += 1
    layer2 = make_layer(m, wl, dict(L, scales=sc), out_f32=True)
    g2 = run_gpu(m, layer2, L["x"], out_f32=True)
    assert np.array_equal(g2["y"], 2.0 * g1["y"])
    layer.close()
    layer2.close()


@pytest.mark.parametrize("flags", [0, 2])
def test_exact_ties_lower_index(m, flags):
    wl = synth.WORKLOADS["tiny"].with_(T=3, E=8, k=3)
    L = synth.gen_layer(wl, 0)
    w = np.zeros((wl.E, wl.d), dtype=np.float32)
    w[[2, 5, 6]] = 0.25  # three identical router rows -> exact ties
    w[1] = 0.125
    L = dict(L, w_router=w)
    g, ref, _ = _parity(m, wl, L, flags=flags)
    for t in range(wl.T):
        s = np.sign(synth.bf16_bits_to_f32(L["x"][t]).sum())
        expect = [2, 5, 6] if s > 0 else [0, 3, 4]
        assert list(g["ids"][t]) == expect


@pytest.mark.parametrize("T,flags", [(16, 0), (16, 2), (40, 0)])
def test_near_ties_need_double_float(m, T, flags):
    """Router rows 3 and 7 differ by one ulp in one element and carry a large bias:
    both are every token's top 2, their order is set by a logit difference far
    below fp32 resolution. The fused path and the multi-kernel path up to 32
    tokens sum every logit in double-float; above 32 tokens the multi-kernel
    path's fp32 bound cannot order them and its double-float recompute must."""
    wl = synth.WORKLOADS["tiny"].with_(T=T, E=16, k=2)
    L = synth.gen_layer(wl, 6)
    w = L["w_router"].copy()
    w[7] = w[3]
    w[7, 5] = np.nextafter(w[3, 5], np.float32(np.inf))
    b = np.zeros(wl.E, dtype=np.float32)
    b[3] = b[7] = 50.0
    g, ref, _ = _parity(m, wl, dict(L, w_router=w, bias=b), flags=flags)
    assert set(np.unique(g["ids"])) == {3, 7}
    assert len({tuple(r) for r in g["ids"]}) == 2  # both orders occur (the sign of x[t, 5] decides)


@pytest.mark.parametrize("T", [2, 8])
def test_near_ties_on_the_fused_kernel(m, T):
    """The same one-ulp construction on calls the fused single-kernel path takes
    (T * k <= 16 pairs, a context without the tcgen05 copy): its router sums every
    logit in double-float inside the kernel, and the order of experts 3 and 7 is
    decided by a logit difference about 1e-7 of one fp32 ulp of the logits. Token
    0 has x[0, 5] = +1 and token 1 has x[1, 5] = -1, so both orders occur."""
    wl = synth.WORKLOADS["tiny"].with_(T=T, E=16, k=2)
    L = synth.gen_layer(wl, 6)
    w = L["w_router"].copy()
    w[7] = w[3]
    w[7, 5] = np.nextafter(w[3, 5], np.float32(np.inf))
    b = np.zeros(wl.E, dtype=np.float32)
    b[3] = b[7] = 50.0
    x = L["x"].copy()
    x[0, 5] = 0x3F80  # bf16 +1.0: expert 7's logit is the larger one
    x[1, 5] = 0xBF80  # bf16 -1.0: expert 3's
    L = dict(L, w_router=w, bias=b, x=x)
    layer = make_layer(m, wl, L, t_max=T)
    assert m.moe_launches_per_forward(layer.ctx, T) == 1, "this case must run on the fused kernel"
    layer.close()
    g, ref, _ = _parity(m, wl, L, t_max=T)
    assert list(g["ids"][0]) == [7, 3] and list(g["ids"][1]) == [3, 7]
    # the pair is far below fp32 resolution: one fp32 ulp of the logits is ~4e-6
    lr = oracle.route(x, w, b, wl.k)["logits"]
    assert 0 < abs(lr[0, 7] - lr[0, 3]) < 1e-6


def test_skewed_all_tokens_one_expert(m):
    wl = synth.WORKLOADS["tiny"].with_(T=16, E=16, k=2)
    L = synth.gen_layer(wl, 4)
    b = np.zeros(wl.E, dtype=np.float32)
    b[11] = 100.0
    b[3] = 90.0
    _parity(m, wl, dict(L, bias=b))


def test_default_context_stores_one_copy(m):
    """A context keeps its experts once: in the tcgen05 layout when its calls can exceed 16 (token, expert)
    pairs (tile padding only: the 13,219,200-byte expert of the decode shapes takes at most 7 % more), in the
    packed layout, exactly the canonical size, otherwise or with MOE_FLAG_NO_TC."""
    wl = synth.WORKLOADS["decode"]  # k = 4
    for t_max in (5, 16, 1024):
        lay = m.MoeLayer(m.LayerShape(wl.d, wl.ffn, wl.E, wl.k, t_max=t_max))
        assert wl.E * wl.expert_bytes() < lay.weight_bytes() <= 1.07 * wl.E * wl.expert_bytes()
        lay.close()
    for t_max, flags in ((1, 0), (4, 0), (16, m.MOE_FLAG_NO_TC)):
        lay = m.MoeLayer(m.LayerShape(wl.d, wl.ffn, wl.E, wl.k, t_max=t_max, flags=flags))
        assert lay.weight_bytes() == wl.E * wl.expert_bytes()
        lay.close()


def test_k_equals_E(m):
    wl = synth.WORKLOADS["tiny"].with_(T=5, E=4, k=4, shared_ffn=32)
    _parity(m, wl, synth.gen_layer(wl, 8), out_f32=True)


def test_empty_batch_and_errors(m):
    wl = synth.WORKLOADS["tiny"]
    L = synth.gen_layer(wl, 0)
    layer = make_layer(m, wl, L, t_max=4)
    import torch
    x = torch.zeros((8, wl.d), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((8, wl.d), dtype=torch.bfloat16, device="cuda")
    layer.forward(x, 0, out)  # T = 0 is a no-op
    torch.cuda.synchronize()
    assert float(out.abs().sum()) == 0.0
    with pytest.raises(m.MoeError) as ei:
        layer.forward(x, 5, out)
    assert ei.value.code == m.MOE_ERR_T_TOO_LARGE
    bad = L["scales"].copy()
    bad[123] = 255
    layer2 = m.MoeLayer(layer.shape)
    with pytest.raises(m.MoeError) as ei:
        layer2.load(L["w_router"], None, L["codes"], bad)
    assert ei.value.code == m.MOE_ERR_NAN_SCALE
    with pytest.raises(m.MoeError) as ei:
        layer2.forward(x, 1, out)
    assert ei.value.code == m.MOE_ERR_NOT_LOADED
    layer.close()
    layer2.close()


def test_forward_host_matches_device(m):
    wl = synth.WORKLOADS["tiny"].with_(T=5)
    L = synth.gen_layer(wl, 2)
    layer = make_layer(m, wl, L, t_max=8)
    g = run_gpu(m, layer, L["x"])
    out = np.zeros((wl.T, wl.d), dtype=np.uint16)
    layer.forward_host(L["x"], wl.T, out)
    y = (out.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(y, g["y"])
    layer.close()


@pytest.mark.parametrize("path,out_f32,T,d", [("fused", False, 7, 288), ("fused-tc", True, 7, 288),
                                              ("fused-tc", False, 7, 288), ("fused-tc", False, 16, 1024),
                                              ("general", True, 40, 288)])
def test_forward_host_mapped_buffers(m, path, out_f32, T, d):
    """Page-locked host buffers: the kernels write y straight into out_host, and a single-launch call on
    at most 16 KB of x also reads x from x_host (T=7, d=288); larger x (T=16, d=1024) and the multi-kernel
    path (T=40) copy x in first. The result equals the device-buffer call's bit for bit on two calls in a
    row (fresh inputs for the second), and x and out that share bytes still give the device result."""
    torch = pytest.importorskip("torch")
    wl = synth.WORKLOADS["tiny"].with_(name="mapped", T=T, d=d, ffn=320, E=32, k=4, shared_ffn=64)
    flags = {"fused": m.MOE_FLAG_NO_TC, "fused-tc": m.MOE_FLAG_TC_GATEUP, "general": m.MOE_FLAG_TC_GATEUP}[path]
    L = synth.gen_layer(wl, 31)
    layer = make_layer(m, wl, L, t_max=max(T, 16), out_f32=out_f32, flags=flags)
    assert (m.moe_launches_per_forward(layer.ctx, T) == 1) == path.startswith("fused")
    odt = torch.float32 if out_f32 else torch.int16
    for call in range(2):
        xb = L["x"] if call == 0 else synth.gen_layer(wl, 32)["x"]
        g = run_gpu(m, layer, xb, out_f32=out_f32)
        x_h = torch.from_numpy(xb.view(np.int16).copy()).pin_memory()
        out_h = torch.full((T, wl.d), -1, dtype=odt).pin_memory()
        layer.forward_host(x_h, T, out_h)
        yo = out_h.numpy()
        y = yo.astype(np.float64) if out_f32 else bf16_bits_to_f64(yo.view(np.uint16))
        assert np.array_equal(y, g["y"]), f"call {call}"
        assert layer.status() == 0
    # in place: out over x (bf16 out only: the same bytes per row)
    if not out_f32:
        buf = torch.from_numpy(L["x"].view(np.int16).copy()).pin_memory()
        layer.forward_host(buf, T, buf)
        g = run_gpu(m, layer, L["x"])
        assert np.array_equal(bf16_bits_to_f64(buf.numpy().view(np.uint16)), g["y"])
    layer.close()


# ---------------------------------------------------------------- full-size workloads (every token)

_FULL_REF = {}


def _full_ref(name: str, layer_idx: int):
    """Inputs and the oracle's output for every token of one full-size layer (fp64 on all host
    cores: the thread-parallel driver evaluates each token with the single-threaded code)."""
    key = (name, layer_idx)
    if key not in _FULL_REF:
        wl = synth.WORKLOADS[name]
        L = synth.gen_layer(wl, layer_idx)
        ref = oracle.layer_tokens_parallel(wl.d, wl.ffn, wl.E, wl.k, wl.shared_ffn, L["x"], L["w_router"],
                                           L["bias"], L["codes"], L["scales"])
        _FULL_REF.clear()  # one full-size layer's inputs at a time
        _FULL_REF[key] = (wl, L, ref)
    return _FULL_REF[key]


@pytest.mark.parametrize("out_f32", [False, True])
@pytest.mark.parametrize("name,layer_idx", [
    ("decode", 0),
    ("decode", 35),
    ("verify", 0),
    ("small", 0),
    ("prefill", 0),
])
def test_full_size_workloads(m, name, layer_idx, out_f32):
    """Every token of a full-size layer, in the launch configuration the benchmark times (one
    context with t_max = T; verify and small take the tcgen05 multi-kernel path, decode the fused
    kernel): routing bit-exact over all tokens, y within the bf16 / fp32 tolerance."""
    wl, L, ref = _full_ref(name, layer_idx)
    layer = make_layer(m, wl, L, out_f32=out_f32)
    g = run_gpu(m, layer, L["x"], out_f32=out_f32)
    assert g["status"] == 0
    check_routing(g, oracle_route(wl, L), wl.E)
    assert np.array_equal(g["ids"], ref["ids"])
    check_output(g["y"], ref["y"], F32_TOL if out_f32 else BF16_TOL)
    layer.close()


def test_ridge_crossing_prefill_chunk(m):
    """The 16,384-token chunk (512 tokens per expert on average) on the tcgen05 multi-kernel path: routing,
    counts, offsets, perm and inv bit-exact over all tokens; y on 64 tokens spread over the chunk (the
    oracle's cost), at the bf16 and fp32 tolerances."""
    wl = synth.WORKLOADS["prefill16k"]
    L = synth.gen_layer(wl, 0)
    tokens = list(range(0, wl.T, wl.T // 64))
    ref = oracle.layer_tokens_parallel(wl.d, wl.ffn, wl.E, wl.k, 0, L["x"], L["w_router"], L["bias"], L["codes"],
                                       L["scales"], tokens=tokens)
    rr = oracle_route(wl, L)
    for out_f32 in (False, True):
        layer = make_layer(m, wl, L, out_f32=out_f32)
        assert m.moe_launches_per_forward(layer.ctx, wl.T) == 8
        g = run_gpu(m, layer, L["x"], out_f32=out_f32)
        assert g["status"] == 0
        check_routing(g, rr, wl.E)
        assert np.min(g["counts"]) >= 300  # every expert well past the ridge
        check_output(g["y"][tokens], ref["y"], F32_TOL if out_f32 else BF16_TOL)
        layer.close()


def test_register_decode_gemms_prefill_sampled(m):
    """The multi-kernel path without the tcgen05 GEMMs (MOE_FLAG_NO_TC) on the full prefill chunk."""
    wl = synth.WORKLOADS["prefill"]
    _parity(m, wl, synth.gen_layer(wl, 2), tokens=[3, 700], flags=m.MOE_FLAG_NO_TC)


MEDIUM_SHAPES = [
    # (T, d, ffn, E, k, shared, zipf): token blocks of 48 with ragged tails, experts over several blocks,
    # K step counts odd and even, M tile counts odd and even
    (17, 256, 320, 16, 2, 0, 0.0),
    (100, 384, 192, 8, 4, 96, 1.1),
    (300, 160, 416, 32, 3, 0, 1.1),
]


@pytest.mark.parametrize("shape", MEDIUM_SHAPES)
@pytest.mark.parametrize("flags", [0, 8])
def test_medium_shapes(m, shape, flags):
    """T > 16: the multi-kernel path with (default) and without (MOE_FLAG_NO_TC) the tcgen05 GEMMs."""
    T, d, F, E, k, S, z = shape
    wl = synth.WORKLOADS["tiny"].with_(name="medium", number=11, T=T, d=d, ffn=F, E=E, k=k, shared_ffn=S,
                                       zipf_bias=z)
    L = synth.gen_layer(wl, 23)
    tokens = None if T <= 100 else list(range(0, T, 7))
    _parity(m, wl, L, out_f32=True, tokens=tokens, flags=flags)


@pytest.mark.parametrize("name", ["decode", "verify", "small"])
def test_fused_and_general_paths_agree_on_full_size(m, name):
    """Both paths, same inputs: routing identical, outputs within fp32 tolerance of each other."""
    wl = synth.WORKLOADS[name]
    L = synth.gen_layer(wl, 1)
    a = make_layer(m, wl, L, out_f32=True, flags=m.MOE_FLAG_NO_TC)  # fused kernel for every T <= 16
    b = make_layer(m, wl, L, out_f32=True, flags=m.MOE_FLAG_GENERAL_PATH | m.MOE_FLAG_NO_TC)
    ga = run_gpu(m, a, L["x"], out_f32=True)
    gb = run_gpu(m, b, L["x"], out_f32=True)
    assert np.array_equal(ga["ids"], gb["ids"]) and np.array_equal(ga["perm"], gb["perm"])
    check_output(ga["y"], gb["y"], 1e-5)
    a.close()
    b.close()
