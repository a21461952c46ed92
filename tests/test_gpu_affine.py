"""Affine group-64 experts on the GPU against the oracle: w = scale * q + bias with a bf16 scale
and bias per 64 weights ("Running Qwen3.8-Flash-Next on a 32 GB Mac with Transformers": routed
experts in 3-bit affine form, group 64, 2.15 MB each; a 16-bit scale and bias per 64 weights).

Routing must match the oracle bit for bit; the layer output within the fp32 / bf16 tolerances of
the MXFP4 tests, at code widths 2, 3, 4 and 8, at shapes whose slots cross the 16-row work blocks
and have ragged tails, with and without the gated shared expert, at the full size of the affine
decode workload (d = 2560, ffn = 640, E = 512, k = 10, shared ffn 640) in the launch configuration
the benchmark times, for expert-parallel shards, and token by token against a batch (batch
invariance). Bad inputs are refused on the host."""
import numpy as np
import pytest

import oracle
import synth
from moe_testlib import BF16_TOL, F32_TOL, build_lib, check_output, check_routing, oracle_route, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU not available for a gpu-marked test")
    return build_lib()


def _wl(T, d, F, E, k, S, bits):
    return synth.WORKLOADS["tiny"].with_(name="affine", number=13, T=T, d=d, ffn=F, E=E, k=k, shared_ffn=S,
                                         affine_bits=bits)


def _layer(m, wl, L, out_f32=False, t_max=None, flags=0, w_shared_gate=None, shard=(0, 0)):
    shape = m.LayerShape(d=wl.d, ffn=wl.ffn, n_experts=wl.E, top_k=wl.k, shared_ffn=wl.shared_ffn,
                         t_max=wl.T if t_max is None else t_max,
                         out_dtype=m.MOE_OUT_F32 if out_f32 else m.MOE_OUT_BF16, flags=flags,
                         expert_begin=shard[0], expert_end=shard[1], weight_format=m.MOE_FORMAT_AFFINE64,
                         weight_bits=wl.affine_bits)
    layer = m.MoeLayer(shape)
    experts = L["experts"]
    if shard != (0, 0):  # the shard's routed experts, then the shared expert on the first shard
        eb = wl.affine_bytes()
        experts = experts[shard[0] * eb:shard[1] * eb]
        if shard[0] == 0 and wl.shared_ffn:
            experts = np.concatenate([experts, L["experts"][wl.E * eb:]])
    layer.load_affine(L["w_router"], L["bias"], np.ascontiguousarray(experts), w_shared_gate=w_shared_gate)
    return layer


def _oracle(wl, L, tokens=None, w_shared_gate=None, parallel=False):
    f = oracle.layer_tokens_affine_parallel if parallel else oracle.layer_tokens_affine
    return f(wl.d, wl.ffn, wl.E, wl.k, wl.shared_ffn, wl.affine_bits, L["x"], L["w_router"], L["bias"],
             L["experts"], tokens=tokens, w_shared_gate=w_shared_gate)


SHAPES = [(5, 256, 128, 16, 4, 128), (37, 192, 192, 8, 2, 64), (1, 128, 64, 4, 1, 0), (70, 320, 256, 6, 3, 128)]


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("shape", SHAPES)
def test_affine_layer_matches_oracle(m, bits, shape):
    wl = _wl(*shape, bits)
    L = synth.gen_layer(wl, bits)
    ref = _oracle(wl, L)
    for out_f32 in (True, False):
        layer = _layer(m, wl, L, out_f32=out_f32)
        assert m.moe_forward_phases(layer.ctx, wl.T) == ["route", "gateup", "down", "combine"]
        g = run_gpu(m, layer, L["x"], out_f32=out_f32)
        assert g["status"] == 0
        check_routing(g, oracle_route(wl, L), wl.E)
        check_output(g["y"], ref["y"], F32_TOL if out_f32 else BF16_TOL)
        layer.close()


def test_affine_gated_shared_expert(m):
    wl = _wl(9, 256, 192, 12, 3, 128, 3)
    L = synth.gen_layer(wl, 1)
    w_sg = synth.gen_shared_gate(L["seed"], wl.d)
    ref = _oracle(wl, L, w_shared_gate=w_sg)
    layer = _layer(m, wl, L, out_f32=True, w_shared_gate=w_sg)
    g = run_gpu(m, layer, L["x"], out_f32=True)
    assert g["status"] == 0
    check_output(g["y"], ref["y"], F32_TOL)
    plain = _oracle(wl, L)
    assert not np.allclose(ref["y"], plain["y"])


@pytest.mark.parametrize("T", [1, 16, 64])
def test_affine_full_size_every_token(m, T):
    """The affine decode workload's layer (E = 512, d = 2560, ffn = 640, k = 10, shared 640, 3-bit),
    every token against the oracle; T = 1 is the configuration the benchmark times."""
    wl = synth.WORKLOADS["affine3"].with_(T=T)
    L = synth.gen_layer(wl, 0)
    ref = _oracle(wl, L, parallel=True)
    for out_f32 in (True, False):
        layer = _layer(m, wl, L, out_f32=out_f32)
        g = run_gpu(m, layer, L["x"], out_f32=out_f32)
        assert g["status"] == 0
        assert np.array_equal(g["ids"], ref["ids"])
        check_output(g["y"], ref["y"], F32_TOL if out_f32 else BF16_TOL)
        layer.close()


def test_affine_tokens_alone_equal_the_batch(m):
    """Each token's output bits do not depend on the other tokens of the call."""
    wl = _wl(24, 256, 128, 16, 4, 128, 4)
    L = synth.gen_layer(wl, 2)
    layer = _layer(m, wl, L, out_f32=True)
    yb = run_gpu(m, layer, L["x"], out_f32=True)["y"]
    for t in (0, 7, 23):
        y1 = run_gpu(m, layer, np.ascontiguousarray(L["x"][t:t + 1]), out_f32=True)["y"]
        assert np.array_equal(y1[0], yb[t])


def test_affine_expert_shards_add_up(m):
    wl = _wl(11, 192, 128, 10, 3, 64, 3)
    L = synth.gen_layer(wl, 3)
    ref = _oracle(wl, L)
    total = np.zeros((wl.T, wl.d))
    for shard in ((0, 4), (4, 10)):
        layer = _layer(m, wl, L, out_f32=True, shard=shard)
        g = run_gpu(m, layer, L["x"], out_f32=True)
        assert g["status"] == 0
        total += g["y"]
        layer.close()
    check_output(total, ref["y"], F32_TOL)


def test_affine_configs_and_loads_are_checked(m):
    ok = dict(d=128, ffn=64, n_experts=4, top_k=2, t_max=4, weight_format=m.MOE_FORMAT_AFFINE64, weight_bits=3)
    for bad in (dict(weight_bits=5), dict(weight_bits=0), dict(d=96), dict(ffn=96), dict(shared_ffn=32),
                dict(flags=m.MOE_FLAG_TC_GATEUP), dict(weight_format=2)):
        with pytest.raises(m.MoeError) as ei:
            m.MoeLayer(m.LayerShape(**{**ok, **bad}))
        assert ei.value.code == m.MOE_ERR_INVALID_ARG
    wl = _wl(4, 128, 64, 4, 2, 0, 3)
    L = synth.gen_layer(wl, 0)
    layer = m.MoeLayer(m.LayerShape(**ok))
    with pytest.raises(m.MoeError) as ei:  # MXFP4 load on an affine context
        m.moe_load_experts(layer.ctx, np.zeros(16, np.uint8), np.zeros(16, np.uint8))
    assert ei.value.code == m.MOE_ERR_INVALID_ARG
    bad = L["experts"].copy()
    n_codes = 3 * wl.ffn * wl.d * 3 // 8
    bad[n_codes:n_codes + 2] = np.frombuffer(np.uint16(0x7FC0).tobytes(), np.uint8)  # a NaN scale
    m.moe_load_router(layer.ctx, L["w_router"], None)
    with pytest.raises(m.MoeError) as ei:
        m.moe_load_experts_affine(layer.ctx, bad)
    assert ei.value.code == m.MOE_ERR_NAN_SCALE
    torch = pytest.importorskip("torch")
    x = torch.zeros((4, wl.d), dtype=torch.int16, device="cuda")
    out = torch.empty((4, wl.d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MoeError) as ei:  # a failed load leaves the context unloaded
        layer.forward(x, 4, out)
    assert ei.value.code == m.MOE_ERR_NOT_LOADED
    m.moe_load_experts_affine(layer.ctx, L["experts"])
    layer.forward(x, 4, out)
    layer.close()
    mx = m.MoeLayer(m.LayerShape(d=128, ffn=64, n_experts=4, top_k=2, t_max=4))
    with pytest.raises(m.MoeError) as ei:  # affine load on an MXFP4 context
        m.moe_load_experts_affine(mx.ctx, L["experts"])
    assert ei.value.code == m.MOE_ERR_INVALID_ARG
    mx.close()


def test_affine_launch_count(m):
    """The affine chain: router (which also prepares the f16 x up to 32 tokens), bucketing with the top k,
    two GEMMs, combine; above 32 tokens a separate x preparation and the two-pass router."""
    lay = m.MoeLayer(m.LayerShape(d=128, ffn=64, n_experts=4, top_k=2, t_max=64,
                                  weight_format=m.MOE_FORMAT_AFFINE64, weight_bits=3))
    assert m.moe_launches_per_forward(lay.ctx, 1) == 5
    assert m.moe_launches_per_forward(lay.ctx, 32) == 5
    assert m.moe_launches_per_forward(lay.ctx, 33) == 7
    lay.close()
