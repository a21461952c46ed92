"""The sigmoid-gated shared expert on the GPU against the oracle: y_t = sum_j g_j part_j +
sigmoid(w_sg . x_t) shared(x_t), on every path (both single-launch kernels, the multi-kernel path with
either GEMM), at shapes with ragged tails and at the full size of the small workload (T = 8, d = 2048,
E = 256, k = 8, shared ffn 2048). A gate row of zeros weighs the shared expert 1/2; removing the row
restores the ungated layer."""
import numpy as np
import pytest

import oracle
import synth
from moe_testlib import BF16_TOL, F32_TOL, build_lib, check_output, check_routing, make_layer, oracle_layer, \
    oracle_route, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU not available for a gpu-marked test")
    return build_lib()


def _flags(m, path):
    return {"fused-tc": m.MOE_FLAG_TC_GATEUP, "fused": m.MOE_FLAG_NO_TC,
            "general": m.MOE_FLAG_GENERAL_PATH | m.MOE_FLAG_NO_TC,
            "general-tc": m.MOE_FLAG_GENERAL_PATH | m.MOE_FLAG_TC_GATEUP}[path]


@pytest.mark.parametrize("path", ["fused-tc", "fused", "general", "general-tc"])
@pytest.mark.parametrize("shape", [(5, 160, 224, 128, 4, 64), (16, 352, 96, 16, 4, 128), (3, 256, 64, 8, 2, 96)])
def test_gated_shared_expert_matches_oracle(m, path, shape):
    T, d, F, E, k, S = shape
    wl = synth.WORKLOADS["tiny"].with_(name="gated", number=12, T=T, d=d, ffn=F, E=E, k=k, shared_ffn=S)
    L = synth.gen_layer(wl, 4)
    w_sg = synth.gen_shared_gate(L["seed"], d)
    ref = oracle_layer(wl, L, w_shared_gate=w_sg)
    for out_f32 in (False, True):
        layer = make_layer(m, wl, L, out_f32=out_f32, flags=_flags(m, path), w_shared_gate=w_sg)
        g = run_gpu(m, layer, L["x"], out_f32=out_f32)
        assert g["status"] == 0
        check_routing(g, oracle_route(wl, L), wl.E)
        check_output(g["y"], ref["y"], F32_TOL if out_f32 else BF16_TOL)
        layer.close()


def test_gated_shared_expert_full_size_small_workload(m):
    wl = synth.WORKLOADS["small"]
    L = synth.gen_layer(wl, 0)
    w_sg = synth.gen_shared_gate(L["seed"], wl.d)
    ref = oracle.layer_tokens_parallel(wl.d, wl.ffn, wl.E, wl.k, wl.shared_ffn, L["x"], L["w_router"], L["bias"],
                                       L["codes"], L["scales"], w_shared_gate=w_sg)
    for out_f32 in (False, True):
        layer = make_layer(m, wl, L, out_f32=out_f32, w_shared_gate=w_sg)
        g = run_gpu(m, layer, L["x"], out_f32=out_f32)
        assert g["status"] == 0
        assert np.array_equal(g["ids"], ref["ids"])
        check_output(g["y"], ref["y"], F32_TOL if out_f32 else BF16_TOL)
        layer.close()


@pytest.mark.parametrize("path", ["fused-tc", "fused", "general"])
def test_zero_gate_row_halves_the_shared_expert_and_removal_restores_it(m, path):
    """sigmoid(0) = 1/2: with a zero gate row the layer matches the oracle's y = routed + shared / 2 and
    differs from the ungated layer; removing the row (NULL) restores the ungated output bit for bit."""
    wl = synth.WORKLOADS["tiny"].with_(name="gated", number=12, T=4, d=256, ffn=128, E=8, k=2, shared_ffn=64)
    L = synth.gen_layer(wl, 5)
    flags = _flags(m, path)
    plain = make_layer(m, wl, L, out_f32=True, flags=flags)
    y1 = run_gpu(m, plain, L["x"], out_f32=True)["y"]
    half = make_layer(m, wl, L, out_f32=True, flags=flags, w_shared_gate=np.zeros(wl.d, dtype=np.float32))
    yh = run_gpu(m, half, L["x"], out_f32=True)["y"]
    ref1 = oracle_layer(wl, L)
    refh = oracle_layer(wl, L, w_shared_gate=np.zeros(wl.d, dtype=np.float32))
    check_output(yh, refh["y"], F32_TOL)
    assert not np.allclose(yh, y1)
    m.moe_load_shared_gate(half.ctx, None)  # remove the gate: the ungated layer again
    y2 = run_gpu(m, half, L["x"], out_f32=True)["y"]
    assert np.array_equal(y2, y1)
    check_output(y1, ref1["y"], F32_TOL)
    plain.close()
    half.close()


def test_gate_on_a_context_without_shared_expert_is_rejected(m):
    wl = synth.WORKLOADS["tiny"]
    L = synth.gen_layer(wl, 0)
    layer = make_layer(m, wl, L)
    with pytest.raises(m.MoeError) as ei:
        m.moe_load_shared_gate(layer.ctx, np.zeros(wl.d, dtype=np.float32))
    assert ei.value.code == m.MOE_ERR_INVALID_ARG
    layer.close()
