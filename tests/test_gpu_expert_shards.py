"""Expert-parallel shards on one GPU against the oracle: a context with [expert_begin, expert_end) holds
only those routed experts (and the shared expert when expert_begin == 0), routes over all experts, and
outputs its part of y; the oracle's layer_tokens_shard defines that part. The parts of a partition of the
experts add up to the layer; routing exports stay global; every path (both single-launch kernels and the
multi-kernel path with either GEMM) and the gated shared expert are covered."""
import numpy as np
import pytest

import oracle
import synth
from moe_testlib import F32_TOL, build_lib, check_output, check_routing, oracle_route, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU not available for a gpu-marked test")
    return build_lib()


FLAGS = {"fused-tc": "MOE_FLAG_TC_GATEUP", "fused": "MOE_FLAG_NO_TC",
         "general": ("MOE_FLAG_GENERAL_PATH", "MOE_FLAG_NO_TC"), "general-tc": ("MOE_FLAG_GENERAL_PATH", "MOE_FLAG_TC_GATEUP")}


def _flags(m, path):
    f = FLAGS[path]
    return getattr(m, f) if isinstance(f, str) else getattr(m, f[0]) | getattr(m, f[1])


def _shard_layer(m, wl, L, b, e, flags, w_sg=None):
    """A context holding experts [b, e) (and the shared expert if b == 0), loaded with their bytes only."""
    cb, sb = wl.code_bytes(), wl.scale_bytes()
    codes = L["codes"][b * cb:e * cb]
    scales = L["scales"][b * sb:e * sb]
    if b == 0 and wl.shared_ffn:
        codes = np.concatenate([codes, L["codes"][wl.E * cb:]])
        scales = np.concatenate([scales, L["scales"][wl.E * sb:]])
    shape = m.LayerShape(d=wl.d, ffn=wl.ffn, n_experts=wl.E, top_k=wl.k, shared_ffn=wl.shared_ffn, t_max=wl.T,
                         out_dtype=m.MOE_OUT_F32, flags=flags, expert_begin=b, expert_end=e)
    layer = m.MoeLayer(shape)
    layer.load(L["w_router"], L["bias"], np.ascontiguousarray(codes), np.ascontiguousarray(scales),
               w_shared_gate=w_sg if b == 0 else None)
    return layer, codes.nbytes + scales.nbytes


# (T, d, ffn, E, k, shared ffn), shard boundaries, gated shared expert (only where there is a shared expert)
SHARD_CASES = [(shape, cuts, gated)
               for shape, cuts in [((6, 256, 192, 16, 4, 64), [0, 5, 11, 16]),
                                   ((16, 160, 96, 8, 2, 0), [0, 3, 8]),
                                   ((20, 224, 128, 32, 4, 96), [0, 16, 32])]
               for gated in (False, True) if shape[5] > 0 or not gated]


@pytest.mark.parametrize("path", ["fused-tc", "fused", "general", "general-tc"])
@pytest.mark.parametrize("shape,cuts,gated", SHARD_CASES)
def test_shards_match_the_oracle_and_add_up(m, path, shape, cuts, gated):
    T, d, F, E, k, S = shape
    wl = synth.WORKLOADS["tiny"].with_(name="shard", number=13, T=T, d=d, ffn=F, E=E, k=k, shared_ffn=S)
    L = synth.gen_layer(wl, 2)
    w_sg = synth.gen_shared_gate(L["seed"], d) if gated else None
    full = oracle.layer_tokens(d, F, E, k, S, L["x"], L["w_router"], L["bias"], L["codes"], L["scales"],
                               w_shared_gate=w_sg)["y"]
    total = np.zeros_like(full)
    for b, e in zip(cuts[:-1], cuts[1:]):
        layer, nbytes = _shard_layer(m, wl, L, b, e, _flags(m, path), w_sg)
        g = run_gpu(m, layer, L["x"], out_f32=True)
        assert g["status"] == 0
        check_routing(g, oracle_route(wl, L), wl.E)  # the routing is the whole layer's
        ref = oracle.layer_tokens_shard(d, F, E, k, S, L["x"], L["w_router"], L["bias"], L["codes"], L["scales"],
                                        b, e, b == 0, w_shared_gate=w_sg)
        # the shard's part, to the fp32 tolerance of the whole layer's scale
        assert np.max(np.abs(g["y"] - ref)) <= F32_TOL * np.max(np.abs(full))
        lw = layer.weight_bytes()
        assert lw >= nbytes and lw <= 1.4 * nbytes + 2 * 17408 * 32  # only this shard's experts (+ tile padding)
        total += g["y"]
        layer.close()
    check_output(total, full, F32_TOL)


def test_full_size_decode_layer_in_four_shards(m):
    """The decode shapes (d = ffn = 2880, E = 128, k = 4) split into four shards of 32 experts."""
    wl = synth.WORKLOADS["decode"].with_(T=4)
    L = synth.gen_layer(wl, 3, T=4)
    full = oracle.layer_tokens_parallel(wl.d, wl.ffn, wl.E, wl.k, 0, L["x"], L["w_router"], L["bias"],
                                        L["codes"], L["scales"])["y"]
    total = np.zeros_like(full)
    for b in range(0, 128, 32):
        layer, _ = _shard_layer(m, wl, L, b, b + 32, 0)
        g = run_gpu(m, layer, L["x"], out_f32=True)
        assert g["status"] == 0
        total += g["y"]
        layer.close()
    check_output(total, full, F32_TOL)


def test_shard_config_is_validated(m):
    wl = synth.WORKLOADS["tiny"]
    for b, e in ((3, 3), (5, 2), (-1, 4), (0, 9)):
        with pytest.raises(m.MoeError) as ei:
            m.MoeLayer(m.LayerShape(wl.d, wl.ffn, wl.E, wl.k, expert_begin=b, expert_end=e))
        assert ei.value.code == m.MOE_ERR_INVALID_ARG
