"""moe_route_static: routing for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (an allocator that owns all device memory,
or a code region where allocation is forbidden). moe_route_static runs the
router, top-k and counting sort with a static device scratch array instead.
This test calls it twice in a row through the C ABI and compares both results
with the routing the regular entry point (moe_forward + moe_get_routing)
produced for the same inputs, and with the CPU oracle's routing: ids, counts,
offsets and perm bit for bit, gates within the gate tolerance of the other
tests.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

import oracle
import synth
from moe_testlib import GATE_TOL, build_lib, make_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU not available for a gpu-marked test")
    return build_lib()


def _routing_via_forward(m, wl, L):
    import torch
    layer = make_layer(m, wl, L, t_max=wl.T)
    x = torch.from_numpy(L["x"].view(np.int16).copy()).cuda()
    out = torch.empty((wl.T, wl.d), dtype=torch.bfloat16, device="cuda")
    r = {"ids": torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda"),
         "gates": torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda"),
         "counts": torch.empty((wl.E,), dtype=torch.int32, device="cuda"),
         "offsets": torch.empty((wl.E + 1,), dtype=torch.int32, device="cuda"),
         "perm": torch.empty((wl.T * wl.k,), dtype=torch.int32, device="cuda")}
    layer.forward(x, wl.T, out)
    layer.routing(r["ids"], r["gates"], r["counts"], r["offsets"], r["perm"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    layer.close()
    return {k: v.cpu().numpy() for k, v in r.items()}


def _routing_static(m, wl, L):
    import torch
    x = torch.from_numpy(L["x"].view(np.int16).copy()).cuda()
    w = torch.from_numpy(L["w_router"]).cuda()
    b = torch.from_numpy(L["bias"]).cuda() if L["bias"] is not None else None
    r = {"ids": torch.full((wl.T, wl.k), -1, dtype=torch.int32, device="cuda"),
         "gates": torch.full((wl.T, wl.k), -1.0, dtype=torch.float32, device="cuda"),
         "counts": torch.full((wl.E,), -1, dtype=torch.int32, device="cuda"),
         "offsets": torch.full((wl.E + 1,), -1, dtype=torch.int32, device="cuda"),
         "perm": torch.full((wl.T * wl.k,), -1, dtype=torch.int32, device="cuda")}
    m.moe_route_static(x, wl.T, wl.d, w, b, wl.E, wl.k, r["ids"], r["gates"], r["counts"], r["offsets"], r["perm"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in r.items()}


@pytest.mark.parametrize("case", [
    synth.WORKLOADS["tiny"],
    synth.WORKLOADS["tiny"].with_(name="zipf40", T=40, E=64, k=4, zipf_bias=1.1),
])
def test_static_routing_matches_forward_twice(m, case):
    L = synth.gen_layer(case, 0)
    ref = _routing_via_forward(m, case, L)
    orc = oracle.route(L["x"], L["w_router"], L["bias"], case.k)
    for _ in range(2):  # two calls in a row share the static scratch
        got = _routing_static(m, case, L)
        for key in ("ids", "counts", "offsets", "perm"):
            assert np.array_equal(got[key], ref[key]), key
            assert np.array_equal(got[key], orc[key]), key + " differs from the oracle"
        assert np.max(np.abs(got["gates"] - ref["gates"])) <= GATE_TOL
        assert np.max(np.abs(got["gates"] - orc["gates"])) <= GATE_TOL


def test_static_routing_rejects_sizes_beyond_its_scratch(m):
    with pytest.raises(m.MoeError) as ei:
        m.moe_route_static(0, 1024, 256, 0, None, 128, 4, 0, 0, 0, 0, 0)  # 1024 * 128 logits > 65536
    assert ei.value.code == m.MOE_ERR_INVALID_ARG
    assert "65536" in str(ei.value)
