"""The C-ABI library builds for sm_103a, loads, and exports every entry point
that include/moe.h declares; host-side argument checks run without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from routed_expert_ffn_warp_gb300 import build
    build.build()
    import routed_expert_ffn_warp_gb300 as m
    return m.load_library()


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for n in ["moe_create", "moe_load_router", "moe_load_experts", "moe_forward", "moe_get_routing",
              "moe_get_status", "moe_last_error", "moe_destroy"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import routed_expert_ffn_warp_gb300 as m
    for name in declared_entry_points():
        assert hasattr(lib, name), name
        assert name in m.EXPORTED, name


def test_invalid_config_rejected_before_touching_the_gpu(lib):
    import routed_expert_ffn_warp_gb300 as m
    bad = [dict(d=48), dict(ffn=0), dict(n_experts=0), dict(top_k=9), dict(t_max=-1), dict(out_dtype=3),
           dict(shared_ffn=40), dict(n_experts=600)]
    for kw in bad:
        c = dict(d=256, ffn=512, n_experts=8, top_k=2, shared_ffn=0, t_max=4, out_dtype=0, flags=0)
        c.update(kw)
        cfg = m.moe_config(**c)
        with pytest.raises(m.MoeError) as ei:
            m.moe_create(cfg, 0)
        assert ei.value.code == m.MOE_ERR_INVALID_ARG, kw
        assert m.moe_last_error(None)


def test_null_context_calls(lib):
    import routed_expert_ffn_warp_gb300 as m
    assert lib.moe_forward(None, None, 1, None, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_load_experts(None, None, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_get_status(None, 0) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_weight_bytes(None) == 0
    lib.moe_destroy(None)


def test_mma_probe_rejects_bad_arguments_without_a_gpu(lib):
    tf = ctypes.c_double()
    assert lib.moe_probe_mma_rate(0, 0, 192, ctypes.byref(tf), None) == -1  # MOE_ERR_INVALID_ARG
    assert lib.moe_probe_mma_rate(0, 1000, 24, ctypes.byref(tf), None) == -1  # N not a multiple of 16
    assert lib.moe_probe_mma_rate(0, 1000, 256, ctypes.byref(tf), None) == -1  # N above the probed widths
    assert b"mmas_per_sm" in lib.moe_probe_error()


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """Without the compiled library the binding raises: there is no CPU fallback to silently take over."""
    import routed_expert_ffn_warp_gb300 as m
    monkeypatch.setattr(m, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        m.load_library(str(tmp_path / "libmoe_gb300.so"))
