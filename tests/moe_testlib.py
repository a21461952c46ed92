"""Shared helpers of the GPU parity tests: run a layer through the C ABI and
compare it with the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np

import oracle
import synth

BF16_TOL = 2e-2  # max |y_gpu - y_ref| <= BF16_TOL * ||y_ref||_inf (bf16 output)
F32_TOL = 1e-4  # max |y_gpu - y_ref| <= F32_TOL * ||y_ref||_inf (fp32 output)
GATE_TOL = 1e-6  # max |g_gpu - g_ref| (gates are in [0, 1])


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def torch_mod():
    import torch
    return torch


def build_lib():
    from routed_expert_ffn_warp_gb300 import build as b
    b.build()
    import routed_expert_ffn_warp_gb300 as m
    m.load_library()
    return m


def make_layer(m, wl: synth.Workload, L: dict, t_max: int | None = None, out_f32: bool = False, device: int = 0,
               flags: int = 0, w_shared_gate=None):
    shape = m.LayerShape(d=wl.d, ffn=wl.ffn, n_experts=wl.E, top_k=wl.k, shared_ffn=wl.shared_ffn,
                         t_max=wl.T if t_max is None else t_max,
                         out_dtype=m.MOE_OUT_F32 if out_f32 else m.MOE_OUT_BF16, flags=flags)
    layer = m.MoeLayer(shape, device)
    layer.load(L["w_router"], L["bias"], L["codes"], L["scales"], w_shared_gate=w_shared_gate)
    return layer


def run_gpu(m, layer, x_bits: np.ndarray, out_f32: bool = False) -> dict:
    """One forward on the GPU via moe_forward (device buffers); returns host copies."""
    torch = torch_mod()
    T, d = x_bits.shape
    E, k = layer.shape.n_experts, layer.shape.top_k
    x = torch.from_numpy(x_bits.view(np.int16).copy()).cuda()
    out = torch.empty((T, d), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    layer.forward(x, T, out, stream)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts = torch.empty((E,), dtype=torch.int32, device="cuda")
    offsets = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
    perm = torch.empty((T * k,), dtype=torch.int32, device="cuda")
    inv = torch.empty((T * k,), dtype=torch.int32, device="cuda")
    lhi = torch.empty((T, E), dtype=torch.float32, device="cuda")
    llo = torch.empty((T, E), dtype=torch.float32, device="cuda")
    layer.routing(ids, gates, counts, offsets, perm, stream, inv=inv)
    layer.logits(lhi, llo, stream)
    torch.cuda.synchronize()
    st = layer.status()
    y = out.float().cpu().numpy().astype(np.float64)
    return {"y": y, "ids": ids.cpu().numpy(), "gates": gates.cpu().numpy(), "counts": counts.cpu().numpy(),
            "offsets": offsets.cpu().numpy(), "perm": perm.cpu().numpy(), "inv": inv.cpu().numpy(),
            "logits": lhi.cpu().numpy().astype(np.float64) + llo.cpu().numpy().astype(np.float64),
            "status": st}


def check_routing(gpu: dict, ref_route: dict, E: int):
    assert np.array_equal(gpu["ids"], ref_route["ids"]), "routing ids differ from the oracle"
    assert np.array_equal(gpu["counts"], ref_route["counts"])
    assert np.array_equal(gpu["offsets"], ref_route["offsets"])
    assert np.array_equal(gpu["perm"], ref_route["perm"])
    assert np.array_equal(gpu["inv"], ref_route["inv"])
    assert np.max(np.abs(gpu["gates"] - ref_route["gates"])) <= GATE_TOL


def check_output(y_gpu: np.ndarray, y_ref: np.ndarray, tol: float):
    scale = np.max(np.abs(y_ref))
    err = np.max(np.abs(y_gpu - y_ref)) if y_ref.size else 0.0
    assert err <= tol * scale, f"max|dy| = {err:.3e} > {tol} * {scale:.3e}"
    return err / scale if scale > 0 else 0.0


def oracle_layer(wl: synth.Workload, L: dict, tokens=None, w_shared_gate=None) -> dict:
    return oracle.layer_tokens(wl.d, wl.ffn, wl.E, wl.k, wl.shared_ffn, L["x"], L["w_router"], L["bias"],
                               L["codes"], L["scales"], tokens=tokens, w_shared_gate=w_shared_gate)


def oracle_route(wl: synth.Workload, L: dict) -> dict:
    return oracle.route(L["x"], L["w_router"], L["bias"], wl.k)
