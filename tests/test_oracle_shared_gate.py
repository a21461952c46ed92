"""Pins of the oracle's sigmoid-gated shared expert (CPU only).

The layer with a shared-expert gate row w_sg [d]:
    y_t = sum_j g_j part_j + s_t * shared(x_t),   s_t = sigmoid(w_sg . x_t)
("Nebula", table of components held on the GPU: one fp32 "shared expert gate"
row of the hidden size per layer; "Running Qwen3.8-Flash-Next on a 32 GB Mac
with Transformers", table of MoE blocks with gate, shared_expert and
shared_expert_gate). Pinned here against things other than the oracle's own
formula: the exact value sigmoid(0) = 1/2, a one-hot gate row whose dot
product is a single exact product, saturation at both ends (the sign of the
exponent), and an independent dense float64 PyTorch restatement.
"""
import math

import numpy as np
import pytest

import oracle
import synth

WL = synth.WORKLOADS["tiny"].with_(name="tiny_shared", T=6, shared_ffn=64)


def _layers(w_sg, wl=WL, layer=3):
    L = synth.gen_layer(wl, layer)
    args = (wl.d, wl.ffn, wl.E, wl.k)
    tail = (L["x"], L["w_router"], L["bias"], L["codes"], L["scales"])
    y_u = oracle.layer_tokens(*args, wl.shared_ffn, *tail)["y"]  # shared expert with weight 1
    y_r = oracle.layer_tokens(*args, 0, *tail)["y"]  # routed experts only (the shared bytes are ignored)
    y_g = oracle.layer_tokens(*args, wl.shared_ffn, *tail, w_shared_gate=w_sg)["y"]
    return L, y_u, y_r, y_g


def _x_f64(L):
    return (L["x"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_zero_gate_row_weighs_the_shared_expert_one_half():
    _, y_u, y_r, y_g = _layers(np.zeros(WL.d, dtype=np.float32))
    assert not np.allclose(y_u, y_r)  # the shared expert contributes
    np.testing.assert_allclose(y_g, y_r + 0.5 * (y_u - y_r), rtol=0, atol=1e-12 * np.abs(y_u).max())


def test_one_hot_gate_row_scales_each_token_by_its_own_sigmoid():
    i, c = 17, np.float32(0.75)
    w = np.zeros(WL.d, dtype=np.float32)
    w[i] = c
    L, y_u, y_r, y_g = _layers(w)
    z = float(c) * _x_f64(L)[:, i]  # one exact product: the whole dot product
    s = np.array([1.0 / (1.0 + math.exp(-v)) for v in z])
    np.testing.assert_allclose(y_g, y_r + s[:, None] * (y_u - y_r), rtol=0, atol=1e-12 * np.abs(y_u).max())
    for t in range(WL.T):
        assert oracle.shared_gate_token(L["x"][t], w) == pytest.approx(s[t], rel=1e-15)


def test_gate_saturates_towards_the_sign_of_its_logit():
    i = 5
    w = np.zeros(WL.d, dtype=np.float32)
    w[i] = 1e4
    L, y_u, y_r, y_g = _layers(w)
    xi = _x_f64(L)[:, i]
    assert (xi > 0).any() and (xi < 0).any()
    scale = np.abs(y_u).max()
    for t in range(WL.T):
        if abs(xi[t]) * 1e4 < 50:
            continue
        target = y_u[t] if xi[t] > 0 else y_r[t]  # sigmoid(+large) = 1, sigmoid(-large) = 0
        np.testing.assert_allclose(y_g[t], target, rtol=0, atol=1e-12 * scale)


def test_gated_layer_matches_dense_torch_float64():
    """Independent restatement with dense float64 matrices and torch.sigmoid / silu / softmax / topk."""
    torch = pytest.importorskip("torch")
    F_ = torch.nn.functional
    wl = WL
    L = synth.gen_layer(wl, 1)
    w_sg = synth.gen_shared_gate(wl.seed(1), wl.d)
    r = oracle.layer_tokens(wl.d, wl.ffn, wl.E, wl.k, wl.shared_ffn, L["x"], L["w_router"], L["bias"],
                            L["codes"], L["scales"], w_shared_gate=w_sg)
    from test_oracle_pins import dense_from_mx, expert_slices
    x = torch.tensor(_x_f64(L))
    logits = x @ torch.tensor(L["w_router"].astype(np.float64)).T
    vals, idx = torch.topk(logits, wl.k, dim=1)
    srt = torch.sort(logits, dim=1, descending=True).values
    assert torch.all(srt[:, wl.k - 1] - srt[:, wl.k] > 1e-9)
    g = torch.softmax(vals, dim=1)
    gate = torch.sigmoid(x @ torch.tensor(w_sg.astype(np.float64)))
    assert 0.05 < float(gate.min()) and float(gate.max()) < 0.95  # a gate that matters
    S = wl.shared_ffn
    cs, ss = expert_slices(L["codes"], L["scales"], wl.d, wl.ffn, wl.E, S)
    Wgu_s = torch.tensor(dense_from_mx(cs, ss, 2 * S, wl.d))
    Wd_s = torch.tensor(dense_from_mx(cs[S * wl.d:], ss[2 * S * wl.d // 32:], wl.d, S))
    y = torch.zeros(wl.T, wl.d, dtype=torch.float64)
    for t in range(wl.T):
        for j in range(wl.k):
            c, s = expert_slices(L["codes"], L["scales"], wl.d, wl.ffn, int(idx[t, j]))
            Wgu = torch.tensor(dense_from_mx(c, s, 2 * wl.ffn, wl.d))
            Wd = torch.tensor(dense_from_mx(c[wl.ffn * wl.d:], s[2 * wl.ffn * wl.d // 32:], wl.d, wl.ffn))
            y[t] += g[t, j] * (Wd @ (F_.silu(Wgu[: wl.ffn] @ x[t]) * (Wgu[wl.ffn:] @ x[t])))
        y[t] += gate[t] * (Wd_s @ (F_.silu(Wgu_s[:S] @ x[t]) * (Wgu_s[S:] @ x[t])))
    ref = y.numpy()
    assert np.max(np.abs(r["y"] - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_gate_row_without_shared_expert_is_rejected():
    L = synth.gen_layer(synth.WORKLOADS["tiny"], 0)
    wl = synth.WORKLOADS["tiny"]
    with pytest.raises(ValueError):
        oracle.layer_tokens(wl.d, wl.ffn, wl.E, wl.k, 0, L["x"], L["w_router"], None, L["codes"], L["scales"],
                            w_shared_gate=np.zeros(wl.d, dtype=np.float32))
