"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test checks the oracle against what the pages or the mathematics fix:
bit-field definitions of E2M1/E8M0, the expert byte count the "Neural Server"
technical page prints, closed-form layers, brute-force routing, invariants,
exact scaling, relabelling, and an independent dense float64 restatement in
PyTorch. The cases are chosen so that a plausible slip in the oracle (a wrong
table entry, swapped nibbles, a transposed matrix, gate/up swapped, a dropped
scale, a wrong tie rule, a softmax over the wrong set) fails at least one.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers (test-side, independent)

def e2m1_from_fields(code: int) -> float:
    """OCP MX v1.0 E2M1: sign, 2-bit exponent with bias 1, 1-bit mantissa; exponent 0 is subnormal."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = (m * 0.5) if e == 0 else (2.0 ** (e - 1)) * (1.0 + m / 2.0)
    return -mag if s else mag


def dense_from_mx(codes: np.ndarray, scales: np.ndarray, R: int, K: int) -> np.ndarray:
    """Dense float64 [R, K] from canonical MXFP4 bytes, written independently of the oracle."""
    b = codes[: R * K // 2].reshape(R, K // 2).astype(np.int64)
    c = np.empty((R, K), dtype=np.int64)
    c[:, 0::2] = b & 15
    c[:, 1::2] = b >> 4
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m / 2.0, (e - 1).astype(np.int32)))
    v = np.where(s == 1, -mag, mag)
    sc = np.ldexp(1.0, scales[: R * K // 32].reshape(R, K // 32).astype(np.int32) - 127)
    return v * np.repeat(sc, 32, axis=1)


def expert_slices(codes, scales, d, F, j, f=None):
    f = F if f is None else f
    cb, sb = 3 * F * d // 2, 3 * F * d // 32
    c = codes[j * cb: j * cb + 3 * f * d // 2]
    s = scales[j * sb: j * sb + 3 * f * d // 32]
    return c, s


def bf16_to_f64(x_bits: np.ndarray) -> np.ndarray:
    return (x_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Exact only for values representable in bf16 (the tests use such values)."""
    f = np.asarray(v, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not representable in bf16"
    return (bits >> 16).astype(np.uint16)


# ---------------------------------------------------------------- element formats

def test_e2m1_table_exhaustive():
    for code in range(16):
        assert oracle.e2m1(code) == e2m1_from_fields(code), code
    assert math.copysign(1.0, oracle.e2m1(8)) == -1.0  # code 8 is -0


def test_e8m0_exhaustive():
    for e in range(255):
        assert oracle.e8m0(e) == math.ldexp(1.0, e - 127), e
    assert math.isnan(oracle.e8m0(255))


def test_bf16_widening():
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3F00: 0.5, 0x4049: 3.140625, 0x0000: 0.0, 0x7F7F: 3.3895313892515355e38,
             0x0001: 2.0 ** -133}
    for bits, v in cases.items():
        assert oracle.bf16(bits) == v, hex(bits)


def test_mx_element_nibble_order_and_scale_blocks():
    K = 64
    codes = np.zeros(2 * K // 2, dtype=np.uint8)
    scales = np.array([127, 128, 130, 126], dtype=np.uint8)  # rows 0,1 x blocks 0,1
    codes[0] = (2 << 4) | 1  # element 0 -> code 1 (0.5), element 1 -> code 2 (1.0)
    codes[15] = (0xF << 4) | 0x7  # elements 30, 31 -> +6, -6
    codes[16] = 0x3  # element 32 -> code 3 (1.5), scale block 1
    codes[32 + 5] = 0x0A << 4  # row 1, element 11 -> code 10 (-1.0)
    assert oracle.mx_element(codes, scales, K, 0, 0) == 0.5
    assert oracle.mx_element(codes, scales, K, 0, 1) == 1.0
    assert oracle.mx_element(codes, scales, K, 0, 30) == 6.0
    assert oracle.mx_element(codes, scales, K, 0, 31) == -6.0
    assert oracle.mx_element(codes, scales, K, 0, 32) == 1.5 * 2.0
    assert oracle.mx_element(codes, scales, K, 1, 11) == -1.0 * 2.0 ** 3
    assert oracle.mx_element(codes, scales, K, 1, 40) == 0.0


# ---------------------------------------------------------------- sizes printed on the pages

def test_expert_bytes_match_page():
    with open(os.path.join(GOLDEN, "expert_bytes.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        got = oracle.expert_code_bytes(case["d"], case["ffn"]) + oracle.expert_scale_bytes(case["d"], case["ffn"])
        assert got == case["expert_bytes"]
    wl = synth.WORKLOADS["decode"]
    assert wl.expert_bytes() == 13_219_200
    assert synth.WORKLOADS["small"].expert_bytes() == 1_671_168
    assert synth.WORKLOADS["small"].expert_bytes(2048) == 6_684_672
    assert synth.WORKLOADS["tiny"].expert_bytes() == 208_896


# ---------------------------------------------------------------- closed-form layers

def _uniform_expert(d, f, code_byte, gu_scale, dn_scale):
    codes = np.full(3 * f * d // 2, code_byte, dtype=np.uint8)
    scales = np.empty(3 * f * d // 32, dtype=np.uint8)
    scales[: 2 * f * d // 32] = gu_scale
    scales[2 * f * d // 32:] = dn_scale
    return codes, scales


def silu(z):
    return z / (1.0 + math.exp(-z))


def test_all_ones_layer_closed_form():
    d = F = 32
    codes, scales = _uniform_expert(d, F, 0x22, 127, 127)  # every element 1.0
    codes = np.concatenate([codes, codes])
    scales = np.concatenate([scales, scales])
    rng = np.random.default_rng(1)
    xv = rng.integers(-8, 9, size=(3, d)) / 8.0
    x = f64_to_bf16_bits(xv)
    w_router = np.zeros((2, d), dtype=np.float32)
    r = oracle.layer_tokens(d, F, 2, 1, 0, x, w_router, None, codes, scales)
    for t in range(3):
        s = float(xv[t].sum())
        expect = F * silu(s) * s
        assert np.all(r["y"][t] == pytest.approx(expect, rel=1e-14, abs=1e-14))
        assert r["ids"][t, 0] == 0 and r["gates"][t, 0] == 1.0  # tie between equal logits -> lower index


def test_scale_exponents_enter_as_powers_of_two():
    d = F = 32
    c1, s1 = _uniform_expert(d, F, 0x22, 127, 127)
    c2, s2 = _uniform_expert(d, F, 0x22, 126, 130)  # gate/up halved, down x8
    xv = np.linspace(-1, 1, d)
    x = f64_to_bf16_bits(np.round(xv * 64) / 64)
    xs = bf16_to_f64(x)
    _, o1 = oracle.expert_ffn(c1, s1, d, F, xs)
    _, o2 = oracle.expert_ffn(c2, s2, d, F, xs)
    s = xs.sum()
    assert o1 == pytest.approx(np.full(d, F * silu(s) * s), rel=1e-14)
    assert o2 == pytest.approx(np.full(d, 8 * F * silu(s / 2) * (s / 2)), rel=1e-14)


def test_zero_gate_rows_give_zero_output():
    d, F = 64, 32
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 256, size=3 * F * d // 2, dtype=np.uint8)
    scales = rng.integers(118, 126, size=3 * F * d // 32, dtype=np.uint8)
    codes[: F * d // 2] = 0  # gate rows [0, F) are all +0
    x = rng.standard_normal(d)
    h, out = oracle.expert_ffn(codes, scales, d, F, x)
    assert np.all(h == 0.0) and np.all(out == 0.0)
    codes2 = codes.copy()
    codes2[: F * d // 2] = 0x88  # -0 codes are zero too
    h2, out2 = oracle.expert_ffn(codes2, scales, d, F, x)
    assert np.all(out2 == 0.0)


def test_one_nonzero_code_per_row_is_a_gather():
    """Non-square (d != F) sparse expert: each row picks one input entry, which fixes
    the row/column orientation of gate/up and down and the gate-vs-up order."""
    d, F = 96, 64
    rng = np.random.default_rng(3)
    codes = np.zeros(3 * F * d // 2, dtype=np.uint8)
    scales = np.full(3 * F * d // 32, 127, dtype=np.uint8)
    col_g = rng.integers(0, d, size=F)
    col_u = rng.integers(0, d, size=F)
    col_d = rng.integers(0, F, size=d)
    val = {2: 1.0, 4: 2.0, 10: -1.0, 13: -3.0}
    cg = rng.choice(list(val), size=F)
    cu = rng.choice(list(val), size=F)
    cd = rng.choice(list(val), size=d)

    def put(base, K, r, c, code):
        i = base + r * (K // 2) + c // 2
        codes[i] |= (code << 4) if (c & 1) else code

    for i in range(F):
        put(0, d, i, col_g[i], cg[i])
        put(0, d, F + i, col_u[i], cu[i])
    for r in range(d):
        put(2 * F * d // 2, F, r, col_d[r], cd[r])
    x = rng.standard_normal(d)
    h, out = oracle.expert_ffn(codes, scales, d, F, x)
    g = np.array([val[cg[i]] * x[col_g[i]] for i in range(F)])
    u = np.array([val[cu[i]] * x[col_u[i]] for i in range(F)])
    h_ref = g / (1 + np.exp(-g)) * u
    out_ref = np.array([val[cd[r]] * h_ref[col_d[r]] for r in range(d)])
    assert np.array_equal(h, h_ref) or np.allclose(h, h_ref, rtol=1e-15, atol=0)
    assert np.allclose(out, out_ref, rtol=1e-15, atol=0)


# ---------------------------------------------------------------- routing

def _brute_topk(l, k):
    """The selected set is the unique k-subset whose every member beats every
    non-member in (value desc, index asc) order; within it, that same order."""
    E = len(l)
    key = lambda e: (l[e], -e)
    winners = [S for S in itertools.combinations(range(E), k)
               if min(key(e) for e in S) > max((key(e) for e in range(E) if e not in S), default=(-math.inf, 0))]
    assert len(winners) == 1
    return sorted(winners[0], key=key, reverse=True)


def test_topk_brute_force_small():
    rng = np.random.default_rng(4)
    for trial in range(300):
        E = int(rng.integers(1, 11))
        k = int(rng.integers(1, E + 1))
        l = rng.integers(-3, 4, size=E).astype(np.float64) if trial % 2 else rng.standard_normal(E)
        ids, gates = oracle.topk_token(l, k)
        assert list(ids) == _brute_topk(list(l), k)
        sel = l[ids]
        ref = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()
        assert np.allclose(gates, ref, rtol=1e-15, atol=1e-16)


def test_gates_equal_renormalised_full_softmax():
    rng = np.random.default_rng(5)
    for _ in range(50):
        E = int(rng.integers(4, 300))
        k = int(rng.integers(1, min(E, 10) + 1))
        l = rng.standard_normal(E) * 3
        ids, gates = oracle.topk_token(l, k)
        full = np.exp(l - l.max())
        full /= full.sum()
        ren = full[ids] / full[ids].sum()
        assert np.allclose(gates, ren, rtol=1e-13, atol=0)
        assert abs(gates.sum() - 1.0) < 1e-15 * k + 1e-16
        assert np.all(np.diff(gates) <= 0)


def test_exact_ties_go_to_lower_index():
    d, E = 32, 8
    w = np.zeros((E, d), dtype=np.float32)
    w[[1, 3, 6], 0] = 2.0  # experts 1, 3, 6 tie at the top
    w[[0, 5], 0] = 1.0  # experts 0, 5 tie next
    x = np.zeros((1, d), dtype=np.uint16)
    x[0, 0] = 0x3F80  # 1.0
    r = oracle.route(x, w, None, 4)
    assert list(r["ids"][0]) == [1, 3, 6, 0]
    assert np.allclose(r["gates"][0][:3], r["gates"][0][0])


def test_logits_are_exact_dot_products():
    """bf16 x fp32 products are exact in fp64; integer-valued cases must come out exact."""
    rng = np.random.default_rng(6)
    d, E = 64, 5
    w = rng.integers(-100, 100, size=(E, d)).astype(np.float32)
    xv = rng.integers(-100, 100, size=d).astype(np.float64)
    b = rng.integers(-5, 5, size=E).astype(np.float32)
    l = oracle.logits_token(f64_to_bf16_bits(xv), w, b)
    assert np.array_equal(l, w.astype(np.float64) @ xv + b)


def test_bucketing_is_stable_counting_sort():
    rng = np.random.default_rng(7)
    for _ in range(50):
        E = int(rng.integers(1, 40))
        P = int(rng.integers(0, 200))
        ids = rng.integers(0, E, size=P).astype(np.int32)
        counts, offsets, perm, inv = oracle.bucket(ids, E)
        assert np.array_equal(counts, np.bincount(ids, minlength=E))
        assert offsets[0] == 0 and offsets[-1] == P and np.array_equal(np.diff(offsets), counts)
        assert np.array_equal(perm, np.argsort(ids, kind="stable"))
        assert np.array_equal(inv[perm], np.arange(P))


# ---------------------------------------------------------------- whole-layer properties

def _tiny_layer(seed_layer=0, wl=None):
    wl = wl or synth.WORKLOADS["tiny"]
    return wl, synth.gen_layer(wl, seed_layer)


def test_layer_matches_dense_torch_float64():
    """Independent restatement: dense float64 matrices + torch ops (silu, matmul, softmax, topk)."""
    torch = pytest.importorskip("torch")
    F_ = torch.nn.functional
    for wl in [synth.WORKLOADS["tiny"],
               synth.WORKLOADS["tiny"].with_(name="tiny_shared", T=5, shared_ffn=64, zipf_bias=1.1)]:
        L = synth.gen_layer(wl, 0)
        r = oracle.layer_tokens(wl.d, wl.ffn, wl.E, wl.k, wl.shared_ffn, L["x"], L["w_router"], L["bias"],
                                L["codes"], L["scales"])
        x = torch.tensor(bf16_to_f64(L["x"]))
        W = torch.tensor(L["w_router"].astype(np.float64))
        logits = x @ W.T + (torch.tensor(L["bias"].astype(np.float64)) if L["bias"] is not None else 0)
        vals, idx = torch.topk(logits, wl.k, dim=1)
        srt = torch.sort(logits, dim=1, descending=True).values
        assert torch.all(srt[:, wl.k - 1] - srt[:, wl.k] > 1e-9)  # no near-ties, so torch.topk is unambiguous
        assert np.array_equal(r["ids"], idx.numpy())
        g = torch.softmax(vals, dim=1)
        y = torch.zeros(wl.T, wl.d, dtype=torch.float64)
        for t in range(wl.T):
            for j in range(wl.k):
                c, s = expert_slices(L["codes"], L["scales"], wl.d, wl.ffn, int(idx[t, j]))
                Wgu = torch.tensor(dense_from_mx(c, s, 2 * wl.ffn, wl.d))
                Wd = torch.tensor(dense_from_mx(c[wl.ffn * wl.d:], s[2 * wl.ffn * wl.d // 32:], wl.d, wl.ffn))
                h = F_.silu(Wgu[: wl.ffn] @ x[t]) * (Wgu[wl.ffn:] @ x[t])
                y[t] += g[t, j] * (Wd @ h)
            if wl.shared_ffn:
                S = wl.shared_ffn
                c, s = expert_slices(L["codes"], L["scales"], wl.d, wl.ffn, wl.E, S)
                Wgu = torch.tensor(dense_from_mx(c, s, 2 * S, wl.d))
                Wd = torch.tensor(dense_from_mx(c[S * wl.d:], s[2 * S * wl.d // 32:], wl.d, S))
                y[t] += Wd @ (F_.silu(Wgu[:S] @ x[t]) * (Wgu[S:] @ x[t]))
        assert np.allclose(r["gates"], g.numpy(), rtol=1e-13, atol=0)
        ref = y.numpy()
        assert np.max(np.abs(r["y"] - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_down_scale_plus_one_doubles_output_exactly():
    wl, L = _tiny_layer()
    r1 = oracle.layer_tokens(wl.d, wl.ffn, wl.E, wl.k, 0, L["x"], L["w_router"], None, L["codes"], L["scales"])
    sc = L["scales"].copy()
    per = wl.scale_bytes()
    gu = 2 * wl.ffn * wl.d // 32
    for e in range(wl.E):
        sc[e * per + gu:(e + 1) * per] += 1
    r2 = oracle.layer_tokens(wl.d, wl.ffn, wl.E, wl.k, 0, L["x"], L["w_router"], None, L["codes"], sc)
    assert np.array_equal(r2["y"], 2.0 * r1["y"])


def test_expert_relabelling_permutes_ids_and_keeps_output():
    wl, L = _tiny_layer()
    rng = np.random.default_rng(8)
    sigma = rng.permutation(wl.E)  # new expert sigma[e] holds old expert e
    cb, sb = wl.code_bytes(), wl.scale_bytes()
    codes = np.empty_like(L["codes"])
    scales = np.empty_like(L["scales"])
    w = np.empty_like(L["w_router"])
    for e in range(wl.E):
        n = sigma[e]
        codes[n * cb:(n + 1) * cb] = L["codes"][e * cb:(e + 1) * cb]
        scales[n * sb:(n + 1) * sb] = L["scales"][e * sb:(e + 1) * sb]
        w[n] = L["w_router"][e]
    r1 = oracle.layer_tokens(wl.d, wl.ffn, wl.E, wl.k, 0, L["x"], L["w_router"], None, L["codes"], L["scales"])
    r2 = oracle.layer_tokens(wl.d, wl.ffn, wl.E, wl.k, 0, L["x"], w, None, codes, scales)
    assert np.array_equal(r2["ids"], sigma[r1["ids"]])
    assert np.array_equal(r2["y"], r1["y"])


def test_token_subset_equals_full_rows():
    wl = synth.WORKLOADS["tiny"].with_(T=7)
    L = synth.gen_layer(wl, 0)
    full = oracle.layer_tokens(wl.d, wl.ffn, wl.E, wl.k, 0, L["x"], L["w_router"], None, L["codes"], L["scales"])
    sub = oracle.layer_tokens(wl.d, wl.ffn, wl.E, wl.k, 0, L["x"], L["w_router"], None, L["codes"], L["scales"],
                              tokens=[6, 2])
    assert np.array_equal(sub["y"], full["y"][[6, 2]])
    rt = oracle.route(L["x"], L["w_router"], None, wl.k)
    assert np.array_equal(rt["ids"], full["ids"])
    assert np.array_equal(rt["gates"], full["gates"])


def test_invalid_inputs_are_rejected():
    d, F = 32, 32
    codes, scales = _uniform_expert(d, F, 0x22, 127, 127)
    scales = scales.copy()
    scales[3] = 255
    with pytest.raises(ValueError):
        oracle.expert_ffn(codes, scales, d, F, np.zeros(d))
    with pytest.raises(ValueError):
        oracle.expert_ffn(codes, scales, 48, F, np.zeros(48))
