"""Pins of the oracle's affine group-64 expert format (CPU only).

"Running Qwen3.8-Flash-Next on a 32 GB Mac with Transformers": routed experts
as "3-bit MLX affine, group 64, 2.15 MB per expert", "a 16-bit scale and bias
per 64 weights", about 3.5 bits per weight, for the model's hidden size 2,560
and expert intermediate size 640. Readings (the pages give neither formula
nor packing): w = scale * q + bias, q unsigned; bf16 scale and bias; each
row's codes one little-endian bit stream.

Pinned against: the page's byte count; a numpy packbits restatement of the
bit layout; and the MXFP4 oracle (pinned on its own), through matrices whose
every weight both formats hold exactly, so the two expert FFNs must agree bit
for bit.
"""
import numpy as np
import pytest

import oracle

BF16 = {0.5: 0x3F00, -1.5: 0xBFC0}


def _bf16_bits(v: float) -> int:
    b = np.array([v], dtype=np.float32).view(np.uint32)[0]
    assert b & 0xFFFF == 0, "value must be exact in bf16"
    return int(b >> 16)


def test_expert_bytes_match_the_page():
    n = oracle.affine_expert_bytes(2560, 640, 3)
    assert n == 2_150_400  # "2.15 MB per expert"
    assert n * 8 / (3 * 640 * 2560) == 3.5  # "about 3.5 bits per weight"


def _pack_rows(q: np.ndarray, bits: int) -> np.ndarray:
    """Independent restatement of the layout: element c's bit b at stream position bits*c + b."""
    R, K = q.shape
    stream = ((q[:, :, None] >> np.arange(bits)) & 1).astype(np.uint8).reshape(R, K * bits)
    return np.packbits(stream, axis=1, bitorder="little")


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_codes_unpack_the_little_endian_bit_stream(bits):
    rng = np.random.default_rng(bits)
    R, K = 5, 192
    q = rng.integers(0, 1 << bits, size=(R, K))
    packed = np.ascontiguousarray(_pack_rows(q, bits))
    assert packed.shape == (R, K * bits // 8)
    for r in range(R):
        for c in range(K):
            assert oracle.affine_code(packed, K, bits, r, c) == q[r, c]


def _mx_code(v: float) -> int:
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    return (8 if v < 0 else 0) | mags.index(abs(v))


def _both_formats(rng, d: int, f: int):
    """One expert in MXFP4 (codes, scales) and in 3-bit affine form, with equal weights:
    w = (0.5 q - 1.5) * 2^k, k per group of 64 along the reduction axis."""
    def matrix(R, K):
        q = rng.integers(0, 8, size=(R, K))
        k = rng.integers(-3, 4, size=(R, K // 64))
        vals = 0.5 * q - 1.5
        mx_codes = np.vectorize(_mx_code)(vals).astype(np.uint8)
        mx_packed = (mx_codes[:, 0::2] | (mx_codes[:, 1::2] << 4)).astype(np.uint8)
        mx_scales = np.repeat(127 + k, 2, axis=1).astype(np.uint8)  # two 32-blocks per group of 64
        sc = np.vectorize(lambda e: _bf16_bits(0.5 * 2.0 ** e))(k).astype(np.uint16)
        bi = np.vectorize(lambda e: _bf16_bits(-1.5 * 2.0 ** e))(k).astype(np.uint16)
        return mx_packed, mx_scales, _pack_rows(q, 3), sc, bi
    gu = matrix(2 * f, d)
    dn = matrix(d, f)
    mx_codes = np.concatenate([gu[0].ravel(), dn[0].ravel()])
    mx_scales = np.concatenate([gu[1].ravel(), dn[1].ravel()])
    affine = np.concatenate([gu[2].ravel(), dn[2].ravel(), gu[3].ravel().view(np.uint8), dn[3].ravel().view(np.uint8),
                             gu[4].ravel().view(np.uint8), dn[4].ravel().view(np.uint8)])
    assert affine.nbytes == oracle.affine_expert_bytes(d, f, 3)
    return mx_codes, mx_scales, affine


def test_affine_expert_equals_mxfp4_expert_on_common_values():
    rng = np.random.default_rng(7)
    d, f = 128, 192
    mx_codes, mx_scales, affine = _both_formats(rng, d, f)
    x = rng.standard_normal(d)
    _, y_mx = oracle.expert_ffn(mx_codes, mx_scales, d, f, x)
    y_af = oracle.expert_ffn_affine(affine, d, f, 3, x)
    assert np.abs(y_mx).max() > 0
    assert np.array_equal(y_af, y_mx)  # same weights, same order of summation


def test_affine_rejects_shapes_off_the_group():
    with pytest.raises(ValueError):
        oracle.expert_ffn_affine(np.zeros(1024, dtype=np.uint8), 96, 64, 3, np.zeros(96))


@pytest.mark.parametrize("gated", [False, True])
def test_affine_layer_equals_mxfp4_layer_on_common_values(gated):
    """The affine layer (routing, gate weights, shared expert) against the MXFP4 layer oracle on
    experts both formats hold exactly: every output bit agrees."""
    rng = np.random.default_rng(11)
    d, F, S, E, k, T = 128, 128, 64, 4, 2, 5
    experts = [_both_formats(rng, d, F) for _ in range(E)] + [_both_formats(rng, d, S)]
    codes = np.concatenate([e[0] for e in experts])
    scales = np.concatenate([e[1] for e in experts])
    affine = np.concatenate([e[2] for e in experts])
    x = (rng.standard_normal((T, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    w_router = rng.standard_normal((E, d)).astype(np.float32) / np.sqrt(d)
    w_sg = rng.standard_normal(d).astype(np.float32) / np.sqrt(d) if gated else None
    mx = oracle.layer_tokens(d, F, E, k, S, x, w_router, None, codes, scales, w_shared_gate=w_sg)
    af = oracle.layer_tokens_affine(d, F, E, k, S, 3, x, w_router, None, affine, w_shared_gate=w_sg)
    assert np.array_equal(af["ids"], mx["ids"])
    assert np.array_equal(af["gates"], mx["gates"])
    assert np.abs(mx["y"]).max() > 0
    assert np.array_equal(af["y"], mx["y"])
    par = oracle.layer_tokens_affine_parallel(d, F, E, k, S, 3, x, w_router, None, affine, threads=3,
                                              w_shared_gate=w_sg)
    assert np.array_equal(par["y"], af["y"])
