"""The seeded input generator: determinism, shapes and the stated distributions."""
import numpy as np

import synth


def test_counter_based_and_deterministic():
    wl = synth.WORKLOADS["tiny"]
    a = synth.gen_layer(wl, 0)
    b = synth.gen_layer(wl, 0)
    for key in ("x", "w_router", "codes", "scales"):
        assert np.array_equal(a[key], b[key])
    # a prefix of a longer x is the shorter x (each value depends on its index only)
    x7 = synth.gen_x(5, 7, 64)
    x3 = synth.gen_x(5, 3, 64)
    assert np.array_equal(x7[:3], x3)
    # an expert's bytes do not depend on how many experts the layer has
    c8, s8 = synth.gen_experts(wl, 11)
    c4, s4 = synth.gen_experts(wl.with_(E=4), 11)
    assert np.array_equal(c8[: c4.size], c4) and np.array_equal(s8[: s4.size], s4)


def test_distributions():
    x = synth.bf16_bits_to_f32(synth.gen_x(1, 64, 2880)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    w = synth.gen_router(1, 128, 2880).astype(np.float64)
    assert abs(w.std() * np.sqrt(2880) - 1.0) < 0.01
    wl = synth.WORKLOADS["tiny"]
    codes, scales = synth.gen_experts(wl, 3)
    nib = np.concatenate([codes & 15, codes >> 4])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * nib.size / 16 and counts.max() < 1.1 * nib.size / 16
    assert scales.min() == 120 and scales.max() == 124


def test_zipf_bias_is_a_permuted_log_rank():
    b = synth.gen_bias(3003, 128, 1.1).astype(np.float64)
    ranks = np.exp(-b / 1.1)
    assert np.allclose(np.sort(ranks), np.arange(1, 129), rtol=1e-5)
    assert not np.all(np.diff(b) <= 0)  # not simply sorted by index


def test_workload_sizes():
    wl = synth.WORKLOADS["small"]
    assert wl.total_code_bytes == 256 * 3 * 512 * 2048 // 2 + 3 * 2048 * 2048 // 2
    assert wl.n_experts_stored == 257
