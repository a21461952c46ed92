"""The bench's roofline arithmetic (CPU): algorithmic bytes and flops per layer.

Pinned to figures fixed outside this code: the 13,219,200-byte MXFP4 expert of
the "Neural Server" technical page (section "What it runs on and what it
runs": hidden 2880, gpt-oss-120B experts), and the per-layer totals that
follow from it for the four measured workloads (router rows in fp32, x in and
y out in bf16, the Zipf bias in fp32 for the verify workload).
"""
import pytest

bench = pytest.importorskip("bench")
import synth  # noqa: E402

EXPERT = 13_219_200  # one d = ffn = 2880 MXFP4 expert (codes + E8M0 scales), from the page


def test_expert_bytes_match_the_page():
    assert synth.WORKLOADS["decode"].expert_bytes() == EXPERT
    assert synth.WORKLOADS["small"].expert_bytes() == 1_671_168
    assert synth.WORKLOADS["small"].expert_bytes(2048) == 6_684_672


def test_decode_layer_bytes():
    # 4 experts + router 128 x 2880 fp32 + x and y of one token in bf16
    assert bench.layer_bytes(synth.WORKLOADS["decode"], 4, 1) == 4 * EXPERT + 1_474_560 + 2 * 5_760 == 54_362_880


def test_verify_small_prefill_layer_bytes():
    wl = synth.WORKLOADS["verify"]
    for U in (1, 16, 51):
        assert bench.layer_bytes(wl, U, 16) == U * EXPERT + 1_474_560 + 512 + 184_320
    wl = synth.WORKLOADS["small"]
    assert bench.layer_bytes(wl, 57, 8) == 57 * 1_671_168 + 6_684_672 + 2_097_152 + 65_536
    assert bench.layer_bytes(synth.WORKLOADS["prefill"], 128, 1024) == 1_705_328_640


def test_phase_bytes_split_the_expert_weights():
    for name, U in (("decode", 4), ("verify", 16), ("small", 57), ("prefill", 128)):
        wl = synth.WORKLOADS[name]
        pb = bench.phase_bytes(wl, U, wl.T)
        weights = U * wl.expert_bytes() + (wl.expert_bytes(wl.shared_ffn) if wl.shared_ffn else 0)
        assert pb["gateup"] + pb["down"] == weights + 2 * wl.T * wl.d  # gate/up also reads x
        assert pb["gateup"] - 2 * wl.T * wl.d == 2 * pb["down"]  # gate/up [2F x d] is twice down [d x F]
        assert pb["layer"] == bench.layer_bytes(wl, U, wl.T)


def test_layer_flops():
    # 2 T E d (router) + 2 T k 3 d F (three expert matrices per pair) + 2 T 3 d S (shared expert)
    assert bench.layer_flops(synth.WORKLOADS["decode"], 1) == 2 * 128 * 2880 + 2 * 4 * 3 * 2880 * 2880
    assert bench.layer_flops(synth.WORKLOADS["prefill"], 1024) == 204_598_149_120  # 204.6 GFLOP per layer
    wl = synth.WORKLOADS["small"]
    assert bench.layer_flops(wl, 8) == 2 * 8 * 256 * 2048 + 2 * 64 * 3 * 2048 * 512 + 2 * 8 * 3 * 2048 * 2048


def test_traffic_key_ignores_comments_and_follows_code(tmp_path, monkeypatch):
    """The key a committed DRAM-traffic figure is stored under: comment and whitespace edits keep it,
    any change to the code (a constant, a string literal) changes it."""
    src = 'int a = 4; // four\n/* block\n comment */ const char* s = "//kept";\n'
    assert bench.code_text(src) == 'int a = 4; const char* s = "//kept";'
    (tmp_path / "k.cu").write_text(src)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash(["k.cu"])
    (tmp_path / "k.cu").write_text(src.replace("// four", "// 4 steps").replace("\n/*", "\n\n  /*"))
    assert bench.kernel_source_hash(["k.cu"]) == h0
    (tmp_path / "k.cu").write_text(src.replace("a = 4", "a = 6"))
    assert bench.kernel_source_hash(["k.cu"]) != h0
    (tmp_path / "k.cu").write_text(src.replace('"//kept"', '"//kepT"'))
    assert bench.kernel_source_hash(["k.cu"]) != h0


def test_provenance_labels():
    """The line says which figures are measured, calculated or assumed."""
    pv = bench.provenance({"source": "measured"}, {"traffic": 54487808}, {"tflops": 4870.0})
    assert pv["roofline.peak"].startswith("MEASURED") and pv["roofline.traffic"].startswith("MEASURED")
    assert pv["mma_probe.fp4_peak_tflops"].startswith("CALCULATED")
    pv = bench.provenance({"source": "fallback"}, {"traffic": None}, None)
    assert pv["roofline.peak"].startswith("ASSUMED") and "none" in pv["roofline.traffic"]
    assert pv["mma_probe.tflops"] == "not run"
