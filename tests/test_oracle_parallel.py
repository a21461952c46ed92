"""The oracle's thread-parallel driver changes only the wall time: every token's
output, ids and gates are bit-identical to one single-threaded call, for any
thread count and for a token list that is not 0..T-1."""
import numpy as np
import pytest

import oracle
import synth


@pytest.mark.parametrize("threads", [1, 3, 8])
def test_parallel_driver_is_bit_identical(threads):
    wl = synth.WORKLOADS["tiny"].with_(T=13, E=16, k=3, shared_ffn=64)
    L = synth.gen_layer(wl, 2)
    tokens = [12, 0, 5, 5, 7, 1, 9]
    a = oracle.layer_tokens(wl.d, wl.ffn, wl.E, wl.k, wl.shared_ffn, L["x"], L["w_router"], L["bias"],
                            L["codes"], L["scales"], tokens=tokens)
    b = oracle.layer_tokens_parallel(wl.d, wl.ffn, wl.E, wl.k, wl.shared_ffn, L["x"], L["w_router"], L["bias"],
                                     L["codes"], L["scales"], tokens=tokens, threads=threads)
    assert b["threads"] == min(threads, len(tokens))
    for key in ("y", "ids", "gates"):
        assert np.array_equal(a[key], b[key]), key
    assert list(b["tokens"]) == tokens


def test_host_threads_is_positive():
    assert oracle.host_threads() >= 1
