"""Expert parallelism, on the oracle (CPU): the layer splits over contiguous
expert shards, one per rank, with routing over all experts on every rank.

Each rank holds experts [r E / G, (r+1) E / G) (the expert-major layout keeps
a shard one contiguous byte range) and rank 0 also the shared expert; the
partial outputs, added in rank order, are the layer output. Checked in one
process for G = 1..4 and across two gloo ranks that exchange their partials
with all_gather and add them in rank order.
"""
import os
import socket

import numpy as np
import pytest

import oracle
import synth

WL = synth.WORKLOADS["tiny"].with_(name="tiny_shared", T=7, E=12, k=3, shared_ffn=64, zipf_bias=1.1)


def _shard(E: int, G: int, r: int):
    return r * E // G, (r + 1) * E // G


def _layer(wl=WL, layer=2):
    L = synth.gen_layer(wl, layer)
    w_sg = synth.gen_shared_gate(wl.seed(layer), wl.d)
    full = oracle.layer_tokens(wl.d, wl.ffn, wl.E, wl.k, wl.shared_ffn, L["x"], L["w_router"], L["bias"],
                               L["codes"], L["scales"], w_shared_gate=w_sg)
    return L, w_sg, full


def _partial(L, w_sg, r, G, wl=WL):
    e0, e1 = _shard(wl.E, G, r)
    return oracle.layer_tokens_shard(wl.d, wl.ffn, wl.E, wl.k, wl.shared_ffn, L["x"], L["w_router"], L["bias"],
                                     L["codes"], L["scales"], e0, e1, r == 0, w_shared_gate=w_sg)


@pytest.mark.parametrize("G", [1, 2, 3, 4])
def test_shards_add_up_to_the_layer(G):
    L, w_sg, full = _layer()
    parts = [_partial(L, w_sg, r, G) for r in range(G)]
    total = np.zeros_like(parts[0])
    for p in parts:  # rank order
        total += p
    if G == 1:
        assert np.array_equal(total, full["y"])  # one shard is the layer, summed in the same order
    np.testing.assert_allclose(total, full["y"], rtol=0, atol=1e-13 * np.abs(full["y"]).max())
    # every (token, slot) pair lands on exactly one shard
    owners = np.zeros_like(full["ids"])
    for r in range(G):
        e0, e1 = _shard(WL.E, G, r)
        owners += (full["ids"] >= e0) & (full["ids"] < e1)
    assert np.all(owners == 1)


def test_a_shard_without_routed_pairs_adds_nothing():
    L, w_sg, full = _layer()
    unused = sorted(set(range(WL.E)) - set(np.unique(full["ids"]).tolist()))
    if not unused:
        pytest.skip("every expert is routed to in this layer")
    e = unused[0]
    y = oracle.layer_tokens_shard(WL.d, WL.ffn, WL.E, WL.k, WL.shared_ffn, L["x"], L["w_router"], L["bias"],
                                  L["codes"], L["scales"], e, e + 1, False)
    assert np.all(y == 0.0)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, ws: int, port: int, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        L, w_sg, full = _layer()
        mine = torch.from_numpy(_partial(L, w_sg, rank, ws))
        parts = [torch.empty_like(mine) for _ in range(ws)]
        dist.all_gather(parts, mine)
        total = torch.zeros_like(mine)
        for p in parts:  # rank order, the same on every rank
            total += p
        out[rank] = (total.numpy().tobytes(), float(np.abs(total.numpy() - full["y"]).max()),
                     float(np.abs(full["y"]).max()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_exchange_partials_in_rank_order():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ws = 2
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank, args=(ws, port, out), nprocs=ws, join=True, start_method="spawn")
    assert out[0][0] == out[1][0]  # both ranks hold the same bits
    assert out[0][1] <= 1e-13 * out[0][2]
