"""bench.py host logic on the CPU: FLOP/byte accounting against the oracle's
mask enumeration, and the multi-rank path (barrier + max-over-ranks) with two
gloo ranks on 127.0.0.1."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
import workloads as W


@pytest.mark.parametrize("wl", [
    W.WORKLOADS["tiny_s128_w32_p4"],
    W.custom((300, 17, 129), 4, 2, window=37, prefix=5),
    W.custom((190,), 4, 2, window=50, prefix=70, causal=False),
    W.custom((64,), 2, 1),
], ids=lambda w: w.name + str(w.seqlens))
def test_visible_pairs_match_oracle(wl):
    assert bench.visible_pairs(wl) == oracle.unmasked_pairs(wl.seqlens, wl.num_heads_q, wl.window, wl.prefix,
                                                            wl.causal)


def test_workload_pair_counts():
    want = {"tiny_s128_w32_p4": 8140, "causal_gqa_s4096": 537001984, "window128_gqa_s4096": 33288192,
            "causal_gqa_b2_s8192": 4295491584, "window128_prefix4_gqa_b2_s8192": 138337024,
            "varlen8_window128": 258421056, "varlen8_causal": 5224652736}
    for name, n in want.items():
        assert bench.visible_pairs(W.WORKLOADS[name]) == n, name


def test_algorithmic_bytes_per_token():
    wl = W.WORKLOADS["causal_gqa_b2_s8192"]
    fwd, bwd = bench.algorithmic_bytes(wl)
    assert fwd == 18688 * wl.total_tokens and bwd == 37120 * wl.total_tokens


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    got = bench.reduce_max([1.0 + rank, 10.0 - rank], world, torch.device("cpu"))
    out[rank] = got
    dist.destroy_process_group()


def test_two_rank_max_reduction():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        assert out[r] == [2.0, 10.0]


@pytest.mark.parametrize("lens,n,window,prefix", [((300, 1, 129), 1, -1, 0), ((700, 2048), 4, 128, 4),
                                                  ((513,), 8, 64, 600), ((90,), 3, 0, 0)])
def test_decode_visible_keys_match_mask_enumeration(lens, n, window, prefix):
    import oracle

    wl = W.custom(lens, 4, 2, window=window, prefix=prefix)
    want = 0
    for L in lens:
        m = oracle.visible(np.arange(L - n, L), np.arange(L), window, prefix, True)
        want += int(np.count_nonzero(m.any(axis=0)))
    assert bench.decode_visible_keys(wl, n) == want
