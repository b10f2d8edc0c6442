"""Sequence-parallel (Ulysses) wrapper on the CPU: gloo ranks on 127.0.0.1.

The wrapper only moves tensors (all-to-all from sequence to head sharding
and back); the attention call on each rank is injected here as the float64
oracle, so the exchange is checked without a GPU.  Every rank's output rows,
log-sum-exp rows and gradients must equal the oracle run on the whole
packed stream in one process (the same per-head arithmetic, so to float64
rounding), and the sink gradients summed over the ranks must equal the
whole-stream dsink.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_fwd(q, k, v, sink, *, cu, window, prefix, causal, scale):
    o, lse = oracle.forward(q.double().numpy(), k.double().numpy(), v.double().numpy(), sink.double().numpy(), cu,
                            window, prefix, causal, scale)
    return torch.from_numpy(o), torch.from_numpy(lse)


def _oracle_bwd(q, k, v, o, lse, dout, sink, *, cu, window, prefix, causal, scale):
    r = oracle.forward_backward(q.double().numpy(), k.double().numpy(), v.double().numpy(), sink.double().numpy(),
                                dout.double().numpy(), cu, window, prefix, causal, scale)
    return tuple(torch.from_numpy(r[n]) for n in ("dq", "dk", "dv", "dsink"))


def _rank_main(rank, world, port, wl, shards, out):
    import torch.distributed as dist

    from sink_aware_masked_gb300 import ulysses

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = W.make_inputs(wl)
    t0 = int(sum(shards[:rank]))
    t1 = t0 + int(shards[rank])
    f = lambda t: t[t0:t1].double().contiguous()  # noqa: E731
    q, k, v, do = f(inp.q_bf16), f(inp.k_bf16), f(inp.v_bf16), f(inp.do_bf16)
    sink = inp.sink.double()
    problem = dict(cu=wl.cu_seqlens(), window=wl.window, prefix=wl.prefix, causal=wl.causal, scale=wl.scale)
    o, lse, saved = ulysses.ulysses_forward(q, k, v, sink, shard_tokens=shards, local_fwd=_oracle_fwd, **problem)
    dq, dk, dv, dsink = ulysses.ulysses_backward(saved, do, shard_tokens=shards, num_heads_q=wl.num_heads_q,
                                                 local_bwd=_oracle_bwd, **problem)
    out[rank] = {n: t.numpy() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv, dsink=dsink).items()}
    dist.destroy_process_group()


CASES = [
    (W.custom((100, 37, 200), 4, 2, window=20, prefix=3, seed=71, name="varlen_w20_p3"), (170, 167)),
    (W.custom((96,), 6, 3, seed=72, name="group2_three_ranks"), (40, 1, 55)),
    (W.custom((64, 64), 4, 4, window=0, seed=73, name="w0_mha"), (64, 64)),
]


@pytest.mark.parametrize("wl,shards", CASES, ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_ulysses_matches_whole_stream(wl, shards):
    world = len(shards)
    assert sum(shards) == wl.total_tokens
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, wl, shards, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    inp = W.make_inputs(wl)
    ref = oracle.forward_backward(inp.f64("q"), inp.f64("k"), inp.f64("v"), inp.f64("sink"), inp.f64("do"),
                                  wl.cu_seqlens(), wl.window, wl.prefix, wl.causal, wl.scale)
    t0 = 0
    dsink = np.zeros(wl.num_heads_q)
    for r in range(world):
        t1 = t0 + shards[r]
        got = out[r]
        for n in ("o", "dq", "dk", "dv"):
            np.testing.assert_allclose(got[n], ref[n][t0:t1], rtol=1e-12, atol=1e-12, err_msg=f"rank {r} {n}")
        np.testing.assert_allclose(got["lse"], ref["lse"][:, t0:t1], rtol=1e-12, atol=1e-12, err_msg=f"rank {r} lse")
        # Each rank fills only its own heads' sink gradient.
        hp = wl.num_heads_q // world
        own = np.zeros(wl.num_heads_q, bool)
        own[r * hp:(r + 1) * hp] = True
        assert np.all(got["dsink"][~own] == 0.0)
        dsink += got["dsink"]
        t0 = t1
    np.testing.assert_allclose(dsink, ref["dsink"], rtol=1e-12, atol=1e-12)


def test_ulysses_rejects_indivisible_heads():
    from sink_aware_masked_gb300 import ulysses

    q = torch.zeros(10, 4, 64)
    k = torch.zeros(10, 1, 64)
    with pytest.raises(ValueError, match="divisible"):
        ulysses._check(q, k, torch.zeros(4), [10, 10], 2, 0)
    with pytest.raises(ValueError, match="shard_tokens"):
        ulysses._check(q, torch.zeros(10, 2, 64), torch.zeros(4), [11, 9], 2, 0)
