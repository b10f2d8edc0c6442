"""Sequence-parallel wrapper with the library on the GPU (needs a GB300).

Two gloo ranks share cuda:0, each holding half of a packed token stream;
through the autograd wrapper each runs the library's forward and backward
for its heads over the whole stream.  Their rows are compared with the
float64 oracle on the whole stream (the parity tolerances), and O and lse
with one library call over the whole stream (the same per-head arithmetic:
bitwise equal).  The ranks' kernels never wait on each other.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import workloads as W
from tests import parity_util as pu

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem(wl, dev):
    cu = wl.cu_seqlens()
    return dict(cu_seqlens=torch.tensor(cu, dtype=torch.int32, device=dev), cu_seqlens_host=[int(x) for x in cu],
                max_seqlen=wl.max_seqlen, window=wl.window, prefix=wl.prefix, causal=wl.causal, scale=wl.scale)


def _rank_main(rank, world, port, wl, shards, out):
    import torch.distributed as dist

    from sink_aware_masked_gb300 import ulysses

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dev = torch.device("cuda:0")
    inp = W.make_inputs(wl)
    t0 = int(sum(shards[:rank]))
    t1 = t0 + int(shards[rank])
    q, k, v = (t[t0:t1].contiguous().to(dev).requires_grad_(True) for t in (inp.q_bf16, inp.k_bf16, inp.v_bf16))
    sink = inp.sink.to(dev).requires_grad_(True)
    o = ulysses.ulysses_sink_attention(q, k, v, sink, shard_tokens=shards, **_problem(wl, dev))
    o.backward(inp.do_bf16[t0:t1].to(dev))
    torch.cuda.synchronize()
    import sink_aware_masked_gb300 as sa

    out[rank] = dict(o=o.detach().float().cpu().numpy(), dq=q.grad.float().cpu().numpy(),
                     dk=k.grad.float().cpu().numpy(), dv=v.grad.float().cpu().numpy(),
                     dsink=sink.grad.float().cpu().numpy(), status=sa.sinkattn_get_device_status())
    dist.destroy_process_group()


def test_two_ranks_on_one_gpu_match_oracle_and_single_call():
    import sink_aware_masked_gb300 as sa
    from sink_aware_masked_gb300 import build

    build.build()
    wl = W.custom((300, 77, 500), 8, 2, window=64, prefix=4, seed=74, sink_dist="uniform2", name="sp2")
    shards = (450, 427)
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, wl, shards, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=600)
        assert p.exitcode == 0
    assert out[0]["status"] == 0 and out[1]["status"] == 0
    got = {n: np.concatenate([out[0][n], out[1][n]], 0) for n in ("o", "dq", "dk", "dv")}
    got["dsink"] = out[0]["dsink"] + out[1]["dsink"]
    inp = W.make_inputs(wl)
    ref = oracle.forward_backward(inp.f64("q"), inp.f64("k"), inp.f64("v"), inp.f64("sink"), inp.f64("do"),
                                  wl.cu_seqlens(), wl.window, wl.prefix, wl.causal, wl.scale)
    errs = {"o": pu.max_abs(got["o"], ref["o"]), "dq": pu.rel_l2(got["dq"], ref["dq"]),
            "dk": pu.rel_l2(got["dk"], ref["dk"]), "dv": pu.rel_l2(got["dv"], ref["dv"]),
            "dsink": pu.rel_l2(got["dsink"], ref["dsink"])}
    pu.assert_within(errs, "two-rank sequence parallel")
    # One library call over the whole stream: the same per-head forward.
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in (inp.q_bf16, inp.k_bf16, inp.v_bf16))
    o, _ = sa.sinkattn_fwd(q, k, v, inp.sink.to(dev), **_problem(wl, dev))
    assert np.array_equal(o.float().cpu().numpy(), got["o"])
