"""Guard regions around every output, and untouched inputs (needs a GB300).

The oracle comparison sees only the elements it compares: a stray write just
past an output (a tile store past a sequence end, a ragged-tail conversion,
a split-tile accumulator overrun) would go unnoticed.  Here every output and
the workspace live inside a larger buffer whose bytes outside the output are
a sentinel; after the call the sentinels must be intact, and the inputs must
equal their copies taken before the call.  This stands in for a
memory-checking tool, which this pool does not offer.

A separate test feeds the oracle the unrounded float32 draws of the tiny
workload (the GPU gets them rounded to bf16) and reports the errors; that
comparison is informative only (bf16 rounding of q and k alone moves the
scores by about 3e-3), so it is checked against loose bounds.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
PAD = 4096  # bytes of sentinel on each side (a multiple of 16 keeps every view 16-byte aligned)
SENTINEL = 0xA5


@pytest.fixture(scope="module", autouse=True)
def built():
    from sink_aware_masked_gb300 import build

    build.build()


class Guarded:
    """A tensor of ``shape``/``dtype`` inside a sentinel-filled byte buffer."""

    def __init__(self, shape, dtype, nbytes=None):
        elt = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape)) if len(shape) else 1
        self.nbytes = n * elt if nbytes is None else int(nbytes)
        self.buf = torch.full((PAD + self.nbytes + PAD,), SENTINEL, dtype=torch.uint8, device=DEV)
        self.t = self.buf[PAD:PAD + self.nbytes].view(dtype)
        if nbytes is None:
            self.t = self.t.view(shape)

    def check(self, name):
        torch.cuda.synchronize()
        head = self.buf[:PAD]
        tail = self.buf[PAD + self.nbytes:]
        bad_h = int((head != SENTINEL).sum())
        bad_t = int((tail != SENTINEL).sum())
        assert bad_h == 0 and bad_t == 0, f"{name}: {bad_h} bytes before and {bad_t} bytes after were written"


def _problem(wl):
    kw = dict(window=wl.window, prefix=wl.prefix, causal=wl.causal, scale=wl.scale)
    if wl.uniform:
        kw["num_seqs"] = wl.num_seqs
    else:
        cu = wl.cu_seqlens()
        kw.update(cu_seqlens=torch.tensor(cu, dtype=torch.int32, device=DEV), cu_seqlens_host=[int(x) for x in cu],
                  max_seqlen=wl.max_seqlen)
    return kw


ATTN_CASES = [
    W.custom((1, 130, 257, 64, 0, 129), 8, 2, window=128, prefix=4, seed=17, name="ragged_varlen_w128_p4"),
    W.custom((1, 130, 257, 64, 0, 129), 8, 2, seed=16, name="ragged_varlen_causal"),
    W.custom((384,), 4, 2, window=16, prefix=200, seed=20, name="split_prefix_tiles"),
    W.custom((2000,), 8, 2, seed=23, name="split_causal_tiles"),
    W.custom((300, 77), 6, 2, window=40, prefix=3, seed=24, name="group3"),
    W.custom((1,), 2, 1, seed=18, name="one_token"),
]


@pytest.mark.parametrize("wl", ATTN_CASES, ids=lambda w: w.name)
def test_attention_writes_stay_inside_outputs(wl):
    import sink_aware_masked_gb300 as sa

    inp = W.make_inputs(wl)
    q, k, v, do = (t.to(DEV) for t in (inp.q_bf16, inp.k_bf16, inp.v_bf16, inp.do_bf16))
    sink = inp.sink.to(DEV)
    kw = _problem(wl)
    T, hq, hkv = wl.total_tokens, wl.num_heads_q, wl.num_heads_kv
    ins = {n: t.clone() for n, t in dict(q=q, k=k, v=v, do=do, sink=sink).items()}
    o = Guarded((T, hq, 64), torch.bfloat16)
    lse = Guarded((hq, T), torch.float32)
    sa.sinkattn_fwd(q, k, v, sink, o=o.t, lse=lse.t, **kw)
    o.check("o")
    lse.check("lse")
    o_in, lse_in = o.t.clone(), lse.t.clone()
    dq = Guarded((T, hq, 64), torch.bfloat16)
    dk = Guarded((T, hkv, 64), torch.bfloat16)
    dv = Guarded((T, hkv, 64), torch.bfloat16)
    dsink = Guarded((hq,), torch.float32)
    ws_bytes = sa.bwd_workspace_bytes(q, k, **kw)
    ws = Guarded((ws_bytes,), torch.uint8)  # its inside holds the sentinel too: nothing needs to be zero
    first = None
    for rep in range(2):  # the second call reuses the workspace as the first left it
        sa.sinkattn_bwd(q, k, v, o.t, lse.t, do, sink, dq=dq.t, dk=dk.t, dv=dv.t, dsink=dsink.t, workspace=ws.t,
                        **kw)
        assert sa.sinkattn_get_device_status() == 0
        for name, g in (("dq", dq), ("dk", dk), ("dv", dv), ("dsink", dsink), ("workspace", ws)):
            g.check(f"{name} (call {rep + 1})")
        if first is None:
            first = [t.clone() for t in (dk.t, dv.t, dsink.t)]
        else:
            for a, b in zip(first, (dk.t, dv.t, dsink.t)):
                assert torch.equal(a, b), "dk, dv and dsink are reproducible"
    ref = pu.oracle_heads(inp, wl, list(range(hq)), parallel=False)
    pu.assert_within(pu.errors(dict(o=o.t, lse=lse.t, dq=dq.t, dk=dk.t, dv=dv.t, dsink=dsink.t), ref,
                               list(range(hq)), list(range(hkv))), wl.name)
    for name, t in ins.items():
        assert torch.equal(t, dict(q=q, k=k, v=v, do=do, sink=sink)[name]), f"input {name} was modified"
    assert torch.equal(o_in, o.t) and torch.equal(lse_in, lse.t), "o or lse was modified by the backward"
    for t in (o.t, dq.t, dk.t, dv.t):
        assert bool(torch.isfinite(t.float()).all())


@pytest.mark.parametrize("lens,hq,hkv,n,w,p", [((300, 1, 129, 2000), 16, 2, 1, -1, 0),
                                               ((700, 2048), 16, 2, 4, 128, 4),
                                               ((3000,), 12, 4, 3, 10, 2000),
                                               ((900, 129), 24, 1, 4, -1, 0)])
def test_decode_writes_stay_inside_outputs(lens, hq, hkv, n, w, p):
    import sink_aware_masked_gb300 as sa

    wl = W.custom(lens, hq, hkv, window=w, prefix=p, seed=61, sink_dist="uniform2")
    inp = W.make_decode_inputs(wl, n)
    q, k, v, sink = (t.to(DEV) for t in (inp.q_bf16, inp.k_bf16, inp.v_bf16, inp.sink))
    kw = _problem(wl)
    R = wl.num_seqs * n
    o = Guarded((R, hq, 64), torch.bfloat16)
    lse = Guarded((hq, R), torch.float32)
    ws_bytes = sa.decode_workspace_bytes(q, k, q_per_seq=n, **kw)
    ws = Guarded((ws_bytes,), torch.uint8)
    ws.t.zero_()  # the chunk counters start at zero (each call leaves them so)
    for rep in range(2):
        sa.sinkattn_decode_fwd(q, k, v, sink, q_per_seq=n, o=o.t, lse=lse.t, workspace=ws.t, **kw)
        assert sa.sinkattn_get_device_status() == 0
        for name, g in (("o", o), ("lse", lse), ("workspace", ws)):
            g.check(f"{name} (call {rep + 1})")
    assert bool(torch.isfinite(o.t.float()).all())


def test_grpo_writes_stay_inside_outputs():
    import sink_aware_masked_gb300 as sa

    wl = W.GrpoWorkload("guard", prompts=5, group_size=3, len_lo=17, len_hi=700, seed=62)
    inp = W.make_grpo_inputs(wl)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    T, R = int(inp.cu_tokens[-1]), len(inp.cu_tokens) - 1
    dlogp = Guarded((T,), torch.float32)
    adv = Guarded((R,), torch.float32)
    stats = Guarded((4,), torch.float32)
    cu_host = [int(x) for x in inp.cu_tokens]
    ws = Guarded((sa.grpo_workspace_bytes(t(inp.cu_tokens), cu_host, group_size=wl.group_size),), torch.uint8)
    ws.t.zero_()
    for rep in range(2):
        sa.grpo_loss(t(inp.logp), t(inp.logp_old), t(inp.mask), t(inp.rewards), t(inp.cu_tokens), cu_host,
                     group_size=wl.group_size, clip_eps=wl.clip_eps, adv_eps=wl.adv_eps, kl_beta=wl.kl_beta,
                     logp_ref=t(inp.logp_ref), dlogp=dlogp.t, workspace=ws.t, stats=stats.t, advantages=adv.t)
        assert sa.sinkattn_get_device_status() == 0
        for name, g in (("dlogp", dlogp), ("advantages", adv), ("stats", stats), ("workspace", ws)):
            g.check(f"{name} (call {rep + 1})")


def test_float32_oracle_inputs_reported():
    """The tiny workload's literal comparison: the oracle on the unrounded
    float32 draws, the GPU on their bf16 roundings.  Reported, not graded."""
    import sink_aware_masked_gb300 as sa

    wl = W.WORKLOADS["tiny_s128_w32_p4"]
    inp = W.make_inputs(wl, keep_f32=True)
    q, k, v, do = (t.to(DEV) for t in (inp.q_bf16, inp.k_bf16, inp.v_bf16, inp.do_bf16))
    sink = inp.sink.to(DEV)
    kw = _problem(wl)
    o, lse = sa.sinkattn_fwd(q, k, v, sink, **kw)
    dq, dk, dv, dsink = sa.sinkattn_bwd(q, k, v, o, lse, do, sink, **kw)
    f64 = lambda x: x.to(torch.float64).numpy()  # noqa: E731
    ref = oracle.forward_backward(f64(inp.q_f32), f64(inp.k_f32), f64(inp.v_f32), f64(inp.sink), f64(inp.do_f32),
                                  wl.cu_seqlens(), wl.window, wl.prefix, wl.causal, wl.scale)
    g = lambda x: x.detach().double().cpu().numpy()  # noqa: E731
    errs = {"o": pu.max_abs(g(o), ref["o"]), "lse": pu.max_abs(g(lse), ref["lse"]),
            "dq": pu.rel_l2(g(dq), ref["dq"]), "dk": pu.rel_l2(g(dk), ref["dk"]),
            "dv": pu.rel_l2(g(dv), ref["dv"]), "dsink": pu.rel_l2(g(dsink), ref["dsink"])}
    print("float32-input comparison (unrated):", errs)
    loose = {"o": 3e-2, "lse": 2e-2, "dq": 5e-2, "dk": 5e-2, "dv": 5e-2, "dsink": 5e-2}
    assert all(errs[n] <= loose[n] for n in loose), errs
