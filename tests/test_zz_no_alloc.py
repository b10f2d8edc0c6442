"""The no-allocation backward entry point against the regular one (GPU).

sinkattn_bwd_noalloc serves callers that cannot allocate device memory: it
runs the same backward on a workspace compiled into the library.  This test
calls both entry points through the C ABI on the same inputs, twice in a
row (the second call reuses the static workspace as the first left it), and
checks that the results agree within the parity tolerances used elsewhere
(dQ is summed with atomics, so its bits may differ; the rest must match
exactly).  It lives in its own file, named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _rel_l2(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def test_noalloc_backward_matches_regular_backward():
    import workloads as W
    from sink_aware_masked_gb300 import _lib, api, build

    build.build()
    lib = _lib.load()
    wl = W.custom((700, 300), 8, 2, window=100, prefix=3, seed=77, sink_dist="uniform2", name="noalloc")
    inp = W.make_inputs(wl)
    q, k, v, do = (t.to(DEV) for t in (inp.q_bf16, inp.k_bf16, inp.v_bf16, inp.do_bf16))
    sink = inp.sink.to(DEV)
    cu = wl.cu_seqlens()
    kw = dict(cu_seqlens=torch.tensor(cu, dtype=torch.int32, device=DEV), cu_seqlens_host=[int(x) for x in cu],
              max_seqlen=wl.max_seqlen, window=wl.window, prefix=wl.prefix, causal=wl.causal, scale=wl.scale)
    o, lse = api.sinkattn_fwd(q, k, v, sink, **kw)
    ref = api.sinkattn_bwd(q, k, v, o, lse, do, sink, **kw)
    torch.cuda.synchronize()

    pr, keep = api.make_problem(q, k, **kw)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        dq, dk, dv = torch.full_like(q, 7.0), torch.full_like(k, 7.0), torch.full_like(v, 7.0)
        dsink = torch.full_like(sink, 7.0)
        st = lib.sinkattn_bwd_noalloc(ctypes.byref(pr), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                      _ptr(sink), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dsink), stream)
        assert st == 0, _lib.STATUS.get(st, st)
        torch.cuda.synchronize()
        assert lib.sinkattn_get_device_status(stream) == 0
        for got, want, name in ((dk, ref[1], "dk"), (dv, ref[2], "dv"), (dsink, ref[3], "dsink")):
            assert torch.equal(got, want), (call, name)
        assert _rel_l2(dq, ref[0]) < 1e-3, call


def test_noalloc_rejects_problems_beyond_its_workspace():
    from sink_aware_masked_gb300 import _lib, build

    build.build()
    lib = _lib.load()
    # 16384 tokens x 64 heads needs ~277 MB of workspace, far beyond 32 MiB.
    pr = _lib.Problem(num_seqs=1, seqlen=16384, cu_seqlens=None, cu_seqlens_host=None, total_tokens=16384,
                      num_heads_q=64, num_heads_kv=8, head_dim=64, window=-1, prefix=0, causal=1, scale=0.125)
    fake = ctypes.c_void_p(0x10000)
    st = lib.sinkattn_bwd_noalloc(ctypes.byref(pr), *([fake] * 11), None)
    assert st == 4  # SINKATTN_ERR_WORKSPACE, nothing launched
