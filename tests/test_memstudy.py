"""The peak-memory study's eager baseline computes the same layer as the oracle,
and on the GPU the library's peak stays below the eager path's."""
import numpy as np
import pytest
import torch

import oracle.sinkattn_ref as ref
from studies import memstudy


@pytest.mark.parametrize("window,prefix", [(-1, 0), (5, 3)])
def test_eager_baseline_matches_oracle(window, prefix):
    B, S, hq, hkv, D = 2, 37, 4, 2, 64
    g = torch.Generator().manual_seed(11)
    q = torch.randn(B, S, hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, S, hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, S, hkv, D, generator=g).to(torch.bfloat16)
    dout = torch.randn(B, S, hq, D, generator=g).to(torch.bfloat16)
    sink = torch.randn(hq, generator=g)
    o, dq, dk, dv, dsink = memstudy.eager_reference_layer(q, k, v, sink, dout, window=window, prefix=prefix)
    f64 = lambda t: t.double().reshape(B * S, t.shape[2], D).numpy()  # noqa: E731
    cu = np.arange(B + 1, dtype=np.int64) * S
    want = ref.forward_backward(f64(q), f64(k), f64(v), sink.double().numpy(), f64(dout), cu,
                                window=window, prefix=prefix)
    for name, got in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(got.double().reshape(B * S, -1, D).numpy(), want[name], atol=2e-4, rtol=2e-4,
                                   err_msg=name)
    np.testing.assert_allclose(dsink.double().numpy(), want["dsink"], atol=2e-4, rtol=2e-4)


def test_eager_scores_bytes():
    assert memstudy.eager_scores_bytes(1, 8192, 64) == 4 * 64 * 8192 * 8193


@pytest.mark.gpu
def test_library_peak_below_eager():
    r = memstudy.measure(1024, hq=64, hkv=8)
    assert r["eager_peak_bytes"] is not None
    assert r["library_peak_bytes"] < r["eager_peak_bytes"]
    assert r["max_abs_diff_o"] < 1e-2
    assert r["rel_diff_dsink"] < 2e-2
