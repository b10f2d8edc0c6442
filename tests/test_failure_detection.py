"""Failure detection without a GPU fault.

The bounded mbarrier wait shared by the tcgen05 kernels is made to run out
on purpose (a barrier nothing arrives on, short limit): the device status
word must report the timeout once, and the context must stay usable.  The
host-side half (argument checks) is covered by test_abi.py."""
import ctypes

import pytest
import torch


@pytest.mark.gpu
def test_bounded_wait_reports_timeout_and_context_survives():
    import sink_aware_masked_gb300 as sa
    from sink_aware_masked_gb300 import _lib, build

    build.build()
    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.sinkattn_get_device_status(stream) == 0
    assert lib.sinkattn_selftest_wait_timeout(2_000_000, stream) == 0  # about 1 ms of SM cycles
    assert lib.sinkattn_get_device_status(stream) == 6  # SINKATTN_ERR_TIMEOUT, reported once
    assert lib.sinkattn_get_device_status(stream) == 0  # cleared
    # The context still works: a normal forward/backward afterwards is clean.
    q = torch.randn(256, 2, 64, device="cuda").to(torch.bfloat16)
    k = torch.randn(256, 1, 64, device="cuda").to(torch.bfloat16)
    sink = torch.zeros(2, device="cuda")
    o, lse = sa.sinkattn_fwd(q, k, k, sink, num_seqs=1)
    sa.sinkattn_bwd(q, k, k, o, lse, q, sink, num_seqs=1)
    torch.cuda.synchronize()
    assert lib.sinkattn_get_device_status(stream) == 0
    assert torch.isfinite(o.float()).all()


def test_selftest_rejects_bad_limits():
    from sink_aware_masked_gb300 import _lib, build

    build.build()
    lib = _lib.load()
    assert lib.sinkattn_selftest_wait_timeout(0, None) == 1
    assert lib.sinkattn_selftest_wait_timeout(3_000_000_000, None) == 1
