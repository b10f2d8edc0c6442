"""The binding rejects, before the C call, what the C ABI cannot see.

The library receives raw pointers: a float32 tensor passed where bf16 is
expected, a transposed view, a tensor on the CPU or shapes that disagree
would be read as garbage.  The binding checks shape, dtype, contiguity and
device first and raises; none of these cases reaches the library, so they
run on the CPU.
"""
import pytest
import torch

from sink_aware_masked_gb300 import api

T, HQ, HKV, D = 16, 4, 2, 64


def _qkv(dtype=torch.bfloat16, t=T, hq=HQ, hkv=HKV, d=D):
    q = torch.zeros((t, hq, d), dtype=dtype)
    k = torch.zeros((t, hkv, d), dtype=dtype)
    v = torch.zeros((t, hkv, d), dtype=dtype)
    sink = torch.zeros((hq,), dtype=torch.float32)
    return q, k, v, sink


def test_forward_rejects_float32_inputs():
    q, k, v, sink = _qkv(torch.float32)
    with pytest.raises(TypeError, match="q has dtype"):
        api.sinkattn_fwd(q, k, v, sink, num_seqs=1)


def test_forward_rejects_wrong_sink_dtype():
    q, k, v, sink = _qkv()
    with pytest.raises(TypeError, match="sink has dtype"):
        api.sinkattn_fwd(q, k, v, sink.double(), num_seqs=1)


def test_forward_rejects_non_contiguous():
    q, k, v, sink = _qkv()
    qt = torch.zeros((HQ, T, D), dtype=torch.bfloat16).transpose(0, 1)
    assert qt.shape == q.shape and not qt.is_contiguous()
    with pytest.raises(ValueError, match="contiguous"):
        api.sinkattn_fwd(qt, k, v, sink, num_seqs=1)


def test_forward_rejects_cpu_tensors():
    q, k, v, sink = _qkv()
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.sinkattn_fwd(q, k, v, sink, num_seqs=1)


def test_forward_rejects_token_count_mismatch():
    q, _, _, sink = _qkv()
    _, k, v, _ = _qkv(t=T + 1)
    with pytest.raises(ValueError, match="tokens"):
        api.sinkattn_fwd(q, k, v, sink, num_seqs=1)


def test_rejects_head_dim_other_than_64():
    q, k, v, sink = _qkv(d=128)
    with pytest.raises(ValueError, match="head_dim"):
        api.sinkattn_fwd(q, k, v, sink, num_seqs=1)


def test_rejects_heads_not_a_multiple():
    q, k, v, sink = _qkv(hq=3, hkv=2)
    with pytest.raises(ValueError, match="multiple"):
        api.sinkattn_fwd(q, k, v, sink, num_seqs=1)


def test_rejects_v_shape_unlike_k():
    q, k, _, sink = _qkv()
    v = torch.zeros((T, HKV + 1, D), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="v has shape"):
        api.sinkattn_fwd(q, k, v, sink, num_seqs=1)


def test_backward_rejects_bad_lse_and_outputs():
    q, k, v, sink = _qkv()
    o = torch.zeros_like(q)
    lse_t = torch.zeros((T, HQ), dtype=torch.float32)  # token-major instead of [Hq, T]
    with pytest.raises(ValueError, match="lse has shape"):
        api.sinkattn_bwd(q, k, v, o, lse_t, o, sink, num_seqs=1)
    lse = torch.zeros((HQ, T), dtype=torch.float32)
    with pytest.raises(TypeError, match="dout has dtype"):
        api.sinkattn_bwd(q, k, v, o, lse, o.float(), sink, num_seqs=1)
    with pytest.raises(TypeError, match="dk has dtype"):
        api.sinkattn_bwd(q, k, v, o, lse, o, sink, dk=torch.zeros((T, HKV, D)), num_seqs=1)
    with pytest.raises(ValueError, match="dv has shape"):
        api.sinkattn_bwd(q, k, v, o, lse, o, sink, dv=torch.zeros_like(q), num_seqs=1)


def test_rejects_int64_offsets():
    q, k, v, sink = _qkv()
    cu = torch.tensor([0, 5, T], dtype=torch.int64)
    with pytest.raises(TypeError, match="cu_seqlens has dtype"):
        api.sinkattn_fwd(q, k, v, sink, cu_seqlens=cu, cu_seqlens_host=[0, 5, T])


def test_decode_rejects_float32_cache():
    q, _, _, sink = _qkv(t=2)
    _, k, v, _ = _qkv(torch.float32, t=T)
    with pytest.raises(TypeError, match="k has dtype"):
        api.sinkattn_decode_fwd(q, k, v, sink, q_per_seq=1, num_seqs=2)


def test_grpo_rejects_bool_mask_and_int64_offsets():
    logp = torch.zeros(10, dtype=torch.float32)
    rewards = torch.zeros(2, dtype=torch.float32)
    cu32 = torch.tensor([0, 4, 10], dtype=torch.int32)
    with pytest.raises(TypeError, match="mask has dtype"):
        api.grpo_loss(logp, logp, torch.zeros(10, dtype=torch.bool), rewards, cu32, [0, 4, 10], group_size=2)
    with pytest.raises(TypeError, match="cu_tokens has dtype"):
        api.grpo_loss(logp, logp, torch.zeros(10, dtype=torch.uint8), rewards, cu32.long(), [0, 4, 10],
                      group_size=2)
    with pytest.raises(ValueError, match="logp_old has shape"):
        api.grpo_loss(logp, logp[:9], torch.zeros(10, dtype=torch.uint8), rewards, cu32, [0, 4, 10], group_size=2)


def test_pack_rejects_float32():
    with pytest.raises(TypeError, match="padded has dtype"):
        api.sinkattn_pack(torch.zeros((2, 4, 2, 64)), torch.zeros(3, dtype=torch.int32), 5)
