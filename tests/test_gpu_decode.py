"""Decode forward (last rows of each sequence against its key/value history):
CUDA path vs the CPU float64 oracle, element by element (needs a GB300)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import parity_util as pu

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    from sink_aware_masked_gb300 import build

    build.build()


def run_decode(wl, n, sink=None, key_gain=None):
    import sink_aware_masked_gb300 as sa

    inp = W.make_decode_inputs(wl, n)
    if key_gain is not None:  # per-token factor on the keys (bf16-exact powers of two)
        inp.k_bf16 = (inp.k_bf16.float() * key_gain[:, None, None]).to(torch.bfloat16)
    q = inp.q_bf16
    s = inp.sink if sink is None else sink
    kw = dict(window=wl.window, prefix=wl.prefix, causal=wl.causal, scale=wl.scale)
    if wl.uniform:
        kw["num_seqs"] = wl.num_seqs
    else:
        cu = wl.cu_seqlens()
        kw.update(cu_seqlens=torch.tensor(cu, dtype=torch.int32, device=DEV), cu_seqlens_host=[int(x) for x in cu],
                  max_seqlen=wl.max_seqlen)
    o, lse = sa.sinkattn_decode_fwd(q.to(DEV), inp.k_bf16.to(DEV), inp.v_bf16.to(DEV), s.to(DEV), q_per_seq=n, **kw)
    assert sa.sinkattn_get_device_status() == 0
    ref_o, ref_lse = oracle.decode_forward(q.to(torch.float64).numpy(), inp.f64("k"), inp.f64("v"),
                                           s.to(torch.float64).numpy(), wl.cu_seqlens(), n, wl.window, wl.prefix,
                                           wl.causal, wl.scale)
    return o.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse


CASES = [
    # seqlens, hq, hkv, rows per sequence, window, prefix, seed
    ((1000, 1000), 16, 2, 1, -1, 0, 91),           # ragged last tile, 8 rows per kv head
    ((300, 1, 129, 2000), 16, 2, 1, -1, 0, 92),     # packed, a one-token sequence, a 129-token one
    ((700, 2048), 16, 2, 4, 128, 4, 93),            # 32 rows, window and prefix
    ((513,), 16, 2, 8, 64, 0, 94),                  # 64 rows
    ((900, 129), 16, 2, 16, -1, 7, 95),             # 128 rows (the largest supported)
    ((4096, 4096, 4096), 64, 8, 2, -1, 0, 97),      # 64/8 heads
    ((32768,), 64, 8, 1, -1, 0, 96),                # long history split over many chunks
    ((3000,), 12, 4, 3, 10, 2000, 98),              # group of 3, prefix wider than the window
    ((1500, 700), 17, 1, 1, -1, 0, 86),             # 17 rows: tensor-core kernel, 15 padding columns
    ((2100, 333), 12, 1, 4, 200, 3, 87),            # 48 rows padded to 64, window and prefix
    ((1800, 97), 24, 1, 4, -1, 0, 88),              # 96 rows padded to 128, a sequence shorter than a tile
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"L{'-'.join(map(str, c[0]))}_h{c[1]}x{c[2]}_n{c[3]}_w{c[4]}")
def test_decode_matches_oracle(case):
    lens, hq, hkv, n, w, p, seed = case
    wl = W.custom(lens, hq, hkv, window=w, prefix=p, seed=seed, sink_dist="uniform2")
    o, lse, ref_o, ref_lse = run_decode(wl, n)
    assert pu.max_abs(o, ref_o) <= pu.TOL["o"], pu.max_abs(o, ref_o)
    assert pu.max_abs(lse, ref_lse) <= pu.TOL["lse"], pu.max_abs(lse, ref_lse)


def test_decode_sink_limits():
    wl = W.custom((600, 257), 16, 2, seed=99)
    hq = wl.num_heads_q
    o, lse, ref_o, ref_lse = run_decode(wl, 2, sink=torch.full((hq,), float("inf")))
    assert np.all(o == 0.0) and pu.max_abs(lse, ref_lse) <= pu.TOL["lse"]
    o, lse, ref_o, ref_lse = run_decode(wl, 2, sink=torch.full((hq,), float("-inf")))
    assert pu.max_abs(o, ref_o) <= pu.TOL["o"] and pu.max_abs(lse, ref_lse) <= pu.TOL["lse"]


@pytest.mark.parametrize("n,hq", [(4, 16), (8, 16), (16, 16), (2, 64)])
def test_decode_growing_scores(n, hq):
    """Keys whose scale doubles every 300 tokens: late tiles score far above
    the early ones, so the running references move in the middle of a chunk
    (the rescale of the accumulated output and row sums), not just on the
    first tile."""
    wl = W.custom((2000, 3100), hq, 8 if hq == 64 else 2, seed=90 + n, sink_dist="uniform2")
    gain = torch.tensor([2.0 ** min((t - 2000 if t >= 2000 else t) // 300, 5) for t in range(5100)])
    o, lse, ref_o, ref_lse = run_decode(wl, n, key_gain=gain)
    assert pu.max_abs(o, ref_o) <= pu.TOL["o"], pu.max_abs(o, ref_o)
    assert pu.max_abs(lse, ref_lse) <= pu.TOL["lse"], pu.max_abs(lse, ref_lse)


def test_decode_growing_scores_16_rows_tensor_core():
    """8 rows per kv head on a step long enough (1032 key tiles per kv head)
    for the tensor-core kernel's 16-column form; the key scale grows 2x every
    300 tokens and restarts every 1800, so references move inside chunks."""
    wl = W.custom((70000, 62000), 16, 2, seed=85, sink_dist="uniform2")
    starts = [0, 70000]
    gain = torch.tensor([2.0 ** (((t - (starts[1] if t >= starts[1] else 0)) // 300) % 6) for t in range(132000)])
    o, lse, ref_o, ref_lse = run_decode(wl, 1, key_gain=gain)
    assert pu.max_abs(o, ref_o) <= pu.TOL["o"], pu.max_abs(o, ref_o)
    assert pu.max_abs(lse, ref_lse) <= pu.TOL["lse"], pu.max_abs(lse, ref_lse)


# Row counts R = group x n across every kernel width (16, 32, 64, 128
# columns, one or two softmax warpgroups) and both routings: few key tiles
# per kv head (warp-MMA kernel for R <= 16) and >= 128 (tensor cores), with
# padding rows, windows, prefixes and causal bounds inside the last tile.
SWEEP = [
    # seqlens, hq, hkv, rows per sequence, window, prefix, seed
    ((5000, 4000, 3000, 4500), 8, 8, 1, -1, 0, 101),       # R = 1, 129 tiles per kv head: tensor cores, 16 columns
    ((700, 300), 8, 8, 3, 40, 2, 102),                     # R = 3, warp-MMA kernel
    ((6000, 5000, 5500), 18, 2, 1, 300, 5, 103),           # R = 9, tensor cores (windowed, but 3 long sequences)
    ((9000, 8000), 12, 1, 2, -1, 0, 104),                  # R = 24: 32 columns, two softmax warpgroups
    ((2500, 129, 1000), 31, 1, 1, 64, 7, 105),             # R = 31: one padding row
    ((3000, 2000), 33, 1, 1, -1, 0, 106),                  # R = 33: 64 columns, 31 padding
    ((1500, 400), 8, 1, 8, 100, 0, 107),                   # R = 64, window
    ((2200, 640), 13, 1, 5, -1, 3, 108),                   # R = 65: 128 columns, group 13
    ((1300, 900), 127, 1, 1, -1, 0, 109),                  # R = 127
    ((777,), 16, 2, 16, 50, 20, 110),                      # R = 128, window and prefix, one sequence
    (tuple(W.random_lengths(300, 4, 900, 111)), 16, 2, 4, -1, 0, 112),  # 300 short sequences: > 256 work items
]


@pytest.mark.parametrize("case", SWEEP, ids=lambda c: f"R{(c[1] // c[2]) * c[3]}_L{'-'.join(map(str, c[0]))}")
def test_decode_row_sweep(case):
    lens, hq, hkv, n, w, p, seed = case
    wl = W.custom(lens, hq, hkv, window=w, prefix=p, seed=seed, sink_dist="uniform2")
    o, lse, ref_o, ref_lse = run_decode(wl, n)
    assert pu.max_abs(o, ref_o) <= pu.TOL["o"], pu.max_abs(o, ref_o)
    assert pu.max_abs(lse, ref_lse) <= pu.TOL["lse"], pu.max_abs(lse, ref_lse)


@pytest.mark.parametrize("name", sorted(W.DECODE_WORKLOADS))
def test_decode_workloads_sampled(name):
    """Full-size decode workloads, checked on every row of every head."""
    wl, n = W.DECODE_WORKLOADS[name]
    o, lse, ref_o, ref_lse = run_decode(wl, n)
    assert pu.max_abs(o, ref_o) <= pu.TOL["o"], pu.max_abs(o, ref_o)
    assert pu.max_abs(lse, ref_lse) <= pu.TOL["lse"], pu.max_abs(lse, ref_lse)
