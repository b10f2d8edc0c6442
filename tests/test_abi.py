"""The C-ABI library builds, loads and exports every declared entry point;
host-side argument checks return their statuses without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sinkattn.h")


@pytest.fixture(scope="module")
def lib():
    from sink_aware_masked_gb300 import _lib, build

    build.build()
    return _lib.load()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sinkattn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("sinkattn_fwd", "sinkattn_bwd", "sinkattn_varlen_plan", "sinkattn_pack", "sinkattn_unpack",
              "sinkattn_fwd_workspace_size", "sinkattn_bwd_workspace_size", "sinkattn_get_device_status",
              "sinkattn_status_string", "sinkattn_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from sink_aware_masked_gb300 import _lib

    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared but not exported"
        assert name in _lib.SIGNATURES, f"{name} has no binding signature"


def test_version_and_status_strings(lib):
    assert lib.sinkattn_version() >= 100
    assert lib.sinkattn_status_string(0) == b"ok"
    assert lib.sinkattn_status_string(3).startswith(b"pointer")
    assert lib.sinkattn_status_string(99) == b"unknown status"


def problem(**kw):
    from sink_aware_masked_gb300 import _lib

    base = dict(num_seqs=1, seqlen=256, cu_seqlens=None, cu_seqlens_host=None, total_tokens=256,
                num_heads_q=8, num_heads_kv=2, head_dim=64, window=-1, prefix=0, causal=1, scale=0.125)
    base.update(kw)
    return _lib.Problem(**base)


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails validation first


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=128), 2),
    (dict(num_heads_q=6, num_heads_kv=4), 1),
    (dict(num_heads_kv=0), 1),
    (dict(num_heads_q=512, num_heads_kv=2), 2),
    (dict(window=-2), 1),
    (dict(prefix=-1), 1),
    (dict(scale=0.0), 1),
    (dict(scale=float("nan")), 1),
    (dict(scale=float("inf")), 1),
    (dict(causal=2), 1),
    (dict(total_tokens=255), 1),
    (dict(num_seqs=-1), 1),
])
def test_invalid_problem(lib, kw, status):
    pr = problem(**kw)
    assert lib.sinkattn_fwd(ctypes.byref(pr), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, None) == status
    assert lib.sinkattn_fwd_workspace_size(ctypes.byref(pr)) == 0
    assert lib.sinkattn_bwd_workspace_size(ctypes.byref(pr)) == 0


def test_null_and_misaligned_pointers(lib):
    pr = problem()
    assert lib.sinkattn_fwd(ctypes.byref(pr), None, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, None) == 1
    assert lib.sinkattn_fwd(ctypes.byref(pr), FAKE + 8, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, None) == 3
    ws = lib.sinkattn_bwd_workspace_size(ctypes.byref(pr))
    args = [FAKE] * 11
    # workspace too small
    assert lib.sinkattn_bwd(ctypes.byref(pr), *args, FAKE, ws - 1, None) == 4
    # misaligned dq
    bad = list(args)
    bad[7] = FAKE + 2
    assert lib.sinkattn_bwd(ctypes.byref(pr), *bad, FAKE, ws, None) == 3
    assert lib.sinkattn_bwd(ctypes.byref(pr), *args, None, ws, None) == 1


def test_workspace_sizes_are_linear_in_tokens(lib):
    """The backward workspace is the fp32 dQ accumulator and one 16-byte bias
    row per (head, token), both linear in T, plus the per-chunk dK/dV slots of
    split key tiles: at most 2 * SMs + (key tiles) * Hkv slot-heads of 64 KB
    (chunks hold at least half an SM's share of the work, so there are at most
    2 * SMs / Hkv more chunks than tiles).  No term grows faster than T."""
    sms = 152  # the host-side plan without a device assumes a GB300
    sizes = []
    for S in (1024, 2048, 4096, 8192, 16384, 32768):
        for window in (-1, 128):
            pr = problem(seqlen=S, total_tokens=S, num_heads_q=64, num_heads_kv=8, window=window)
            ws = lib.sinkattn_bwd_workspace_size(ctypes.byref(pr))
            linear = S * 64 * 64 * 4 + S * 64 * 16
            assert ws >= linear
            tiles = (S + 127) // 128
            assert ws <= linear + (2 * sms + tiles * 8) * 65536 + S * 64 + 4096, (S, window)
            if window == -1:
                sizes.append(ws)
    # Large problems split few tiles: doubling T doubles the workspace.
    assert abs(sizes[-1] - 2 * sizes[-2]) <= 0.01 * sizes[-1]
    assert lib.sinkattn_fwd_workspace_size(ctypes.byref(problem())) == 0


def test_varlen_offsets_validation(lib):
    from sink_aware_masked_gb300 import _lib

    def mk(host, total, seqlen):
        arr = (ctypes.c_int32 * len(host))(*host)
        pr = _lib.Problem(num_seqs=len(host) - 1, seqlen=seqlen, cu_seqlens=FAKE,
                          cu_seqlens_host=ctypes.cast(arr, ctypes.c_void_p).value, total_tokens=total,
                          num_heads_q=4, num_heads_kv=4, head_dim=64, window=-1, prefix=0, causal=1, scale=0.1)
        return pr, arr

    for host, total, seqlen in (([1, 5], 5, 5), ([0, 5, 3], 3, 5), ([0, 5, 9], 8, 5), ([0, 5, 9], 9, 4)):
        pr, keep = mk(host, total, seqlen)
        assert lib.sinkattn_fwd(ctypes.byref(pr), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, None) == 1
    pr, keep = mk([0, 5, 9], 9, 5)
    assert lib.sinkattn_bwd_workspace_size(ctypes.byref(pr)) > 0
    # cu_seqlens given without its host copy
    pr = _lib.Problem(num_seqs=1, seqlen=4, cu_seqlens=FAKE, cu_seqlens_host=None, total_tokens=4,
                      num_heads_q=4, num_heads_kv=4, head_dim=64, window=-1, prefix=0, causal=1, scale=0.1)
    assert lib.sinkattn_fwd(ctypes.byref(pr), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, None) == 1


def test_pack_validation(lib):
    assert lib.sinkattn_pack(FAKE, FAKE, -1, 4, 2, 64, FAKE, None) == 1
    assert lib.sinkattn_pack(FAKE, FAKE, 2, 4, 1, 4, FAKE, None) == 2       # 8-byte rows
    assert lib.sinkattn_unpack(FAKE + 4, FAKE, 2, 4, 2, 64, FAKE, None) == 3
    assert lib.sinkattn_varlen_plan(FAKE, -3, FAKE, None) == 1
    assert lib.sinkattn_varlen_plan(None, 3, FAKE, None) == 1


@pytest.mark.parametrize("n,kw,status", [
    (0, {}, 1),                                        # no query rows
    (33, {}, 2),                                       # 4 heads per group x 33 rows > 128
    (20, dict(seqlen=16, total_tokens=16), 1),         # more query rows than cached positions
    (1, dict(head_dim=128), 2),
    (1, dict(num_seqs=4097, seqlen=1, total_tokens=4097), 2),
])
def test_decode_validation(lib, n, kw, status):
    pr = problem(**kw)
    assert lib.sinkattn_decode_fwd(ctypes.byref(pr), n, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, None) == status
    assert lib.sinkattn_decode_workspace_size(ctypes.byref(pr), n) == 0


def test_decode_pointers_and_workspace(lib):
    pr = problem()
    ws = lib.sinkattn_decode_workspace_size(ctypes.byref(pr), 2)
    assert ws > 0
    assert lib.sinkattn_decode_fwd(ctypes.byref(pr), 2, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, None) == 1
    assert lib.sinkattn_decode_fwd(ctypes.byref(pr), 2, FAKE, FAKE + 4, FAKE, FAKE, FAKE, FAKE, FAKE, ws, None) == 3
    assert lib.sinkattn_decode_fwd(ctypes.byref(pr), 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws - 1, None) == 4


def grpo_problem(**kw):
    from sink_aware_masked_gb300 import _lib

    host = (ctypes.c_int32 * 3)(0, 5, 9)
    base = dict(num_rollouts=2, group_size=2, cu_tokens=FAKE, cu_tokens_host=ctypes.cast(host, ctypes.c_void_p).value,
                total_tokens=9, clip_eps=0.2, adv_eps=1e-6, kl_beta=0.0)
    base.update(kw)
    return _lib.GrpoProblem(**base), host


@pytest.mark.parametrize("kw,status", [
    (dict(group_size=0), 1),
    (dict(group_size=3), 1),            # does not divide the rollouts
    (dict(clip_eps=0.0), 1),
    (dict(adv_eps=-1.0), 1),
    (dict(kl_beta=float("nan")), 1),
    (dict(total_tokens=10), 1),         # offsets end elsewhere
])
def test_grpo_validation(lib, kw, status):
    g, host = grpo_problem(**kw)
    assert lib.sinkattn_grpo_loss(ctypes.byref(g), FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 20,
                                  None) == status
    assert lib.sinkattn_grpo_workspace_size(ctypes.byref(g)) == 0


def test_grpo_pointers(lib):
    g, host = grpo_problem(kl_beta=0.1)
    ws = lib.sinkattn_grpo_workspace_size(ctypes.byref(g))
    assert ws > 0
    # logp_ref is required when the KL term is on
    assert lib.sinkattn_grpo_loss(ctypes.byref(g), FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, FAKE, ws, None) == 1
    assert lib.sinkattn_grpo_loss(ctypes.byref(g), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, ws - 1,
                                  None) == 4


def test_grpo_alignment(lib):
    g, host = grpo_problem()
    ws = lib.sinkattn_grpo_workspace_size(ctypes.byref(g))
    assert lib.sinkattn_grpo_loss(ctypes.byref(g), FAKE + 4, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, FAKE, ws,
                                  None) == 3
    assert lib.sinkattn_grpo_loss(ctypes.byref(g), FAKE, FAKE, None, FAKE + 1, FAKE, FAKE, FAKE, None, FAKE, ws,
                                  None) == 3


def _decode_plan_items(lens, hq, hkv, n, window=-1, prefix=0, sms=152):
    """The decode planner's chunk count, restated: 128-key tiles per sequence
    (prefix tiles, then the band of the last n rows), a chunk factor of 4 x the
    SMs per kv head for a single 16-row block with >= 1024 tiles, else 2, at
    least two tiles per chunk."""
    tiles = []
    for L in lens:
        q0, hi = L - n, L - 1
        lo = 0 if window < 0 else max(0, q0 - window)
        pre_end = max(0, min(min(prefix, lo), hi + 1))
        lo_t = lo // 128
        n_pre = min((pre_end + 127) // 128, lo_t)
        tiles.append(n_pre + (hi // 128 - lo_t + 1))
    total = sum(tiles)
    rows = (hq // hkv) * n
    items_at = lambda t: sum(-(-x // t) for x in tiles)  # noqa: E731
    if rows <= 16 and total < 128:
        factor = 4 if total >= 1024 else 2
        want = max(1, factor * sms // hkv)
        tps = max(2, -(-total // want))
        while items_at(tps) > 4096:
            tps *= 2
        return items_at(tps)
    # Tensor-core kernel: the smallest chunk length whose grid fits one wave
    # of resident CTAs (two per SM up to 64 rows, one above).
    per_sm = 2 if rows <= 64 else 1
    target = min(max(max(1, per_sm * sms // hkv), len(tiles)), 4096)
    tps = max(2, -(-total // target))
    while items_at(tps) > target:
        tps += 1
    return items_at(tps)


@pytest.mark.parametrize("lens,n,window,prefix", [
    ([8192] * 32, 1, -1, 0),                                       # 32 x 8192: tensor cores, one wave
    ([32768] * 8, 4, -1, 0),                                       # 32 rows per kv head: factor 2
    ([6111, 5036, 1589, 6459, 1056, 6459, 3018, 2085], 1, -1, 0),  # packed: 253 tiles per kv head, tensor cores
    ([8192] * 32, 1, 128, 4),                                      # window and prefix
    ([8192] * 32, 8, -1, 0),                                       # 64 rows: tensor-core kernel, 2 CTAs per SM
    ([5000, 300, 9000], 16, 200, 3),                               # 128 rows: one CTA per SM
])
def test_decode_plan_chunk_count(lib, lens, n, window, prefix):
    """The workspace size encodes the plan: counters, one partial (O and
    (max, sum for O, sum for lse, 0)) per chunk, kv head and row, each region
    256-byte aligned."""
    from sink_aware_masked_gb300 import _lib

    hq, hkv = 64, 8
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    arr = (ctypes.c_int32 * len(cu))(*cu)
    pr = _lib.Problem(num_seqs=len(lens), seqlen=max(lens), cu_seqlens=FAKE,
                      cu_seqlens_host=ctypes.cast(arr, ctypes.c_void_p).value, total_tokens=cu[-1],
                      num_heads_q=hq, num_heads_kv=hkv, head_dim=64, window=window, prefix=prefix, causal=1,
                      scale=0.125)
    items = _decode_plan_items(lens, hq, hkv, n, window, prefix)
    R = (hq // hkv) * n
    r256 = lambda x: -(-x // 256) * 256  # noqa: E731
    want = r256(len(lens) * hkv * 4) + r256(items * hkv * R * 64 * 4) + r256(items * hkv * R * 16) + 256
    assert lib.sinkattn_decode_workspace_size(ctypes.byref(pr), n) == want


@pytest.mark.parametrize("total", [9, 2048 * 4, 2048 * 4 + 3, 2_434_425])
def test_grpo_workspace_layout(lib, total):
    """Two 128-byte lines of barrier words, then one (sum J, sum k3,
    clipped) partial per CTA, 256-byte aligned; the grid is at most one CTA
    per 512-vector stage and two CTAs per SM (152 SMs without a device)."""
    host = (ctypes.c_int32 * 3)(0, total // 2, total)
    g, _ = grpo_problem(cu_tokens_host=ctypes.cast(host, ctypes.c_void_p).value, total_tokens=total)
    ctas = min(max(1, -(-(total // 4) // 512)), 2 * 152)
    assert lib.sinkattn_grpo_workspace_size(ctypes.byref(g)) == 256 + -(-(ctas * 16) // 256) * 256


@pytest.mark.parametrize("name,fwd,bwd", [
    # backward: preprocess, main, conversion (dQ, the split key tiles' dK/dV, dsink)
    ("causal_gqa_b2_s8192", 1, 3),
    ("causal_gqa_s4096", 1, 3),                 # key tiles split into chunks
    ("window128_prefix4_gqa_b2_s8192", 1, 3),   # the always-visible prefix tiles are split
    ("window128_gqa_s4096", 1, 3),
    ("varlen8_causal", 1, 3),
])
def test_kernel_launch_counts(lib, name, fwd, bwd):
    """The launches the library reports for the benchmark's workloads (its
    own work lists, host arithmetic only)."""
    import workloads as W
    from sink_aware_masked_gb300 import _lib

    wl = W.WORKLOADS[name]
    cu = wl.cu_seqlens()
    arr = (ctypes.c_int32 * len(cu))(*[int(x) for x in cu])
    pr = _lib.Problem(num_seqs=wl.num_seqs, seqlen=wl.max_seqlen, cu_seqlens=FAKE,
                      cu_seqlens_host=ctypes.cast(arr, ctypes.c_void_p).value, total_tokens=wl.total_tokens,
                      num_heads_q=wl.num_heads_q, num_heads_kv=wl.num_heads_kv, head_dim=64,
                      window=wl.window, prefix=wl.prefix, causal=int(wl.causal), scale=wl.scale)
    assert lib.sinkattn_kernel_launches(ctypes.byref(pr), 1) == fwd
    assert lib.sinkattn_kernel_launches(ctypes.byref(pr), 2) == bwd
    assert lib.sinkattn_kernel_launches(ctypes.byref(pr), 3) == -1


@pytest.mark.parametrize("window,max_tokens", [(128, 1923), (-1, 1408)])
def test_noalloc_limit_at_64_by_8_heads(lib, window, max_tokens):
    """The no-allocation backward holds 32 MiB: 272 bytes per (token, query
    head) for the dQ accumulator and bias rows, plus the dsink partials and,
    for long causal tiles, the per-chunk dK/dV slots.  One sequence at 64/8
    heads fits up to 1,923 tokens with a 128-token window and 1,408 fully
    causal; one token more is rejected before anything is launched."""
    def pr(S):
        return problem(seqlen=S, total_tokens=S, num_heads_q=64, num_heads_kv=8, window=window)

    limit = 32 << 20
    assert lib.sinkattn_bwd_workspace_size(ctypes.byref(pr(max_tokens))) <= limit
    assert lib.sinkattn_bwd_workspace_size(ctypes.byref(pr(max_tokens + 1))) > limit
    assert lib.sinkattn_bwd_noalloc(ctypes.byref(pr(max_tokens + 1)), *([FAKE] * 11), None) == 4
