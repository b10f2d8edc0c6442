"""Checks that pin the CPU oracle to something other than itself.

Each check takes the oracle module as an argument so that the mutation tests
can run the same checks against copies of the oracle with planted mistakes.
A check returns None when it passes and a short message when it fails.

Independent routes used here (none re-types the oracle's formulas):
* a hand-worked example with exact fractions (tests/golden);
* PyTorch float64 scaled_dot_product_attention with one appended key/value
  column (key and value zero, additive mask entry = the sink logit), masks
  built from torch.tril / torch.triu bands, gradients from autograd;
* the closed form alpha = sigmoid(l - s_h) of the summary page, with l taken
  from torch.logsumexp;
* closed forms for window 0 and for one token;
* central finite differences of L = <dO, O>;
* closed-form counts of visible (query, key) pairs.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------- helpers
def rand_problem(seqlens, hq, hkv, d, seed, sink_scale=1.0):
    rng = np.random.default_rng(seed)
    T = int(sum(seqlens))
    q = rng.standard_normal((T, hq, d))
    k = rng.standard_normal((T, hkv, d))
    v = rng.standard_normal((T, hkv, d))
    do = rng.standard_normal((T, hq, d))
    sink = rng.standard_normal(hq) * sink_scale
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int64)
    return q, k, v, do, sink, cu


def torch_mask(n, window, prefix, causal):
    """Visibility built from library band matrices: triu keeps k >= q - w."""
    ones = torch.ones(n, n, dtype=torch.bool)
    band = ones if window < 0 else torch.triu(ones, diagonal=-int(window))
    pre = torch.zeros(n, n, dtype=torch.bool)
    pre[:, : min(int(prefix), n)] = True
    m = band | pre
    if causal:
        m = m & torch.tril(ones)
    return m


def sdpa_with_sink(q, k, v, sink, do, cu, window, prefix, causal, scale):
    """Sink attention through torch SDPA with an appended zero key/value column."""
    T, hq, d = q.shape
    hkv = k.shape[1]
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    ts = torch.tensor(sink, requires_grad=True)
    outs, lses = [], []
    for b in range(len(cu) - 1):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        n = t1 - t0
        if n == 0:
            continue
        Q = tq[t0:t1].permute(1, 0, 2)                                  # [hq, n, d]
        K = tk[t0:t1].permute(1, 0, 2).repeat_interleave(hq // hkv, 0)  # [hq, n, d]
        V = tv[t0:t1].permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
        zero = torch.zeros(hq, 1, d, dtype=torch.float64)
        Ke = torch.cat([K, zero], 1)
        Ve = torch.cat([V, zero], 1)
        allowed = torch_mask(n, window, prefix, causal)
        add = torch.zeros(n, n, dtype=torch.float64).masked_fill(~allowed, float("-inf"))
        add = add.unsqueeze(0).expand(hq, n, n)
        mask = torch.cat([add, ts.view(hq, 1, 1).expand(hq, n, 1)], 2)
        O = torch.nn.functional.scaled_dot_product_attention(Q, Ke, Ve, attn_mask=mask, scale=scale)
        outs.append(O.permute(1, 0, 2))
        with torch.no_grad():
            sc = (Q @ K.transpose(1, 2)) * scale
            lses.append(torch.logsumexp(sc.masked_fill(~allowed, float("-inf")), dim=2))
    O = torch.cat(outs, 0)
    (O * torch.tensor(do)).sum().backward()
    return dict(o=O.detach().numpy(), lse=torch.cat(lses, 1).numpy(), dq=tq.grad.numpy(),
                dk=tk.grad.numpy(), dv=tv.grad.numpy(), dsink=ts.grad.numpy())


def run_oracle(mod, q, k, v, sink, do, cu, window, prefix, causal, scale):
    return mod.forward_backward(q, k, v, sink, do, cu, window, prefix, causal, scale)


def _maxerr(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return float("inf")
    if a.size == 0:
        return 0.0
    if np.any(np.isnan(a)) or np.any(np.isnan(b)):
        return float("inf")
    same_inf = np.isinf(a) & (a == b)
    with np.errstate(invalid="ignore"):
        d = np.where(same_inf, 0.0, np.abs(a - b))
    return float(np.max(np.nan_to_num(d, nan=np.inf)))


def _cmp(got, want, keys, tol, label):
    for key in keys:
        e = _maxerr(got[key], want[key])
        if not e <= tol:
            return f"{label}: {key} max abs err {e:.3g} > {tol}"
    return None


# ----------------------------------------------------------------- checks
def check_hand_example(mod):
    """The 4-token example worked out by hand (tests/golden/hand_s4_w1_p1.json)."""
    with open(os.path.join(GOLDEN, "hand_s4_w1_p1.json")) as f:
        g = json.load(f)

    def val(x):
        if isinstance(x, str) and x.startswith("ln"):
            return math.log(float(x[2:]))
        return float(Fraction(x)) if isinstance(x, str) else float(x)

    arr = lambda a: np.array([[val(x) for x in row] for row in a], dtype=np.float64)
    q = arr(g["q"])[:, None, :]
    k = arr(g["k"])[:, None, :]
    v = arr(g["v"])[:, None, :]
    do = arr(g["dout"])[:, None, :]
    sink = np.array([val(g["sink"])])
    res = run_oracle(mod, q, k, v, sink, do, np.array([0, 4]), g["window"], g["prefix"], g["causal"], g["scale"])
    want = dict(o=arr(g["o"])[:, None, :], lse=np.array([[val(x) for x in g["lse"]]]),
                dq=arr(g["dq"])[:, None, :], dk=arr(g["dk"])[:, None, :], dv=arr(g["dv"])[:, None, :],
                dsink=np.array([val(g["dsink"])]))
    return _cmp(res, want, ["o", "lse", "dq", "dk", "dv", "dsink"], 1e-12, "hand example")


SDPA_CASES = [
    # seqlens, hq, hkv, d, window, prefix, causal, seed
    ((37,), 4, 2, 16, 5, 3, True, 1),
    ((64,), 2, 2, 8, -1, 0, True, 2),
    ((19, 1, 40), 8, 2, 8, 7, 2, True, 3),
    ((23,), 2, 1, 8, 4, 2, False, 4),
    ((33,), 3, 3, 8, 0, 5, True, 5),
]


def check_sdpa(mod):
    """Library cross-check: torch SDPA with a sink column and autograd."""
    for seqlens, hq, hkv, d, w, p, causal, seed in SDPA_CASES:
        q, k, v, do, sink, cu = rand_problem(seqlens, hq, hkv, d, seed)
        scale = 0.7 / math.sqrt(d)
        got = run_oracle(mod, q, k, v, sink, do, cu, w, p, causal, scale)
        want = sdpa_with_sink(q, k, v, sink, do, cu, w, p, causal, scale)
        msg = _cmp(got, want, ["o", "lse", "dq", "dk", "dv", "dsink"], 1e-10, f"sdpa {seqlens} w={w} p={p}")
        if msg:
            return msg
    return None


def check_alpha_closed_form(mod):
    """O with an explicit sink equals sigmoid(l - s_h) times plain masked attention."""
    q, k, v, do, sink, cu = rand_problem((50,), 4, 2, 16, 11, sink_scale=2.0)
    scale = 0.25
    got = run_oracle(mod, q, k, v, sink, do, cu, 9, 3, True, scale)
    n = 50
    Q = torch.tensor(q).permute(1, 0, 2)
    K = torch.tensor(k).permute(1, 0, 2).repeat_interleave(2, 0)
    V = torch.tensor(v).permute(1, 0, 2).repeat_interleave(2, 0)
    allowed = torch_mask(n, 9, 3, True)
    plain = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=allowed, scale=scale)
    l = torch.logsumexp(((Q @ K.transpose(1, 2)) * scale).masked_fill(~allowed, float("-inf")), 2)
    alpha = torch.sigmoid(l - torch.tensor(sink)[:, None])
    o_alpha = (alpha[..., None] * plain).permute(1, 0, 2).numpy()
    return _cmp(got, dict(o=o_alpha, lse=l.numpy()), ["o", "lse"], 1e-12, "alpha closed form")


def check_window0(mod):
    """w = 0, p = 0: one visible key per row, so every output has a closed form."""
    q, k, v, do, sink, cu = rand_problem((21,), 2, 1, 8, 21)
    scale = 0.3
    got = run_oracle(mod, q, k, v, sink, do, cu, 0, 0, True, scale)
    hq = 2
    kk = np.repeat(k, hq, axis=1)
    vv = np.repeat(v, hq, axis=1)
    sqq = scale * np.sum(q * kk, axis=2)                   # [T, hq]
    a = 1.0 / (1.0 + np.exp(sink[None, :] - sqq))         # alpha
    g = np.sum(do * vv, axis=2)                            # <dO_q, v_q>
    ds = a * (1 - a) * g                                   # dS_qq
    want = dict(o=a[..., None] * vv, lse=sqq.T, dq=scale * ds[..., None] * kk,
                dk=(scale * ds[..., None] * q).sum(1, keepdims=True),
                dv=(a[..., None] * do).sum(1, keepdims=True),
                dsink=-np.sum((1 - a) * a * g, axis=0))
    return _cmp(got, want, ["o", "lse", "dq", "dk", "dv", "dsink"], 1e-12, "window 0")


def check_single_token(mod):
    """S = 1: l = s_00 and O = sigmoid(s_00 - s_h) v_0 for any window/prefix."""
    q, k, v, do, sink, cu = rand_problem((1,), 2, 2, 4, 31)
    for w, p in ((-1, 0), (5, 3), (0, 0)):
        got = run_oracle(mod, q, k, v, sink, do, cu, w, p, True, 0.5)
        s = 0.5 * np.sum(q * k, axis=2)
        a = 1.0 / (1.0 + np.exp(sink[None, :] - s))
        msg = _cmp(got, dict(o=a[..., None] * v, lse=s.T), ["o", "lse"], 1e-12, f"single token w={w}")
        if msg:
            return msg
    return None


def check_finite_differences(mod):
    """Analytic gradients match central differences of L = <dO, O>."""
    rng = np.random.default_rng(7)
    for seqlens, w, p in (((7,), 2, 1), ((2,), -1, 0), ((13, 5), 3, 2)):
        q, k, v, do, sink, cu = rand_problem(seqlens, 4, 2, 6, 100 + len(seqlens))
        scale = 0.45
        res = run_oracle(mod, q, k, v, sink, do, cu, w, p, True, scale)

        def L(q_, k_, v_, s_):
            o, _ = mod.forward(q_, k_, v_, s_, cu, w, p, True, scale)
            return float(np.sum(o * do))

        h = 1e-6
        for name, arr, grad in (("q", q, res["dq"]), ("k", k, res["dk"]), ("v", v, res["dv"]),
                                ("sink", sink, res["dsink"])):
            flat = arr.reshape(-1)
            idx = range(flat.size) if flat.size <= 8 else rng.choice(flat.size, 12, replace=False)
            for i in idx:
                old = flat[i]
                flat[i] = old + h
                lp = L(q, k, v, sink)
                flat[i] = old - h
                lm = L(q, k, v, sink)
                flat[i] = old
                fd = (lp - lm) / (2 * h)
                an = grad.reshape(-1)[i]
                if not abs(fd - an) <= 1e-6 * max(1.0, abs(fd)):
                    return f"finite differences {seqlens}: d{name}[{i}] analytic {an:.9g} vs fd {fd:.9g}"
    return None


def check_pair_counts(mod):
    """Visible-pair counts against closed forms.

    Causal, window w, prefix p: row q sees the keys lo .. q with
    lo = max(0, q - w), plus the prefix keys below lo, min(p, lo) of them.
    """
    def closed(n, w, p):
        tot = 0
        for qq in range(n):
            lo = 0 if w < 0 else max(0, qq - w)
            tot += (qq - lo + 1) + min(p, lo)
        return tot

    for n, w, p in ((128, 32, 4), (100, 0, 0), (100, -1, 0), (77, 5, 9), (64, 70, 0)):
        got = mod.unmasked_pairs([n], 1, w, p, True)
        if got != closed(n, w, p):
            return f"pair count n={n} w={w} p={p}: {got} != {closed(n, w, p)}"
    if mod.unmasked_pairs([4096], 64, -1, 0, True) != 64 * 4096 * 4097 // 2:
        return "pair count full causal 4096"
    if mod.unmasked_pairs([9], 1, -1, 0, False) != 81:
        return "pair count non-causal"
    return None


def check_sink_limits(mod):
    """sink = -inf is plain attention with dsink = 0; sink = +inf gives O = 0."""
    q, k, v, do, sink, cu = rand_problem((29,), 2, 1, 8, 41)
    scale = 0.35
    neg = np.array([-np.inf, -np.inf])
    got = run_oracle(mod, q, k, v, neg, do, cu, 6, 2, True, scale)
    want = sdpa_with_sink(q, k, v, np.array([-1e300, -1e300]), do, cu, 6, 2, True, scale)
    want["dsink"] = np.zeros(2)
    msg = _cmp(got, want, ["o", "lse", "dq", "dk", "dv", "dsink"], 1e-10, "sink -inf")
    if msg:
        return msg
    pos = np.array([np.inf, np.inf])
    got = run_oracle(mod, q, k, v, pos, do, cu, 6, 2, True, scale)
    z = dict(o=np.zeros_like(q), dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v), dsink=np.zeros(2))
    return _cmp(got, z, ["o", "dq", "dk", "dv", "dsink"], 0.0, "sink +inf")


def check_mask_equivalences(mod):
    """w >= S - 1 and p >= S both equal full causal; packed equals per-sequence."""
    q, k, v, do, sink, cu = rand_problem((31,), 4, 2, 8, 51)
    full = run_oracle(mod, q, k, v, sink, do, cu, -1, 0, True, 0.3)
    for w, p in ((30, 0), (1000, 0), (0, 31), (3, 40)):
        msg = _cmp(run_oracle(mod, q, k, v, sink, do, cu, w, p, True, 0.3), full,
                   ["o", "lse", "dq", "dk", "dv", "dsink"], 1e-12, f"w={w} p={p} vs full")
        if msg:
            return msg
    lens = (9, 1, 14)
    q, k, v, do, sink, cu = rand_problem(lens, 4, 2, 8, 52)
    packed = run_oracle(mod, q, k, v, sink, do, cu, 3, 2, True, 0.3)
    acc_dsink = np.zeros(4)
    for b in range(3):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        one = run_oracle(mod, q[t0:t1], k[t0:t1], v[t0:t1], sink, do[t0:t1], np.array([0, t1 - t0]), 3, 2, True, 0.3)
        acc_dsink += one["dsink"]
        for key in ("o", "dq", "dk", "dv"):
            if _maxerr(packed[key][t0:t1], one[key]) > 1e-12:
                return f"packed vs per-sequence: {key} of sequence {b}"
        if _maxerr(packed["lse"][:, t0:t1], one["lse"]) > 1e-12:
            return f"packed vs per-sequence: lse of sequence {b}"
    if _maxerr(packed["dsink"], acc_dsink) > 1e-12:
        return "packed vs per-sequence: dsink"
    return None


def check_gqa_vs_mha(mod):
    """GQA equals MHA on replicated K/V, with dK/dV summed over each group."""
    q, k, v, do, sink, cu = rand_problem((25,), 6, 2, 8, 61)
    gqa = run_oracle(mod, q, k, v, sink, do, cu, 5, 1, True, 0.3)
    kk, vv = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    mha = run_oracle(mod, q, kk, vv, sink, do, cu, 5, 1, True, 0.3)
    mha["dk"] = mha["dk"].reshape(25, 2, 3, 8).sum(2)
    mha["dv"] = mha["dv"].reshape(25, 2, 3, 8).sum(2)
    return _cmp(gqa, mha, ["o", "lse", "dq", "dk", "dv", "dsink"], 1e-12, "gqa vs mha")


def check_invariants(mod):
    """dsink = -sum (1 - alpha) <dO, O> with alpha = sigmoid(l - s); 0 < alpha < 1."""
    q, k, v, do, sink, cu = rand_problem((40, 17), 4, 4, 8, 71, sink_scale=3.0)
    res = run_oracle(mod, q, k, v, sink, do, cu, 11, 3, True, 0.3)
    D = np.sum(do * res["o"], axis=2)                      # [T, hq]
    alpha = 1.0 / (1.0 + np.exp(sink[:, None] - res["lse"]))
    if not np.all((alpha > 0) & (alpha < 1)):
        return "alpha outside (0, 1)"
    e = _maxerr(res["dsink"], -np.sum((1 - alpha) * D.T, axis=1))
    return None if e < 1e-12 else f"dsink identity err {e:.3g}"


def check_decode_sdpa(mod):
    """Decode rows equal the last rows of SDPA over the whole sequence."""
    for (lens, n, window, prefix, hq, hkv, seed) in [((40, 17, 9), 3, 11, 3, 4, 2, 81), ((33, 5), 1, -1, 0, 6, 3, 82),
                                                     ((20,), 4, 2, 0, 2, 1, 83)]:
        q, k, v, do, sink, cu = rand_problem(lens, hq, hkv, 8, seed)
        want = sdpa_with_sink(q, k, v, sink, do, cu, window, prefix, True, 0.35)
        last = np.concatenate([np.arange(int(cu[b + 1]) - n, int(cu[b + 1])) for b in range(len(lens))])
        o, lse = mod.decode_forward(q[last], k, v, sink, cu, n, window, prefix, True, 0.35)
        msg = _cmp({"o": o, "lse": lse}, {"o": want["o"][last], "lse": want["lse"][:, last]}, ["o", "lse"], 1e-12,
                   f"decode lens={lens} n={n}")
        if msg:
            return msg
    return None


ALL_CHECKS = [check_hand_example, check_sdpa, check_alpha_closed_form, check_window0, check_single_token,
              check_finite_differences, check_pair_counts, check_sink_limits, check_mask_equivalences,
              check_gqa_vs_mha, check_invariants, check_decode_sdpa]


def run_all(mod):
    """name -> None (pass) or failure message; exceptions count as failures."""
    out = {}
    for fn in ALL_CHECKS:
        try:
            out[fn.__name__] = fn(mod)
        except Exception as e:  # a planted mistake may break shapes
            out[fn.__name__] = f"raised {type(e).__name__}: {e}"
    return out
