"""Plant plausible mistakes in a copy of the oracle and show the pins catch each.

Every mutation edits the oracle's source text, loads the edited copy as a
separate module on the CPU and runs the full pin suite against it.  A
mutation that no pin detects fails this test.
"""
import importlib.util
import os
import sys
import types

import pytest

from tests import oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "sinkattn_ref.py")

MUTATIONS = {
    "exclusive_window": ("in_window = (qq - kk) <= window", "in_window = (qq - kk) < window"),
    "prefix_inclusive": ("in_prefix = kk < prefix", "in_prefix = kk <= prefix"),
    "drop_causal": ("m = m & (kk <= qq)", "m = m"),
    "strict_causal": ("m = m & (kk <= qq)", "m = m & (kk < qq)"),
    "lse_includes_sink": ("lse = np.log(np.sum(np.exp(scores - safe[:, None]), axis=1)) + safe",
                          "lse = np.log(np.sum(np.exp(scores - safe[:, None]), axis=1) + np.exp(sink_logit - safe)) + safe"),
    "sink_not_in_softmax": ("ext = np.concatenate([scores, np.full((R, 1), sink_logit, dtype=np.float64)], axis=1)",
                            "ext = np.concatenate([scores, np.full((R, 1), -np.inf, dtype=np.float64)], axis=1)"),
    "sink_scaled": ("p, p_sink, l = _extended_softmax(s, float(sink[h]))",
                    "p, p_sink, l = _extended_softmax(s, scale * float(sink[h]))"),
    "dsink_sign": ("dsink[h] += np.sum(ds_sink)", "dsink[h] -= np.sum(ds_sink)"),
    "dsink_drops_alpha": ("ds_sink = p_sink * (dp_sink - D)", "ds_sink = (dp_sink - D)"),
    "D_without_p": ("D = np.sum(p * dp, axis=1) + p_sink * dp_sink", "D = np.sum(dp, axis=1) + p_sink * dp_sink"),
    "dq_no_scale": ("dq[t0 + r0:t0 + r1, h, :] = scale * (ds @ K)", "dq[t0 + r0:t0 + r1, h, :] = (ds @ K)"),
    "dk_uses_p": ("dk[t0:t1, g, :] += scale * (ds.T @ Q[r0:r1])", "dk[t0:t1, g, :] += scale * (p.T @ Q[r0:r1])"),
    "dv_uses_ds": ("dv[t0:t1, g, :] += p.T @ dO", "dv[t0:t1, g, :] += ds.T @ dO"),
    "gqa_modulo": ("        g = h // group\n        if with_bwd:", "        g = h % hkv\n        if with_bwd:"),
    "ds_sign": ("ds = p * (dp - D[:, None])", "ds = p * (D[:, None] - dp)"),
    "decode_position_shift": ("m = visible(np.arange(L - n, L), np.arange(L), window, prefix, causal)",
                              "m = visible(np.arange(L - n + 1, L + 1), np.arange(L), window, prefix, causal)"),
    "decode_head_map": ("            g = h // group\n            s = scale * (q[rows, h, :]",
                        "            g = h % hkv\n            s = scale * (q[rows, h, :]"),
}


def load_mutant(old, new):
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(text.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name):
    mod = load_mutant(*MUTATIONS[name])
    results = pins.run_all(mod)
    failed = [k for k, v in results.items() if v is not None]
    assert failed, f"planted mistake {name!r} passed every pin"
