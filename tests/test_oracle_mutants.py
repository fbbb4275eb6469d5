"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each.

Each mutant is the oracle's source with one textual substitution, executed
as a throw-away module on the CPU.  A mutant counts as caught when a golden
fixture or one of the closed-form checks below fails (or the mutant raises).
"""
import glob
import json
import os
import types

import numpy as np
import pytest

import oracle.reference as ref

SRC = open(ref.__file__).read()
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

MUTANTS = {
    "gqa_mapping_modulo": ("h = j // G", "h = j % hkv"),
    "lora_sign": ("return V_base + delta", "return V_base - delta"),
    "lora_dropped": ("return V_base + delta.reshape(V_base.shape[0], hkv, d)", "return V_base"),
    "scale_one_over_d": ("scale = 1.0 / np.sqrt(d)", "scale = 1.0 / d"),
    "causal_off_by_one": ("vis = n0 + p + 1", "vis = n0 + p + 2"),
    "agent_block_ignored": ("start = a * agent_stride", "start = 0"),
    "b_head_slice_transposed": ("delta.reshape(V_base.shape[0], hkv, d)",
                                "delta.reshape(V_base.shape[0], d, hkv).transpose(0, 2, 1)"),
    "softmax_not_normalised": ("w /= w.sum()", "w /= len(w)"),
    "build_blocks_shifted": ("return to_f64(X) @ to_f64(A_cat)",
                             "return to_f64(X) @ np.roll(to_f64(A_cat), 1, axis=1)"),
    "rebase_k_v_swapped": ("K_base = (X @ to_f64(W_k))", "K_base = (X @ to_f64(W_v))"),
    "rebase_head_layout_transposed": ("V_base = (X @ to_f64(W_v)).reshape(n, hkv, d)",
                                      "V_base = (X @ to_f64(W_v)).reshape(n, d, hkv).transpose(0, 2, 1)"),
    "ragged_offset_shift": ("t0, t1 = offs[q_req], offs[q_req + 1]\n        Kq",
                            "t0, t1 = offs[q_req], offs[q_req + 1] + (1 if q_req + 2 < len(offs) else 0)\n        Kq"),
}


def _mutant(old, new):
    assert SRC.count(old) >= 1, old
    m = types.ModuleType("oracle_mutant")
    exec(compile(SRC.replace(old, new), "oracle_mutant", "exec"), m.__dict__)
    return m


def _arr(x):
    return np.asarray(x, dtype=np.float64)


def _golden_ok(m):
    for path in sorted(glob.glob(os.path.join(GOLDEN, "*.json"))):
        c = json.load(open(path))
        if c["kind"] == "decode":
            O = m.decode(_arr(c["Q"]), _arr(c["K_base"]), _arr(c["V_base"]), _arr(c["L"]),
                         _arr(c["B"]), c["offsets"], rank=c["rank"], agent_stride=c.get("agent_stride"))
            want = _arr(c["O"])
        elif c["kind"] == "prefill":
            O = m.prefill(_arr(c["Q"]), _arr(c["K_base"]), _arr(c["V_base"]), _arr(c["L"]),
                          _arr(c["B"]), n0=c["n0"], rank=c["rank"])
            want = _arr(c["O"])
        elif c["kind"] == "rebase":
            K, V, L = m.rebase_kv_lr_build(_arr(c["X"]), _arr(c["W_k"]), _arr(c["W_v"]), _arr(c["A_cat"]),
                                           hkv=c["hkv"], d=c["d"])
            O = np.concatenate([K.ravel(), V.ravel(), L.ravel()])
            want = np.concatenate([_arr(c["K_base"]).ravel(), _arr(c["V_base"]).ravel(), _arr(c["L"]).ravel()])
        else:
            O = m.lr_cache_build(_arr(c["X"]), _arr(c["A_cat"]))
            want = _arr(c["L"])
        if O.shape != want.shape or not np.allclose(O, want, rtol=0, atol=1e-12):
            return False
    return True


def test_unmutated_oracle_passes_the_pins():
    m = _mutant("", "")
    assert _golden_ok(m)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    m = _mutant(old, new)
    try:
        ok = _golden_ok(m)
    except Exception:
        ok = False
    assert not ok, f"mutant {name} survived the golden fixtures"
