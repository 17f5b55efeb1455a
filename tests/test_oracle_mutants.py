"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutant is a one-line textual change to ``oracle/attention_ref.c`` of the
kind a careless restatement of the formula could make; the copy is compiled
into a temporary directory, the committed oracle is untouched.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attention_ref.c")

MUTANTS = {
    "dropped_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "exponent_sign": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "diagonal_excluded": ("jb->causal ? i + 1 : jb->S", "jb->causal ? (i > 0 ? i : 1) : jb->S"),
    "mask_ignored": ("jb->causal ? i + 1 : jb->S", "jb->S"),
    "keys_as_values": ("o[d] += a * (double)V[j * D + d];", "o[d] += a * (double)K[j * D + d];"),
    "feature_index_reversed": ("dot += (double)q[d] * (double)K[j * D + d];",
                               "dot += (double)q[d] * (double)K[j * D + (D - 1 - d)];"),
    "no_normalisation": ("double a = s[j] / Z;", "double a = s[j];"),
    "lse_without_max": ("*lse = m + log(Z);", "*lse = log(Z);"),
    "max_not_subtracted_from_lse": ("*lse = m + log(Z);", "*lse = m * 0.5 + log(Z);"),
    "key_lens_ignored": ("int64_t L = jb->key_lens[bh / jb->H];", "int64_t L = jb->S;"),
    "key_lens_indexed_by_head": ("int64_t L = jb->key_lens[bh / jb->H];",
                                 "int64_t L = jb->key_lens[bh % jb->B];"),
    "decode_ignores_sequence_offset": ("jb->Kc + ((jb->offs[b] + t) * H + h) * D",
                                       "jb->Kc + ((t) * H + h) * D"),
    "decode_value_offset": ("jb->Vc + ((jb->offs[b] + t) * H + h) * D",
                            "jb->Vc + ((jb->offs[b] + t) * H + (H - 1 - h)) * D"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "attention_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.load_library(oracle.build(str(mutated), str(tmp_path / "libmutant.so")))
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(lib)
        except AssertionError:
            caught.append(check.__name__)
            break
    assert caught, f"no pin fails for planted mistake {name}"


# The fused projection is numpy (no C): its planted mistakes are textual
# changes to oracle.qkv_projection's source, executed in place of it.
PY_MUTANTS = {
    "qkv_q_and_k_swapped": ("return Y[0].copy(), Y[1].copy(), Y[2].copy()",
                            "return Y[1].copy(), Y[0].copy(), Y[2].copy()"),
    "qkv_heads_and_features_swapped": ("Y = Y.reshape(B, S, 3, H, D).transpose(2, 0, 3, 1, 4)",
                                       "Y = Y.reshape(B, S, 3, D, H).transpose(2, 0, 4, 1, 3)"),
    "qkv_float32_product": ("Y = np.matmul(X.reshape(B * S, hidden), W)",
                            "Y = np.matmul(X.reshape(B * S, hidden).astype(np.float32), "
                            "W.astype(np.float32))"),
}


OUT_MUTANTS = {
    "out_proj_features_head_minor": ("A = O.transpose(0, 2, 1, 3).reshape(B * S, H * D)",
                                     "A = O.transpose(0, 2, 3, 1).reshape(B * S, H * D)"),
    "out_proj_float32_product": ("return np.matmul(A, W).reshape(B, S, W.shape[1])",
                                 "return np.matmul(A.astype(np.float32), W.astype(np.float32))"
                                 ".reshape(B, S, W.shape[1])"),
}


@pytest.mark.parametrize("name", sorted(OUT_MUTANTS))
def test_out_projection_mutant_is_caught(name, monkeypatch):
    import inspect
    import numpy as np
    old, new = OUT_MUTANTS[name]
    src = inspect.getsource(oracle.out_projection)
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    ns = {"np": np}
    exec(src.replace(old, new), ns)
    monkeypatch.setattr(oracle, "out_projection", ns["out_projection"])
    caught = False
    for check in (oracle_pins.check_out_proj_bruteforce_fsum, oracle_pins.check_out_proj_head_order):
        try:
            check(None)
        except AssertionError:
            caught = True
            break
    assert caught, f"no pin fails for planted mistake {name}"


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_projection_mutant_is_caught(name, monkeypatch):
    import inspect
    import numpy as np
    old, new = PY_MUTANTS[name]
    src = inspect.getsource(oracle.qkv_projection)
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    ns = {"np": np}
    exec(src.replace(old, new), ns)
    monkeypatch.setattr(oracle, "qkv_projection", ns["qkv_projection"])
    caught = False
    for check in (oracle_pins.check_qkv_bruteforce_fsum, oracle_pins.check_qkv_selection_and_layout):
        try:
            check(None)
        except AssertionError:
            caught = True
            break
    assert caught, f"no pin fails for planted mistake {name}"
