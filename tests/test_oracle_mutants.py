"""The pins must be able to fail: plant plausible mistakes in a copy of the oracle (on the CPU)
and check that at least one pin in test_oracle_pins.py catches each of them."""
import os
import shutil
import subprocess
import tempfile
import ctypes

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.cpp")

MUTANTS = {
    "silu_sign": ("z / (1.0 + std::exp(-z))", "z / (1.0 + std::exp(z))"),
    "nibble_order": ("(k & 1) ? (b >> 4) : (b & 0xF)", "(k & 1) ? (b & 0xF) : (b >> 4)"),
    "offset_binary": ("n >= 8 ? n - 16 : n", "n - 8"),
    "one_scale_per_row": ("f16_to_double(sc[g])", "f16_to_double(sc[0])"),
    "ties_to_higher_index": ("for (int e = 0; e < E; ++e) order[e] = e;", "for (int e = 0; e < E; ++e) order[e] = E - 1 - e;"),
    "no_renormalisation": ("for (int k = 0; k < K; ++k) w[k] = p[idx[k]] / kept;", "for (int k = 0; k < K; ++k) w[k] = p[idx[k]];"),
    "shared_dropped": ("for (int j = 0; j < d; ++j) yt[j] += o[j];", "for (int j = 0; j < d; ++j) yt[j] += 0.0 * o[j];"),
    "gate_up_swapped": ("h[i] = silu(g) * u;", "h[i] = silu(u) * g;"),
    "bias_dropped": ("if (bias) acc += bias[e];", "if (bias) acc += 0.0;"),
    "rmsnorm_no_eps": ("ss / d + eps", "ss / d"),
    "f16_bias": ("ex - 15", "ex - 14"),
    "dispatch_unstable": ("return idx[a] < idx[b]; });", "return idx[a] < idx[b] || (idx[a] == idx[b] && a > b); });"),
    "down_row_offset": ("weight_row(wfmt, dn, dn_s, j, f, row.data());", "weight_row(wfmt, dn, dn_s, (j + 1) % d, f, row.data());"),
}

PIN_TESTS = [
    (pins.test_int4_nibbles_match_hand_table, {}),
    (pins.test_int4_group_scales_apply_per_32_columns, {}),
    (pins.test_f16_decode_matches_numpy_all_patterns, {}),
    (pins.test_topk_equals_bruteforce_full_sort, {"E": 16, "K": 4}),
    (pins.test_exact_ties_go_to_lower_index, {}),
    (pins.test_two_expert_weights_closed_form, {}),
    (pins.test_full_softmax_when_k_equals_e, {}),
    (pins.test_dispatch_matches_stable_argsort, {"T": 7, "K": 4, "E": 16}),
    (pins.test_single_expert_is_dense_swiglu, {"wfmt": "int4", "d": 128, "f": 64}),
    (pins.test_k_equals_e_is_full_softmax_mixture, {"shared": True}),
    (pins.test_topk_layer_matches_torch_gather_mixture, {}),
    (pins.test_rmsnorm_closed_forms, {}),
]


def _compile(src_text, out_dir):
    src = os.path.join(out_dir, "mutant.cpp")
    lib = os.path.join(out_dir, "libmutant.so")
    with open(src, "w") as fh:
        fh.write(src_text)
    subprocess.check_call(["g++", "-std=c++17", "-O1", "-fopenmp", "-fPIC", "-shared", src, "-o", lib])
    return lib


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    before, after = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(before) == 1, f"mutation site for {name} not unique"
    tmp = tempfile.mkdtemp()
    try:
        lib = ctypes.CDLL(_compile(text.replace(before, after), tmp))
        monkeypatch.setattr(oracle, "_lib", lib)
        caught = []
        for fn, kw in PIN_TESTS:
            try:
                fn(**kw)
            except AssertionError:
                caught.append(fn.__name__)
        assert caught, f"no pin caught the mutant {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
