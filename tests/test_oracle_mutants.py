"""Mutation check of the oracle pins.

Each case below plants one plausible slip in a private copy of oracle/la_oracle.c (compiled with
gcc into a temporary directory, on the CPU), binds it in place of the real oracle, and runs the
pins of test_oracle_pins.py against it.  A slip that no pin catches fails this test.  The real
oracle source is never modified.
"""
import inspect
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "la_oracle.c")

MUTANTS = {
    "decay_after_add": ("S[(size_t)i * D + j] = S[(size_t)i * D + j] * decay + kt[i] * vt[j];",
                        "S[(size_t)i * D + j] = (S[(size_t)i * D + j] + kt[i] * vt[j]) * decay;"),
    "decay_sign": ("const double decay = exp(-slope);", "const double decay = exp(slope);"),
    "decay_dropped": ("S[(size_t)i * D + j] * decay + kt[i] * vt[j];",
                      "S[(size_t)i * D + j] + kt[i] * vt[j];"),
    "outer_transposed": ("* decay + kt[i] * vt[j];", "* decay + kt[j] * vt[i];"),
    "scale_dropped": ("ot[j] = acc * scale;", "ot[j] = acc;"),
    "scale_inverted": ("const double scale = 1.0 / sqrt((double)D);",
                       "const double scale = sqrt((double)D);"),
    "readout_transposed": ("acc += qt[i] * S[(size_t)i * D + j];",
                           "acc += qt[i] * S[(size_t)j * D + i];"),
    "prefix_ignored": ("if (a->prefix_mask[b])", "if (0)"),
    "prefix_always_read": ("if (a->prefix_mask[b])", "if (1)"),
    "final_state_not_written": ("memcpy(slot, S, sizeof(double) * dd); /* final state",
                                "(void)slot; /* final state"),
    "layer_factor_sign": ("factor = 1.0 - (double)layer_id / (double)(L - 1) + 1e-5;",
                          "factor = 1.0 + (double)layer_id / (double)(L - 1) + 1e-5;"),
    "layer_factor_eps_dropped": ("factor = 1.0 - (double)layer_id / (double)(L - 1) + 1e-5;",
                                 "factor = 1.0 - (double)layer_id / (double)(L - 1);"),
    "single_layer_factor": ("factor = 1.0 + 1e-5;", "factor = 1.0;"),
    "alibi_index": ("pow(2.0, -8.0 * (double)(i + 1) / (double)H)",
                    "pow(2.0, -8.0 * (double)i / (double)H)"),
    "verify_writes_pool": ("inter, (size_t)H * dd);",
                           "inter, (size_t)H * dd);\n        memcpy(slot, S, sizeof(double) * dd);"),
    "verify_inter_lag": ("memcpy(inter + (size_t)t * inter_stride, S,",
                         "memcpy(inter + (size_t)(t + 1 < n ? t + 1 : t) * inter_stride, S,"),
    "decode_zero_start": ("        memcpy(S, slot, sizeof(double) * dd);\n"
                          "        const size_t off = (size_t)b * row + (size_t)h * D;",
                          "        memset(S, 0, sizeof(double) * dd);\n"
                          "        const size_t off = (size_t)b * row + (size_t)h * D;"),
    "request_length_short": ("n = a->cu_seqlens[b + 1] - t0;", "n = a->cu_seqlens[b + 1] - t0 - 1;"),
    "wrong_head_slope": ("recur(S, D, a->slopes[h], n1,", "recur(S, D, a->slopes[0], n1,"),
    "tree_forks_from_previous": ("par < 0 ? root : inter + (((size_t)b * N + par) * H + h) * dd;",
                                 "(t == 0) ? root : inter + (((size_t)b * N + t - 1) * H + h) * dd;"),
    "tree_forks_from_root": ("par < 0 ? root : inter + (((size_t)b * N + par) * H + h) * dd;",
                             "root;"),
    "commit_reads_first_token": ("pool + (size_t)state_idx[b] * hdd, inter + ((size_t)b * N + a) * hdd,",
                                 "pool + (size_t)state_idx[b] * hdd, inter + ((size_t)b * N) * hdd,"),
    "commit_skip_taken_as_zero": ("        if (a < 0)\n            continue;",
                                  "        if (a < 0)\n            a = 0;"),
    "commit_other_request": ("pool + (size_t)state_idx[b] * hdd, inter + ((size_t)b * N + a) * hdd,",
                             "pool + (size_t)state_idx[b] * hdd, inter + ((size_t)(B - 1 - b) * N + a) * hdd,"),
    "track_snapshot_one_late": ("const int n1 = tl >= 0 ? tl : n;",
                                "const int n1 = tl >= 0 ? (tl < n ? tl + 1 : tl) : n;"),
    "track_snapshot_to_own_slot": ("memcpy(a->pool + ((size_t)a->track_idx[b] * H + h) * dd, S,",
                                   "memcpy(a->pool + ((size_t)a->state_idx[b] * H + h) * dd, S,"),
    "track_rest_not_processed": ("recur(S, D, a->slopes[h], n - n1, a->q + off2,",
                                 "recur(S, D, a->slopes[h], 0, a->q + off2,"),
    # grouped-query heads
    "gqa_kv_head_by_modulo": ("const size_t kvo = (size_t)t0 * kv_row + (size_t)j * D;",
                              "const size_t kvo = (size_t)t0 * kv_row + (size_t)((j * G) % a->Hkv) * D;"),
    "gqa_slope_of_query_head": ("recur_group(S, D, a->slopes[j], n, G,",
                                "recur_group(S, D, a->slopes[(j * G) % a->Hkv], n, G,"),
    "gqa_state_advanced_per_query_head": (
        "        for (int g = 0; g < G; g++) {\n            const double *qt",
        "        for (int g = 0; g < G; g++) {\n            if (g > 0)\n                for (int i = 0; i < D; i++)\n"
        "                    for (int j = 0; j < D; j++)\n"
        "                        S[(size_t)i * D + j] = S[(size_t)i * D + j] * decay + kt[i] * vt[j];\n"
        "            const double *qt"),
    "gqa_every_head_reads_the_first_query": ("const double *qt = qg + (size_t)t * q_stride + (size_t)g * D;",
                                             "const double *qt = qg + (size_t)t * q_stride;"),
    "gqa_group_offset_of_kv_head": ("const size_t qo = (size_t)t0 * q_row + (size_t)j * G * D;",
                                    "const size_t qo = (size_t)t0 * q_row + (size_t)j * D;"),
    "gqa_prefix_ignored": ("            if (a->prefix_mask[b])\n                memcpy(S, slot, sizeof(double) * dd);\n            else\n                memset(S, 0, sizeof(double) * dd);\n        }\n        const size_t qo",
                           "            memset(S, 0, sizeof(double) * dd);\n        }\n        const size_t qo"),
}


def _pin_calls():
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = inspect.signature(fn).parameters
        if "split" in params:
            for sp in (0, 64, 129):
                calls.append((f"{name}[{sp}]", lambda fn=fn, sp=sp: fn(sp)))
        elif not params:
            calls.append((name, fn))
    return calls


@pytest.fixture(scope="module")
def base_source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_mutant(mutant, base_source, tmp_path, monkeypatch):
    old, new = MUTANTS[mutant]
    assert base_source.count(old) >= 1, f"mutation anchor not found: {old!r}"
    src = base_source.replace(old, new, 1)
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "libmutant.so"
    c_path.write_text(src)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so_path),
                    str(c_path), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.load_library(str(so_path)))
    caught = []
    for name, call in _pin_calls():
        try:
            call()
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(name)
    assert caught, f"no pin catches the planted slip '{mutant}'"


def test_unmutated_oracle_passes_every_pin():
    for name, call in _pin_calls():
        call()
