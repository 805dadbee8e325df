"""The pins must catch plausible mistakes in the oracle.

Each mutant is a copy of the oracle source with one planted mistake (a
dropped term, a wrong sign, a wrong or transposed index), compiled on the CPU
into a temporary library.  Every mutant must fail at least one pin; the real
oracle passes them all (test_oracle.py)."""
import ctypes
import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")

MUTANTS = {
    "scale_dropped": ("scores[j] = scale * dot;", "scores[j] = dot;"),
    "softmax_sign": ("scores[j] = exp(scores[j] - smax);",
                     "scores[j] = exp(smax - scores[j]);"),
    "max_not_subtracted_from_first": ("for (int32_t j = 0; j < ctx; ++j) {\n        scores[j] = exp(",
                                      "for (int32_t j = 1; j < ctx; ++j) {\n        scores[j] = exp("),
    "first_value_dropped": ("for (int32_t j = 0; j < ctx; ++j) {\n        double p",
                            "for (int32_t j = 1; j < ctx; ++j) {\n        double p"),
    "denominator_not_divided": ("double p = scores[j] / denom;", "double p = scores[j];"),
    "block_offset_swapped": ("int32_t logical_block = j / bs;\n        int32_t offset = j % bs;",
                             "int32_t logical_block = j % bs;\n        int32_t offset = j / bs;"),
    "head_offset_transposed": ("(((physical * Hkv + h) * (int64_t)bs + offset) * D)",
                               "(((physical * bs + offset) * (int64_t)Hkv + h) * D)"),
    "gqa_interleaved": ("int32_t hkv = hq / group;", "int32_t hkv = hq % job->Hkv;"),
    "contig_ignores_head": ("((((int64_t)req_id * Hkv + h) * S + j) * D)",
                            "((((int64_t)req_id * Hkv + 0) * S + j) * D)"),
    "contig_offset_without_S": ("((((int64_t)req_id * Hkv + h) * S + j) * D)",
                                "((((int64_t)req_id + h) * S + j) * D)"),
    "append_offset_wrong": ("int64_t offset = slot % bs;", "int64_t offset = (slot + 1) % bs;"),
    "append_v_from_k": ("memcpy(v_cache + dst, v + src,", "memcpy(v_cache + dst, k + src,"),
    "copy_only_k": ("memmove(v_caches[l] + dst * block_elems,\n                    v_caches[l] + src * block_elems,",
                    "memmove(v_caches[l] + src * block_elems,\n                    v_caches[l] + src * block_elems,"),
    "copy_direction": ("memmove(k_caches[l] + dst * block_elems,\n                    k_caches[l] + src * block_elems,",
                       "memmove(k_caches[l] + src * block_elems,\n                    k_caches[l] + dst * block_elems,"),
    "prefill_causal_off_by_one": ("int32_t n = pos + 1; /* positions 0 .. pos */",
                                  "int32_t n = pos; /* positions 0 .. pos */"),
    "prefill_positions_from_zero": ("int32_t pos = ctx - Lq + (t - job->cu_q[i]);",
                                    "int32_t pos = (t - job->cu_q[i]);"),
    "prefill_gqa_interleaved": ("int32_t kv_head = hq / group;",
                                "int32_t kv_head = hq % job->Hkv;"),
    "prefill_wrong_sequence": ("while (i + 1 < job->B && job->cu_q[i + 1] <= t)",
                               "while (i + 1 < job->B && job->cu_q[i + 1] < t)"),
    "bf16_widen_wrong": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
}


def _build_mutant(tmp_path, name):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, "mutation site for %s must be unique" % name
    path = tmp_path / ("%s.c" % name)
    path.write_text(src.replace(old, new))
    lib = tmp_path / ("lib%s.so" % name)
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-shared",
                    "-fPIC", "-pthread", str(path), "-o", str(lib), "-lm"],
                   check=True)
    return oracle.configure(ctypes.CDLL(str(lib)))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, monkeypatch, name):
    monkeypatch.setattr(oracle, "_lib", _build_mutant(tmp_path, name))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(oracle)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, "no pin caught the planted mistake %r" % name
