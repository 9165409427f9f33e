"""Planted mistakes: each mutant of the oracle source must fail at least one pin.

A mutant is oracle.c with one plausible slip written in (a wrong head map, a
dropped scale, a floor turned into a ceiling, the V half read as K, ...).  It
is compiled to a temporary library on the CPU and the pins of
test_oracle_pins.py are run against it; the test passes only when some pin
catches the slip.  The oracle itself is never modified.
"""
import json
import os
import subprocess
import sys
import tempfile

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "gqa head map modulo": ("const int hk = h / G;\n            const long L", "const int hk = h % Hkv;\n            const long L"),
    "k_scale dropped": ("const double bmm1 = scale * q_scale * k_scale;", "const double bmm1 = scale * q_scale;"),
    "v_scale dropped": ("const double bmm2 = v_scale;", "const double bmm2 = 1.0;"),
    "window start ceil": ("long sp = orc_floor_div(L - span, P);", "long sp = orc_floor_div(L - span + P - 1, P);"),
    "window span off by one": ("long span = window + sq - 1;", "long span = window + sq;"),
    "V read from the K half": ("* 2L * D + D);", "* 2L * D);"),
    "slot from the wrong token": ("long page = block_table[(long)b * bt_stride + j / P];\n                    if (page < 0 || page >= num_pages) {",
                                  "long page = block_table[(long)b * bt_stride + (j + 1) / P];\n                    if (page < 0 || page >= num_pages) {"),
    "lse in base 2": ("*lse_out = m + log(sum);", "*lse_out = m + log2(sum);"),
    "segment prior dropped": ("denom += exp(l[g] + prior - mx);", "denom += exp(l[g] - mx);"),
    "dead segment kept": ("if (used[(long)i * groups + g] <= 0) continue;\n                    double prior = g < topk ? bias[(long)i * topk + g] : 0.0;\n                    acc",
                          "double prior = g < topk ? bias[(long)i * topk + g] : 0.0;\n                    acc"),
    "local segment offset": (": (long)topk * bs);", ": (long)topk * bs + 1);"),
    "merge ignores live mask": ("if (live && live[nn * S + s] <= 0) continue;\n                    double lg = part_lse[(nn * S + s) * H + h] + (prior ? prior[nn * S + s] : 0.0);\n                    if (lg == -INFINITY) continue;\n                    acc",
                                "double lg = part_lse[(nn * S + s) * H + h] + (prior ? prior[nn * S + s] : 0.0);\n                    if (lg == -INFINITY) continue;\n                    acc"),
    "bf16 decoded as low half": ("uint32_t u = ((uint32_t)h) << 16;", "uint32_t u = ((uint32_t)h) << 15;"),
    "e4m3 exponent bias 8": ("v = ldexp((double)(8 + m), e - 10);", "v = ldexp((double)(8 + m), e - 11);"),
    "causal position off by one": ("long pos = L - sq + i;", "long pos = L - sq + i - 1;"),
    "e4m3 mantissa truncated": ("double t = nearbyint((ldexp(a, -e) - 1.0) * 8.0);",
                                "double t = floor((ldexp(a, -e) - 1.0) * 8.0);"),
    "e4m3 overflow to the NaN code": ("if (a >= 448.0) return sign | 0x7E;", "if (a >= 448.0) return sign | 0x7F;"),
    "cache write V over K": ("((uint16_t*)cache)[dst + D + d] = ((const uint16_t*)value)[src + d];",
                             "((uint16_t*)cache)[dst + d] = ((const uint16_t*)value)[src + d];"),
    "cache write slot offset": ("const long page = (long)(s / P), off = (long)(s % P);",
                                "const long page = (long)(s / P), off = (long)((s + 1) % P);"),
    "cache write key scale ignored": ("orc_encode_e4m3(kx / k_scale);", "orc_encode_e4m3(kx);"),
    "paged segment key off by one": ("const long j = st + t;\n                    const long page = block_table[(long)i * bt_stride + j / P];\n                    const size_t kbase",
                                     "const long j = st + t + 1;\n                    const long page = block_table[(long)i * bt_stride + j / P];\n                    const size_t kbase"),
}

PINS = [
    pins.test_decode_bf16_all_codes_match_torch,
    pins.test_decode_e4m3_all_codes_match_torch,
    pins.test_window_start_matches_hand_worked_rows,
    pins.test_two_key_worked_example,
    pins.test_lse_merge_worked_example,
    pins.test_single_key_returns_its_value,
    pins.test_zero_query_gives_log_count_and_mean,
    pins.test_gqa_equals_mha_with_repeated_heads,
    pins.test_fp8_power_of_two_scales_equal_bf16_on_dequantised_values,
    pins.test_tiny_workload_matches_brute_force,
    pins.test_segments_match_brute_force,
    pins.test_segments_combine_equals_union_attention_with_bias,
    pins.test_lse_merge_dead_parts_and_all_dead,
    lambda: pins.test_paged_decode_matches_brute_force(dict(sq=3, causal=True, window=10)),
    lambda: pins.test_paged_decode_matches_brute_force(dict(sq=3, window=20)),
    pins.test_encode_e4m3_exact_values_round_trip,
    pins.test_encode_e4m3_matches_torch_round_to_nearest_even,
    pins.test_encode_e4m3_saturates,
    pins.test_cache_write_16bit_places_rows_by_slot,
    pins.test_cache_write_fp8_quantises_each_element,
    pins.test_paged_segments_equal_contiguous_segments_after_gathering,
    pins.test_paged_segments_single_segment_is_window_decode,
]


def _compile(src_text, out_path):
    with tempfile.NamedTemporaryFile("w", suffix=".c", delete=False) as f:
        f.write(src_text)
        c_path = f.name
    try:
        subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", c_path,
                        "-o", out_path, "-lm"], check=True, capture_output=True)
    finally:
        os.unlink(c_path)


def run_pins() -> list:
    """Names of the pins that fail against the oracle library currently bound."""
    caught = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError):
            caught.append(getattr(pin, "__name__", "lambda"))
    return caught


# A mutant may read past an array (an index slip), so its pins run in a child
# process: a crash there is a caught mistake, not a crash of the test run.
_CHILD = """
import ctypes, json, sys
import oracle
from tests import test_oracle_mutants as m
oracle._lib = oracle._bind(ctypes.CDLL(sys.argv[1]))
print("CAUGHT " + json.dumps(m.run_pins()))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name!r} not found in oracle.c"
    so = str(tmp_path / "mutant.so")
    _compile(src.replace(old, new, 1), so)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CHILD, so], cwd=root, capture_output=True, text=True, timeout=600)
    if r.returncode < 0:
        return  # the slip crashed the oracle: caught
    assert r.returncode == 0, r.stderr[-2000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("CAUGHT ")][-1]
    caught = json.loads(line[len("CAUGHT "):])
    assert caught, f"no pin caught mutant {name!r}"
