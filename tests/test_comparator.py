"""Comparator self-test: 1-ULP corruption at three offsets must be seen and localised
(vllm.cpp PR #425, EVIDENCE section, 'Comparator self-test' paragraph)."""
import json
import os

import numpy as np

import compare
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "comparator_selftest.json")


def test_comparator_detects_and_localises_one_ulp():
    g = json.load(open(GOLDEN))
    n = g["n_elements"]
    z = synth.normal(4242, np.arange(n, dtype=np.uint64)) * 0.1
    ref = synth.f32_to_bf16_bits(z.astype(np.float32))
    clean = compare.compare(ref.copy(), ref)
    assert clean.bitwise_pct == g["expect_bitwise_percent_clean"] and clean.max_abs == 0
    bad = ref.copy()
    for off in g["corrupt_offsets"]:
        bad[off] = np.uint16(int(bad[off]) + 1)   # one unit in the last place
    s = compare.compare(bad, ref)
    assert round(s.bitwise_pct, 4) == g["expect_bitwise_percent_corrupt"]
    assert s.differing.tolist() == g["corrupt_offsets"]
    ulp = max(abs(float(synth.bf16_bits_to_f32(bad[o:o + 1])[0] - synth.bf16_bits_to_f32(ref[o:o + 1])[0]))
              for o in g["corrupt_offsets"])
    assert s.max_abs == ulp > 0


def test_comparator_flags_nan():
    ref = np.zeros(8)
    got = synth.f32_to_bf16_bits(np.zeros(8, dtype=np.float32))
    got[3] = synth.BF16_NAN
    s = compare.compare(got, ref)
    assert not s.ok() and s.worst_index == 3
