"""RED proofs for the pins: plant one plausible mistake at a time in a copy of
the oracle's C source (on the CPU, never in the product), compile it, and
check that at least one pin rejects the mutant.  Every mutation keeps all
memory accesses in bounds."""
import os
import subprocess

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

MUTANTS = {
    "kv_head_modulo": ("int g = h / G; /* contiguous grouping */", "int g = h % Hkv;"),
    "scale_dropped": ("s[t - t0] = scale * dot;", "s[t - t0] = dot;"),
    "window_off_by_one": ("? L - window : 0;", "? L - window + 1 : 0;"),
    "slot_shifted": ("int64_t slot = t % P;\n    const uint16_t *kr", "int64_t slot = (t + 1) % P;\n    const uint16_t *kr"),
    "normaliser_without_max": ("Z += exp(s[t - t0] - m);", "Z += exp(s[t - t0]);"),
    "lse_without_max": ("*lse = m + log(Z);", "*lse = log(Z);"),
    "merge_weight_uses_max": ("double w = exp(parts_lse[s] - lse);", "double w = exp(parts_lse[s] - m);"),
    "values_from_k_pool": ("const uint16_t *vr = v_pool", "const uint16_t *vr = k_pool"),
    "mla_rope_dropped": ("dot += bf16_to_double(qr[r]) * bf16_to_double(c[MLA_LAT + r]);", "dot += 0.0 * r;"),
    "mla_wuk_transposed": ("wk[(int64_t)d * MLA_LAT + j]", "wk[(int64_t)j * MLA_NOPE + d]"),
    "mla_wuv_transposed": ("wv[(int64_t)dv * MLA_LAT + j]", "wv[(int64_t)j * MLA_VDIM + dv]"),
    "mla_scale_dropped": ("s[t] = scale * dot;", "s[t] = dot;"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not unique"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    lib_path = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(lib_path),
                    str(src), "-lm"], check=True)
    lib = oracle.bind(str(lib_path))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError) as e:
            caught.append(f"{pin.__name__}: {str(e)[:80]}")
    assert caught, f"no pin rejects the mutant {name}"
