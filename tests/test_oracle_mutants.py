"""Plants plausible mistakes in copies of the oracle's C source and checks that the pins
catch every one of them: evidence that the pins constrain each part of the oracle (scale,
softmax normalisation, LSE, the P.V contraction, each backward product).  The mistakes are
planted on the CPU, in temporary copies; the committed oracle is untouched."""
import os

import pytest

import oracle
from _pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

# (name, text to replace, replacement, occurrence index)
MUTANTS = [
    ("scores_without_scale", "s[i * n + j] = scale * dot(q + i * d, k + j * d, d);",
     "s[i * n + j] = dot(q + i * d, k + j * d, d);", 0),
    ("softmax_not_normalised", "for (int64_t j = 0; j < n; ++j) p[j] /= sum;", "", 0),
    ("lse_missing_max", "return m + log(sum);", "return log(sum);", 0),
    ("pv_transposed_p", "const double pij = p[i * n + j];", "const double pij = p[j * n + i];", 0),
    ("ds_wrong_sign_of_D", "(dpij - dh[i])", "(dpij + dh[i])", 0),
    ("dq_missing_scale", "row[c] *= scale;", "(void)0;", 0),
    ("dk_uses_keys", "rk[c] += wk * qh[i * d + c];", "rk[c] += wk * kh[i * d + c];", 0),
    ("dv_uses_ds", "const double wk = ds[i * n + j], wv = p[i * n + j];",
     "const double wk = ds[i * n + j], wv = ds[i * n + j];", 0),
    ("dk_missing_scale", "rk[c] *= scale;", "(void)0;", 0),
    ("dp_uses_q", "const double dpij = dot(doh + i * d, vh + j * d, d);",
     "const double dpij = dot(doh + i * d, qh + j * d, d);", 0),
    ("rows_lse_missing_max", "return m + log(sum);", "return log(sum) + 0.0 * m;", 0),
    ("rows_bwd_dv_uses_ds", "rv[c] += pij * dout[i * d + c];", "rv[c] += dsij * dout[i * d + c];", 0),
    ("vector_sub", "c[i] = a[i] + b[i];", "c[i] = a[i] - b[i];", 0),
    ("vector_twice_a", "c[i] = a[i] + b[i];", "c[i] = a[i] + a[i];", 0),
    ("vector_in_double_then_halfway_up", "c[i] = a[i] + b[i];", "c[i] = (float)((double)a[i] + (double)b[i] + 1e-30);", 0),
]


def _mutate(text, old, new, occurrence):
    start = -1
    for _ in range(occurrence + 1):
        start = text.index(old, start + 1)
    return text[:start] + new + text[start + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, occ, tmp_path):
    with open(SRC) as f:
        text = f.read()
    assert old in text, f"mutation site for {name} not found"
    src = tmp_path / f"{name}.c"
    src.write_text(_mutate(text, old, new, occ))
    lib_path = str(tmp_path / f"lib{name}.so")
    oracle.compile_shared(str(src), lib_path)
    lib = oracle.load_library(lib_path)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
