"""CPU-only: plant plausible mistakes in a copy of the oracle and check that
the pins catch every one of them.  The committed oracle is never modified;
each mutant is a temporary copy of its C source with one textual change."""
import os

import pytest

import oracle
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "linattn_oracle.c")

# (label, text in the source, replacement, expected occurrences)
MUTANTS = [
    ("eps dropped from the denominator", "den += p->eps;", "", 1),
    ("elu map without the +1", "x > 0.0 ? x + 1.0 : exp(x)", "x > 0.0 ? x : exp(x)", 1),
    ("relu map without eps", "(x > 0.0 ? x : 0.0) + eps", "(x > 0.0 ? x : 0.0)", 1),
    ("read-out with a transposed state",
     "num += fq[i] * S[(size_t)i * Dv + j];", "num += fq[i] * S[(size_t)(j % Dk) * Dv + (i % Dv)];", 1),
    ("outer product transposed",
     "S[(size_t)i * Dv + j] += fk[i] * vt[j];", "S[(size_t)i * Dv + j] += fk[j % Dk] * vt[i % Dv];", 2),
    ("interleaved GQA head map", "const int32_t h = hk * G + r;",
     "const int32_t h = r * Hkv + hk;", 1),
    ("per-dim decay index dropped", "J->decay[(tok * Hkv + hk) * Dk + i]",
     "J->decay[(tok * Hkv + hk) * Dk]", 1),
    ("decay sign flipped", "double a = exp(g);", "double a = exp(-g);", 1),
    ("delta residual sign", "u[j] = vt[j] - acc;", "u[j] = vt[j] + acc;", 1),
    ("beta layout ignored", "J->beta[tok * Hkv + hk] : J->beta[tok]", "J->beta[tok] : J->beta[tok]", 1),
    ("scale dropped", "yt[j] = p->scale * (num / den);", "yt[j] = (num / den);", 1),
    ("initial S ignored", "if (J->S0) memcpy(", "if (0) memcpy(", 1),
    ("initial Z ignored", "if (J->Z0) memcpy(", "if (0) memcpy(", 1),
    ("current token excluded from Z",
     "for (int32_t i = 0; i < Dk; ++i) Z[i] += fk[i];\n        }",
     "for (int32_t i = 0; i < Dk; ++i) Z[i] += 0.0 * fk[i];\n        }", 1),
    ("final state not written", "if (J->S_out) memcpy(", "if (0) memcpy(", 1),
    ("masked causal step still updates the state",
     "            continue;\n        }\n        if (J->causal) {", "        }\n        if (J->causal) {", 1),
    ("masked keys kept in the non-causal sums",
     "if (J->mask && !J->mask[b * T + t]) continue; /* invalid key/value */", "", 1),
    ("mask read at the wrong batch row", "if (J->mask && !J->mask[tok]) {", "if (J->mask && !J->mask[t]) {", 1),
]


@pytest.mark.parametrize("label,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, label, old, new, count):
    src = open(SRC).read()
    assert src.count(old) == count, f"mutation anchor for '{label}' not found as expected"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    so = str(tmp_path / "mutant.so")
    oracle.build(str(mutated), so)
    lib = oracle.load(so)
    failed = pins.run_all(lib)
    assert failed, f"no pin caught the planted mistake: {label}"


def test_committed_oracle_passes_every_pin():
    assert pins.run_all() == []
