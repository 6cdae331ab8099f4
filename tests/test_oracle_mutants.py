"""The oracle's whole-pass pins are strong enough: each plausible slip, planted by hand in a
copy of the oracle's C source on the CPU, makes the closed-form test fail.

A mutant is ``pe_oracle.c`` with one exact text replacement (the test fails loudly if the
text is no longer there), compiled to a temporary library and swapped in for the oracle's
own for the duration of one check.  Nothing here touches the CUDA path.
"""

import os
import shutil

import pytest

import oracle
from test_oracle_pins import closed_form_failures, closed_form_pass_checks

_Q_ROPE = "oc_rope(q + (size_t)r * qd + (size_t)h * hd, hd, position[r], cfg->rope_theta);"
_K_ROPE = "oc_rope(kn + (size_t)r * kvd + (size_t)g * hd, hd, position[r], cfg->rope_theta);"
_V_ROPE = "oc_rope(vn + (size_t)r * kvd + (size_t)g * hd, hd, position[r], cfg->rope_theta);"
_SWIGLU = "oc_silu(gu[(size_t)r * 2 * F + f]) * gu[(size_t)r * 2 * F + F + f]"
_Q_COPY = "memcpy(q + (size_t)r * qd, src, sizeof(double) * qd);"
_K_COPY = "memcpy(kn + (size_t)r * kvd, src + qd, sizeof(double) * kvd);"

# name -> (replacements, checks that must fail)
MUTANTS = {
    "rope_on_v_too": ([(_K_ROPE, "{ " + _K_ROPE + " " + _V_ROPE + " }")], {"v_block_unrotated", "attention_q_rope"}),
    "q_rope_at_p_plus_1": ([(_Q_ROPE, _Q_ROPE.replace("position[r]", "position[r] + 1"))], {"attention_q_rope"}),
    "k_rope_at_p_plus_1": ([(_K_ROPE, _K_ROPE.replace("position[r]", "position[r] + 1"))], {"k_block_rope"}),
    "q_not_rotated": ([(_Q_ROPE, "(void)0;")], {"attention_q_rope"}),
    "silu_on_up_half": ([(_SWIGLU, "oc_silu(gu[(size_t)r * 2 * F + F + f]) * gu[(size_t)r * 2 * F + f]")],
                        {"swiglu_roles"}),
    "k_block_before_q": ([(_Q_COPY, "memcpy(q + (size_t)r * qd, src + kvd, sizeof(double) * qd);"),
                          (_K_COPY, "memcpy(kn + (size_t)r * kvd, src, sizeof(double) * kvd);")],
                         {"k_block_rope"}),
    "no_residual_after_mlp": ([("for (size_t i = 0; i < (size_t)n * d; ++i) x[i] += tmp[i];\n    }",
                                "for (size_t i = 0; i < (size_t)n * d; ++i) x[i] = tmp[i];\n    }")],
                              {"residual_stream"}),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_fails_closed_form_pins(name, source, tmp_path, monkeypatch):
    edits, must_fail = MUTANTS[name]
    src = source
    for old, new in edits:
        assert src.count(old) == 1, f"mutation site not found exactly once: {old!r}"
        src = src.replace(old, new)
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(src)
    mutant = oracle.load_library(oracle.compile_source(path, os.path.join(tmp_path, "libmutant.so")))
    monkeypatch.setattr(oracle, "_lib", mutant)
    failed = set(closed_form_failures(closed_form_pass_checks()))
    assert must_fail <= failed, f"{name}: pins that still pass {sorted(must_fail - failed)}"


def test_unmutated_source_passes(source, tmp_path, monkeypatch):
    """Control: the same compile-and-swap route with the source unchanged passes every check."""
    path = os.path.join(tmp_path, "same.c")
    with open(path, "w") as f:
        f.write(source)
    monkeypatch.setattr(oracle, "_lib", oracle.load_library(oracle.compile_source(path, os.path.join(tmp_path,
                                                                                                     "libsame.so"))))
    assert closed_form_failures(closed_form_pass_checks()) == []
