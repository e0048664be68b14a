"""The pins must catch plausible mistakes in the oracle.

Each case copies the oracle to a temporary folder, plants one mistake in its C
source (on the CPU only), and checks that the pin suite then fails.  The
mistakes are the ones a restatement of the routing article most plausibly
makes: weights from the biased score, a wrong group score, ties to the higher
index, a dropped scaling factor, selection without the bias, strided instead
of contiguous groups, gate and up swapped, no bf16 rounding of the SwiGLU
intermediate, a missing shared expert, a transposed down projection.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "weights_from_biased": ("float q = s[cand[a]] / den;", "float q = b[cand[a]] / den;"),
    "group_top1_only": ("g[j] = m1 + m2;", "g[j] = m1;"),
    "group_plus_extra_term": ("g[j] = m1 + m2;", "g[j] = m1 + m2 + b[j * GS];"),
    "ties_to_higher_index": ("return va > vb || (va == vb && ia < ib);",
                             "return va > vb || (va == vb && ia > ib);"),
    "no_scaling_factor": ("w[(size_t)t * K + a] = q * c->rsf;", "w[(size_t)t * K + a] = q;"),
    "selection_without_bias": ("b[e] = s[e] + (bias ? bias[e] : 0.0f);", "b[e] = s[e];"),
    "strided_groups": ("float v = b[j * GS + q];", "float v = b[q * G + j];"),
    "gate_up_swapped": ("double act = G / (1.0 + exp(-G)) * U;", "double act = U / (1.0 + exp(-U)) * G;"),
    "no_bf16_intermediate": ("a[i] = round_act ? orc_bf16_value(orc_bf16_round((float)act)) : act;",
                             "a[i] = act;"),
    "no_shared_expert": ("if (sgu && sd)\n", "if (0)\n"),
    "down_transposed": ("acc[h] += ai * orc_bf16_value(wd[h]);",
                        "acc[h] += ai * orc_bf16_value(Wd[(size_t)h * I + i]);"),
}


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    before, after = MUTATIONS[name]
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "tests"), tmp_path / "tests",
                    ignore=shutil.ignore_patterns("__pycache__", "test_oracle_mutations.py", "test_gpu*",
                                                  "test_zz*"))
    src_path = tmp_path / "oracle" / "moe_oracle.c"
    src = src_path.read_text()
    assert before in src, "mutation site moved: " + name
    src_path.write_text(src.replace(before, after))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, "planted mistake %r passed every pin:\n%s" % (name, r.stdout[-2000:])
