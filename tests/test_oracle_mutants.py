"""Mutation check of the oracle pins (CPU only).

Each case plants one plausible mistake in a copy of the oracle's C source,
builds it, and runs the pin suite against that copy in a child process.  The
pins must reject every mutant; a mutant that survives means a pin is missing.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "msa_oracle.c")

MUTANTS = {
    "tie_break_to_higher_id": ("if (best < 0 || s[j] > s[best]) best = j;",
                               "if (best < 0 || s[j] >= s[best]) best = j;"),
    "no_causal_mask_in_scores": ("if ((int64_t)j * page + t > p) break;      /* causal */", ";"),
    "own_block_not_forced": ("pick[n_pick++] = own;                                  /* own block always kept */",
                             "pick[n_pick++] = (own > 0 && !taken[0]) ? 0 : own;"),
    "head_to_group_modulo": ("int32_t g = h / hpg;\n            int32_t n = 0;",
                             "int32_t g = h % G;\n            int32_t n = 0;"),
    "key_read_from_values": ("const uint16_t *kv = k_cache + (((size_t)tok_page[i] * page + tok_slot[i]) * G + g) * D;",
                             "const uint16_t *kv = v_cache + (((size_t)tok_page[i] * page + tok_slot[i]) * G + g) * D;"),
    "merge_weight_uses_max": ("double wgt = exp(l - total);", "double wgt = exp(l - m);"),
    "lse_in_base_two": ("return m + log(sum);", "return m + log2(sum);"),
    "inversion_rows_descending": ("blk_ent[cursor[key]++] = q * topk + s;",
                                  "blk_ent[blk_off[key + 1] - 1 - (cursor[key]++ - blk_off[key])] = q * topk + s;"),
    "row_len_not_clipped": ("if (vis > page) vis = page;\n", "\n"),
    "scale_dropped": ("logit[i] = dot * sm_scale;\n            }\n            double *o = out",
                      "logit[i] = dot;\n            }\n            double *o = out"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(before, after))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
                           "-o", str(lib), str(mutated), "-lm"])
    env = dict(os.environ, MSA_ORACLE_LIB=str(lib))
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"mutant {name} survived the pins:\n{res.stdout[-2000:]}"
