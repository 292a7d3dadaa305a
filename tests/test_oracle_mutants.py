"""The oracle's pins catch plausible mistakes in the oracle.

Each case below plants one mistake in a copy of ``oracle/attn_ref.c`` (a dropped
term, a wrong sign, a transposed or swapped operand, a wrong index or head map,
an off-by-one mask, a wrong bit order), builds the copy with the oracle's own
compiler flags, and runs the pin suite that covers that part of the oracle in a
child process that loads the copy (``ATTN_REF_LIB``).  The suite must fail:
a planted mistake that every pin let through would mean the oracle's
arithmetic there is not pinned.  Only the copies are changed; the oracle
itself, and anything the GPU tests use, is untouched.

Mistakes that leave the result unchanged in exact arithmetic (the max used for
stability taken as any other value, the order of a sum) are not plausible
failures of a pin and are not planted.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "attn_ref.c")

FWD = "tests/test_oracle.py"
BWD = "tests/test_oracle_backward.py"
MASK = "tests/test_oracle_blockmask.py"

# (name, pin suite, exact text in attn_ref.c, replacement)
MUTANTS = [
    ("normaliser_dropped", FWD, "pj = exp(s[j] - m) / l;", "pj = exp(s[j] - m);"),
    ("lse_sign", FWD, "*lse = m + log(l);", "*lse = m - log(l);"),
    ("lse_without_max", FWD, "*lse = m + log(l);", "*lse = log(l);"),
    ("scale_dropped", FWD, "s[j] = scale * acc;", "s[j] = acc;"),
    ("logits_against_values", FWD, "acc += bf16_bits_to_f64(q_row[d]) * bf16_bits_to_f64(kh[j * D + d]);",
     "acc += bf16_bits_to_f64(q_row[d]) * bf16_bits_to_f64(vh[j * D + d]);"),
    ("output_from_keys", FWD, "o_row[d] += pj * bf16_bits_to_f64(vh[j * D + d]);",
     "o_row[d] += pj * bf16_bits_to_f64(kh[j * D + d]);"),
    ("bottom_right_read_as_top_left", FWD, "last = (causal == 1) ? (i + Sk - Sq) : i;", "last = i;"),
    ("diagonal_key_excluded", FWD, "return last < 0 ? 0 : last + 1;", "return last < 0 ? 0 : last;"),
    ("kv_heads_interleaved", FWD, "const int64_t kvh = h / G;", "const int64_t kvh = h % Hkv;"),
    ("normaliser_without_shift", FWD, "l += exp(s[j] - m);", "l += exp(s[j]);"),
    ("bf16_widened_wrong", FWD, "uint32_t u = ((uint32_t)bits) << 16;", "uint32_t u = ((uint32_t)bits) << 15;"),
    ("empty_row_lse_zero", FWD, "*lse = -INFINITY;\n        return;", "*lse = 0.0;\n        return;"),
    ("ds_without_row_term", BWD, "const double ds = p[j] * (s[j] - Di);", "const double ds = p[j] * s[j];"),
    ("ds_sign", BWD, "const double ds = p[j] * (s[j] - Di);", "const double ds = p[j] * (Di - s[j]);"),
    ("dk_scale_dropped", BWD, "dkh[j * D + d] += scale64 * ds * bf16_bits_to_f64(qrow[d]);",
     "dkh[j * D + d] += ds * bf16_bits_to_f64(qrow[d]);"),
    ("dv_from_queries", BWD, "dvh[j * D + d] += p[j] * bf16_bits_to_f64(dorow[d]);",
     "dvh[j * D + d] += p[j] * bf16_bits_to_f64(qrow[d]);"),
    ("dq_against_values", BWD, "dq[r * D + d] += scale64 * ds * bf16_bits_to_f64(kh[j * D + d]);",
     "dq[r * D + d] += scale64 * ds * bf16_bits_to_f64(vh[j * D + d]);"),
    ("dp_against_keys", BWD, "dp += bf16_bits_to_f64(dorow[d]) * bf16_bits_to_f64(vh[j * D + d]);",
     "dp += bf16_bits_to_f64(dorow[d]) * bf16_bits_to_f64(kh[j * D + d]);"),
    ("row_term_without_p", BWD, "Di += p[j] * dp;", "Di += dp;"),
    ("mask_bit_order_reversed", MASK, "return (int)((mask_row[kb / 32] >> (kb % 32)) & 1u);",
     "return (int)((mask_row[kb / 32] >> (31 - kb % 32)) & 1u);"),
    ("per_head_masks_ignored", MASK, "const int64_t hm = (mask_heads == 1) ? 0 : h;", "const int64_t hm = 0;"),
    ("mask_ignored", MASK, "if (!mask_row) return 1;", "return 1;"),
]


@pytest.mark.parametrize("name,suite,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(name, suite, old, new, tmp_path):
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"the text to change for {name} must occur exactly once in attn_ref.c"
    mutant_c = tmp_path / f"attn_ref_{name}.c"
    mutant_c.write_text(src.replace(old, new))
    mutant_so = tmp_path / f"libattn_ref_{name}.so"
    subprocess.run(["gcc", "-std=c99", "-O2", "-fopenmp", "-shared", "-fPIC", str(mutant_c), "-o", str(mutant_so),
                    "-lm"], check=True, capture_output=True)
    env = dict(os.environ, ATTN_REF_LIB=str(mutant_so))
    proc = subprocess.run([sys.executable, "-m", "pytest", suite, "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    tail = "\n".join((proc.stdout + proc.stderr).strip().splitlines()[-5:])
    assert proc.returncode != 0, f"planted mistake '{name}' passed every pin of {suite}:\n{tail}"
    assert proc.returncode == 1, f"the pin run for '{name}' did not complete (exit {proc.returncode}):\n{tail}"


def test_unchanged_copy_passes_every_pin(tmp_path):
    """Control: a copy built and loaded the same way, with nothing planted, passes all three pin suites."""
    copy_so = tmp_path / "libattn_ref_copy.so"
    subprocess.run(["gcc", "-std=c99", "-O2", "-fopenmp", "-shared", "-fPIC", SRC, "-o", str(copy_so), "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, ATTN_REF_LIB=str(copy_so))
    proc = subprocess.run([sys.executable, "-m", "pytest", FWD, BWD, MASK, "-q", "-m", "not gpu",
                           "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    tail = "\n".join((proc.stdout + proc.stderr).strip().splitlines()[-5:])
    assert proc.returncode == 0, f"the unchanged copy failed a pin:\n{tail}"
