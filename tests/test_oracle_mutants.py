"""Planted mistakes in the oracle must fail at least one pin.

Each mutant is a copy of the oracle's C source with one plausible mistake
(an off-by-one in the key length, a dropped scale, a flipped sign, a wrong
GQA mapping, transposed strides, ...), compiled on the CPU into a temporary
library.  The pins run against it in a child process (a mutant may also
crash, which counts as caught).  The real oracle is never modified.
"""

import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "paged_decode_oracle.c")

MUTANTS = {
    "causal_off_by_one": ("n = (int64_t)a->seq_lens[s] - a->M + (t % a->M) + 1;",
                          "n = (int64_t)a->seq_lens[s] - a->M + (t % a->M);"),
    "varlen_left_search": ("if (a->qsl[mid + 1] <= t)", "if (a->qsl[mid + 1] < t)"),
    "varlen_klen_off_by_one": ("n = (int64_t)a->seq_lens[s] - q_len + (t - a->qsl[s]) + 1;",
                               "n = (int64_t)a->seq_lens[s] - q_len + (t - a->qsl[s]);"),
    "varlen_uniform_qlen": ("n = (int64_t)a->seq_lens[s] - q_len + (t - a->qsl[s]) + 1;",
                            "n = (int64_t)a->seq_lens[s] - a->M + (t - a->qsl[s]) + 1;"),
    "varlen_padding_kept": ("if (s >= a->num_seqs) return 0;",
                            "if (s >= a->num_seqs) s = a->num_seqs - 1;"),
    "window_off_by_one": ("*lo = n - a->window;", "*lo = n - a->window + 1;"),
    "gqa_modulo": ("int h = hq / G;", "int h = hq % a->Hkv;"),
    "dropped_scale": ("x[k - lo] = a->scale * dot;", "x[k - lo] = dot;"),
    "softmax_sign": ("double p = exp(x[k - lo] - m);", "double p = exp(m - x[k - lo]);"),
    "token_index": ("int64_t tok = k % a->P;", "int64_t tok = k / a->P;"),
    "half_exponent": ("v = ldexp((double)(f | 0x400), e - 25);", "v = ldexp((double)(f | 0x400), e - 24);"),
    "bf16_shift": ("uint32_t u = ((uint32_t)b) << 16;", "uint32_t u = ((uint32_t)b) << 15;"),
    "dropped_key": ("widen(a, qrow[d * a->q_s2]) * widen(a, kr[d * a->kv_sd])",
                    "widen(a, qrow[d * a->q_s2]) * widen(a, qrow[d * a->q_s2])"),
    "no_normalise": ("o[d] = (l > 0.0) ? acc[d] / l : 0.0;", "o[d] = acc[d];"),
    "values_from_keys": ("key_row(a, a->v, s, k, h)", "key_row(a, a->k, s, k, h)"),
    "window_ignored": ("if (a->window > 0 && n - a->window > 0)", "if (0)"),
    "page_ignored": ("int64_t phys = a->block_table[(int64_t)s * a->bt_stride + page];",
                     "int64_t phys = page;"),
    "empty_rows_clamp": ("if (n < 0) n = 0;", "if (n < 1) n = 1;"),
}

RUNNER = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle, oracle_pins
lib = oracle.load_library({lib!r})
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(lib)
    except Exception as e:
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
sys.exit(1 if failed else 0)
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not found exactly once: {old}"
    with tempfile.TemporaryDirectory() as d:
        csrc = os.path.join(d, "m.c")
        lib = os.path.join(d, "m.so")
        open(csrc, "w").write(src.replace(old, new))
        subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", lib, csrc, "-lm"])
        code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout}\n{r.stderr[-2000:]}"
