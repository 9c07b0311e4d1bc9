"""Plant plausible mistakes in copies of the CPU oracle and check that the
pins catch each one.  The mistakes are planted in the oracle's C source on
the CPU (never in the GPU path): the source is copied, one textual
substitution is applied, the copy is compiled into a temporary directory
and every pin is run against it; at least one must fail."""
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

# (name, text to find, replacement); sites inside one_row unless the name
# starts with "probs_", which targets oracle_attn_probs
MUTANTS = [
    ("scale_dropped", "s[j] = jb->scale * dot;", "s[j] = dot;"),
    ("max_not_subtracted_in_sum", "l += exp(s[j] - m);", "l += exp(s[j]);"),
    ("wrong_sign_in_exponent", "const double p = exp(s[j] - m) / l;",
     "const double p = exp(m - s[j]) / l;"),
    ("not_normalised", "const double p = exp(s[j] - m) / l;",
     "const double p = exp(s[j] - m);"),
    ("value_row_of_query", "o_out[c] += p * V[j * d + c];", "o_out[c] += p * V[i * d + c];"),
    ("causal_off_by_one", "jb->causal ? i + 1 : N;", "jb->causal ? (i > 0 ? i : 1) : N;"),
    ("query_from_wrong_head", "const double *qi = jb->q + flat * d;",
     "const double *qi = jb->q + i * d;"),
    ("lse_without_max", "*lse_out = m + log(l);", "*lse_out = log(l);"),
    ("lse_log2", "*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    ("keys_from_first_head", "const double *K = jb->k + bh * N * d;",
     "const double *K = jb->k;"),
    ("probs_mask_reversed", "prow[j] = (j < nvis) ?", "prow[j] = (j > nvis) ?"),
    ("probs_not_normalised", "exp(s[j] - m) / l : 0.0;", "exp(s[j] - m) : 0.0;"),
    ("probs_scale_dropped", "s[j] = scale * dot;", "s[j] = dot;"),
]


def _function_span(src: str, name: str) -> tuple[int, int]:
    if name.startswith("probs_"):
        start = src.index("int oracle_attn_probs(")
        return start, len(src)
    return src.index("static void one_row("), src.index("static void *run_job(")


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, find, repl):
    src = open(SRC).read()
    a, b = _function_span(src, name)
    body = src[a:b]
    assert find in body, f"mutation site for {name} no longer in the oracle source"
    mutated = src[:a] + body.replace(find, repl, 1) + src[b:]
    c_path = tmp_path / f"{name}.c"
    so_path = tmp_path / f"{name}.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-std=c99", "-o", str(so_path),
                    str(c_path), "-lm", "-lpthread"], check=True)
    lib = oracle.load_library(str(so_path))
    failures = []
    for check in pins.ALL_CHECKS:
        try:
            check(lib=lib)
        except AssertionError:
            failures.append(check.__name__)
        except (RuntimeError, ValueError, FloatingPointError):
            failures.append(check.__name__)
    assert failures, f"no pin caught the planted mistake {name}"
