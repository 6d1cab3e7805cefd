"""The pins are sharp: plant one plausible mistake at a time in a copy of
the oracle's source (a dropped term, a wrong sign, a wrong index, a
transposed operand, a stale carry) and check that some pin fails."""
import os
import shutil

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "m3_oracle.c")

# (name, text to find, replacement) — each replacement is one plausible slip
MUTANTS = [
    ("drop_trapezoid_term", "+ bscale * alpha[k] * uprev[i]", ""),
    ("trapezoid_term_without_decay", "bscale * alpha[k] * uprev[i]", "bscale * uprev[i]"),
    ("trapezoid_uses_current_token", "bscale * alpha[k] * uprev[i]", "bscale * alpha[k] * u[i]"),
    ("gamma_uses_one_minus_lam", "const double g = lmt * dtt;", "const double g = (1.0 - lmt) * dtt;"),
    ("beta_uses_lam", "const double bscale = (1.0 - lmt) * dtt;", "const double bscale = lmt * dtt;"),
    ("rotation_sign", "(Ah + I * rd(theta", "(Ah - I * rd(theta"),
    ("decay_sign", "cexp(dtt * (Ah +", "cexp(dtt * (-Ah +"),
    ("no_conjugate_on_C", "creal(conj(ch) *", "creal(ch *"),
    ("conjugate_on_B", "acc += bh *", "acc += conj(bh) *"),
    ("pairing_index", "I * rd(B, b_off + (int64_t)r * N + 2 * k + 1, dtype)",
     "I * rd(B, b_off + (int64_t)r * N + (2 * k + 3) % N, dtype)"),
    ("mimo_rank_mixup_in_u", "rd(x, x_off + (int64_t)r * P + p, dtype)",
     "rd(x, x_off + (int64_t)((r + 1) % R) * P + p, dtype)"),
    ("skip_term_rank0_only", "Dh * rd(x, xo + (int64_t)r * P + p, dtype)", "Dh * rd(x, xo + p, dtype)"),
    ("drop_skip_term", "acc + Dh * rd(x, xo + (int64_t)r * P + p, dtype)", "acc"),
    ("carry_from_first_token", "const int64_t t = un->ntok - 1;", "const int64_t t = 0;"),
    ("initial_carry_ignored", "outer(R, P, N, prevB, 0, prevx, 0, M3O_F64, uprev);",
     "outer(R, P, N, prevB, 0, prevx, 0, M3O_F64, uprev); for (int64_t j = 0; j < (int64_t)K * P; ++j) uprev[j] = 0;"),
    ("theta_index_off_by_one", "rd(theta, qo + k, dtype)", "rd(theta, qo + (k + 1) % K, dtype)"),
]


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, find, repl):
    src = open(SRC).read()
    assert find in src, f"mutation site for {name} not found"
    mutated = src.replace(find, repl, 1)
    p = tmp_path / "mut.c"
    p.write_text(mutated)
    so = str(tmp_path / "libmut.so")
    oracle.compile_lib(str(p), so)
    lib = oracle.load(so)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"


def test_unmutated_passes_all():
    lib = oracle.load()
    for pin in pins.ALL_PINS:
        pin(lib)
