"""The pins are sharp: plant one plausible mistake at a time in a copy of
the oracle's source (a dropped term, a wrong sign, a wrong index, a
transposed operand, a stale carry) and check that some pin fails."""
import os

import numpy as np
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


# The fused prologue lives in the oracle's Python wrapper: plant slips there
# (monkeypatched for one test) and check that a prologue pin fails.
def _prologue_pins():
    import test_oracle_prologue as t

    return [t.test_softplus_closed_forms, t.test_softplus_matches_the_generators_formula,
            t.test_bias_enters_before_softplus, t.test_rms_normalize_definition,
            lambda: t.test_norm_undoes_a_positive_scale_of_each_row(2),
            t.test_prologue_on_already_normalised_inputs_is_the_plain_scan]


def _apply_prologue_variant(bias_after=False, skip_prev_B=False):
    def f(inp, dtype, *, dt_softplus=False, bc_norm=False, dt_bias=None):
        out = {k: (v if (v is None or k in ("A", "D", "h0", "dt_bias")) else oracle._widen(v, dtype))
               for k, v in inp.items()}
        bias = 0.0 if dt_bias is None else np.asarray(dt_bias, np.float64)
        if dt_softplus:
            out["dt"] = oracle.softplus(out["dt"]) + bias if bias_after else oracle.softplus(out["dt"] + bias)
        if bc_norm:
            for k in ("B", "C") if skip_prev_B else ("B", "C", "prev_B"):
                if out.get(k) is not None:
                    out[k] = oracle.rms_normalize(out[k])
        return out
    return f


def _rms(axis=-1, sqrt=True, mean=True):
    def f(a, eps=1e-6):
        a = np.asarray(a, np.float64)
        ms = (np.mean if mean else np.sum)(a * a, axis=axis, keepdims=True) + eps
        return a / (np.sqrt(ms) if sqrt else ms)
    return f


PROLOGUE_MUTANTS = {
    "rms_sum_not_mean": ("rms_normalize", _rms(mean=False)),
    "rms_over_wrong_axis": ("rms_normalize", _rms(axis=-2)),
    "rms_without_sqrt": ("rms_normalize", _rms(sqrt=False)),
    "softplus_without_abs": ("softplus", lambda z: np.maximum(z, 0.0) + np.log1p(np.exp(-np.asarray(z, float)))),
    "softplus_as_relu": ("softplus", lambda z: np.maximum(np.asarray(z, float), 0.0)),
    "bias_after_softplus": ("apply_prologue", _apply_prologue_variant(bias_after=True)),
    "carried_B_not_normalised": ("apply_prologue", _apply_prologue_variant(skip_prev_B=True)),
}


@pytest.mark.parametrize("name", list(PROLOGUE_MUTANTS))
def test_prologue_mutant_is_caught(monkeypatch, name):
    attr, fn = PROLOGUE_MUTANTS[name]
    monkeypatch.setattr(oracle, attr, fn)
    failed = []
    for pin in _prologue_pins():
        try:
            pin()
        except AssertionError:
            failed.append(getattr(pin, "__name__", "pin"))
    assert failed, f"no prologue pin caught {name}"
