"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of ``oracle/gdn_oracle.c`` (a dropped term, a
flipped sign, a wrong index), compiles the copy with gcc into a temporary directory and
runs the pins of ``test_oracle_pins.py`` against it. At least one pin must fail. The
real oracle is never modified.
"""
import inspect
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.oracle.__file__), "gdn_oracle.c")

MUTATIONS = [
    ("delta_sign", "*s = alpha * (*s - bt * kt[i] * x[j])", "*s = alpha * (*s + bt * kt[i] * x[j])"),
    ("drop_decay", "*s = alpha * (*s - bt * kt[i] * x[j])", "*s = (*s - bt * kt[i] * x[j])"),
    ("drop_beta_write", "+ bt * kt[i] * vt[j];", "+ kt[i] * vt[j];"),
    ("drop_scale", "out[(size_t)t * Dv + j] = c->scale * acc;", "out[(size_t)t * Dv + j] = acc;"),
    ("read_with_key", "acc += qt[i] * St[(size_t)i * Dv + j];", "acc += kt[i] * St[(size_t)i * Dv + j];"),
    ("gqa_tiled", "const int kh = h / (c->Hv / c->Hk);\n    const int S = c->S, Dk = c->Dk, Dv = c->Dv;\n",
     "const int kh = h % c->Hk;\n    const int S = c->S, Dk = c->Dk, Dv = c->Dv;\n"),
    ("chunk_drop_gamma_q", "c->scale * (exp(gam[r]) * qs + pu)", "c->scale * (qs + pu)"),
    ("chunk_pu_sign", "c->scale * (exp(gam[r]) * qs + pu)", "c->scale * (exp(gam[r]) * qs - pu)"),
    ("chunk_A_beta_index", "(j < r) ? bc[r] * kk * d", "(j < r) ? bc[j] * kk * d"),
    ("chunk_state_decay", "double acc = exp(gl) * St[(size_t)i * Dv + n];",
     "double acc = St[(size_t)i * Dv + n];"),
    ("inverse_transposed", "acc -= A[(size_t)r * n + m] * T[(size_t)m * n + j];",
     "acc -= A[(size_t)m * n + r] * T[(size_t)m * n + j];"),
    ("sigmoid_sign", "return 1.0 / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(x));"),
    ("softplus_log", "log1p(exp(-fabs(x)))", "log(exp(-fabs(x)))"),
    ("decode_head_major", "const int h = (int)(bh % c->H);", "const int h = (int)(bh / (c->BH / c->H));"),
    ("decode_drop_gamma", "y[j] = o[j] * rr * c->norm_weight[j] * silu;", "y[j] = o[j] * rr * silu;"),
    ("decode_gate_linear", "const double silu = zr[j] * sigmoid(zr[j]);", "const double silu = zr[j];"),
    ("decode_l2_unnormalised_k", "kn[i] = kr[i] * rk;", "kn[i] = kr[i];"),
]

# every pin, with the parameters of the parametrised ones
_PIN_CALLS = []
for _name, _fn in inspect.getmembers(pins, inspect.isfunction):
    if not _name.startswith("test_"):
        continue
    marks = getattr(_fn, "pytestmark", [])
    params = [m for m in marks if m.name == "parametrize"]
    if not params:
        _PIN_CALLS.append((_name, _fn, {}))
        continue
    argnames, values = params[0].args
    names = [a.strip() for a in argnames.split(",")]
    for val in values:
        val = val if isinstance(val, tuple) else (val,)
        _PIN_CALLS.append((_name, _fn, dict(zip(names, val))))


def _run_pins(orc):
    failed = []
    for name, fn, kw in _PIN_CALLS:
        try:
            fn(orc, **kw)
        except AssertionError:
            failed.append(name)
        except (ValueError, FloatingPointError):
            failed.append(name)
    return failed


def test_real_oracle_passes_every_pin(oracle_mod):
    assert _run_pins(oracle.default()) == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", str(mutated),
                    "-o", str(lib), "-lm"], check=True)
    failed = _run_pins(oracle.Oracle(str(lib)))
    assert failed, f"no pin caught the planted mistake {name}"
