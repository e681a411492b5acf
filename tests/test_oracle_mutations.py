"""The oracle pins catch plausible mistakes.

Each case compiles a copy of the oracle's C source with one deliberate slip
(on the CPU, in a temporary directory), points the oracle module at it, and
requires at least one pin of ``test_oracle_pins`` to fail.  The real oracle is
restored afterwards.
"""
import ctypes
import inspect
import os
import pathlib
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

_READ = """    if (o_row) {
        for (int64_t j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i < dk; ++i) acc += S[i * dv + j] * q[i];
            o_row[j] = acc * scale;
        }
    }
"""
_WRITE = """    for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += k[i] * d[j];
"""
_DECAY = """        const double a = exp(log_alpha[i]);
        for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= a;
"""

MUTATIONS = {
    "residual_sign": [("d[j] = beta * (v[j] - p);", "d[j] = beta * (v[j] + p);")],
    "beta_on_value_only": [("d[j] = beta * (v[j] - p);", "d[j] = beta * v[j] - p;")],
    "no_output_scale": [("o_row[j] = acc * scale;", "o_row[j] = acc;")],
    "read_before_write": [(_WRITE + "    /* read from the updated state */\n" + _READ,
                           _READ + _WRITE)],
    "decay_on_value_columns": [(_DECAY, """        for (int64_t j = 0; j < dv; ++j)
            S[i * dv + j] *= exp(log_alpha[j % dk]);
""")],
    "decay_after_prediction": [
        # predict on the undecayed state, then decay (the page's Gated DeltaNet order)
        ("""    /* decay: row i of S is multiplied by alpha_i */
    for (int64_t i = 0; i < dk; ++i) {
""" + _DECAY + """    }
""", ""),
        ("""        d[j] = beta * (v[j] - p);
    }
""", """        d[j] = beta * (v[j] - p);
    }
    for (int64_t i = 0; i < dk; ++i) {
""" + _DECAY + """    }
"""),
    ],
    "initial_state_ignored": [("    if (J->init_state)\n        memcpy", "    if (0)\n        memcpy")],
    "state_not_reset_between_units": [
        ("    else\n        memset(S, 0, (size_t)(dk * dv) * sizeof(double));\n", "\n")],
    "decay_by_log_not_exp": [("const double a = exp(log_alpha[i]);",
                              "const double a = 1.0 + log_alpha[i];")],
}


def _pin_functions():
    fns = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = inspect.signature(fn).parameters
        if "b" in params:
            fns.append((name, lambda fn=fn: fn(0.5)))
        elif not params:
            fns.append((name, fn))
    return fns


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_pins_catch_mutation(mutation, tmp_path):
    src = pathlib.Path(SRC).read_text()
    for old, new in MUTATIONS[mutation]:
        assert src.count(old) == 1, f"mutation {mutation} no longer matches the oracle source"
        src = src.replace(old, new)
    c_path = tmp_path / "mutant.c"
    c_path.write_text(src)
    so_path = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so_path),
                           str(c_path), "-lm", "-lpthread"])
    real = oracle._load()
    mutant = ctypes.CDLL(str(so_path))
    for fname in ("kda_oracle_prefill", "kda_oracle_decode_step"):
        getattr(mutant, fname).restype = getattr(real, fname).restype
        getattr(mutant, fname).argtypes = getattr(real, fname).argtypes
    caught = []
    try:
        oracle._lib = mutant
        for name, fn in _pin_functions():
            try:
                fn()
            except AssertionError:
                caught.append(name)
    finally:
        oracle._lib = real
    assert caught, f"no pin caught the mutation {mutation}"
