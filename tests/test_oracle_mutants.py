"""Plant plausible mistakes in copies of the oracle (CPU only) and show that the
pins catch every one of them.  The mutants are compiled to temporary libraries;
the real oracle is untouched."""
import ctypes
import os
import subprocess

import pytest

import oracle
import oracle_checks as oc

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

# (name, original text, mutated text)
MUTANTS = [
    ("dropped_beta_in_correction", "alpha * (sij - beta * u[i] * k[j])", "alpha * (sij - u[i] * k[j])"),
    ("wrong_sign_correction", "alpha * (sij - beta * u[i] * k[j])", "alpha * (sij + beta * u[i] * k[j])"),
    ("alpha_on_write_too", "alpha * (sij - beta * u[i] * k[j]) + beta * v[i] * k[j]",
     "alpha * (sij - beta * u[i] * k[j] + beta * v[i] * k[j])"),
    ("dropped_write_beta", "+ beta * v[i] * k[j]", "+ v[i] * k[j]"),
    ("left_multiplied_transition", "acc += S[(size_t)i * dk + j] * k[j];\n        u[i] = acc;",
     "acc += S[(size_t)j * dk + i] * k[j];\n        u[i] = acc;"),
    ("transposed_write", "+ beta * v[i] * k[j]", "+ beta * v[j % dv] * k[i % dk]"),
    ("readout_before_update",
     "gdn_step(dk, dv, S, kt, vt, alpha[t - 1], beta[t - 1], u);\n        if (o) gdn_readout(dk, dv, S, q + (size_t)(t - 1) * dk, o + (size_t)(t - 1) * dv);",
     "if (o) gdn_readout(dk, dv, S, q + (size_t)(t - 1) * dk, o + (size_t)(t - 1) * dv);\n        gdn_step(dk, dv, S, kt, vt, alpha[t - 1], beta[t - 1], u);"),
    ("readout_with_key", "gdn_readout(dk, dv, S, q + (size_t)(t - 1) * dk", "gdn_readout(dk, dv, S, k + (size_t)(t - 1) * dk"),
    ("ckpt_before_token", "ckpt_pos[next] == t", "ckpt_pos[next] == t + 1"),
    ("replay_floor", "(num + (int64_t)r_den - 1) / (int64_t)r_den", "num / (int64_t)r_den"),
    ("replay_round", "(num + (int64_t)r_den - 1) / (int64_t)r_den", "(num + (int64_t)r_den / 2) / (int64_t)r_den"),
    ("select_strict", "if (c[i] <= d) best = i;", "if (c[i] < d) best = i;"),
    ("select_first", "if (c[i] <= d) best = i;", "if (c[i] <= d && best < 0) best = i;"),
    ("stale_key", "const double* kt = k + (size_t)(t - 1) * dk;", "const double* kt = k + (size_t)(t > 1 ? t - 2 : 0) * dk;"),
]


@pytest.fixture(scope="module")
def src_text():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, src_text, name, orig, mut):
    assert orig in src_text, f"mutation anchor for {name} not found in the oracle source"
    path = tmp_path / "mut.c"
    path.write_text(src_text.replace(orig, mut, 1))
    so = tmp_path / f"lib_{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-ffp-contract=off", "-shared", "-o", str(so), str(path)],
                   check=True)
    real = oracle._load()
    lib = ctypes.CDLL(str(so))
    for f in ("gdn_oracle_replay_plan", "gdn_oracle_select_ckpt", "gdn_oracle_scan"):
        getattr(lib, f).argtypes = getattr(real, f).argtypes
        getattr(lib, f).restype = getattr(real, f).restype
    caught = []
    oracle._lib = lib
    try:
        for check in oc.ALL_CHECKS + [lambda: oc.check_replay_plan_exhaustive(2000)]:
            try:
                check()
            except (AssertionError, ValueError):
                caught.append(getattr(check, "__name__", "plan"))
    finally:
        oracle._lib = real
    assert caught, f"mutant {name} survived every pin"
