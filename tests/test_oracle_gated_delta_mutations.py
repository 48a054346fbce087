"""The gated-delta oracle's pins must catch plausible mistakes.

Each case plants one mistake in a private copy of oracle/gdn_oracle.c (a flipped sign, a term
decayed that should not be, a dropped factor, a wrong head mapping, a transposed state, the
initial state ignored), builds it with gcc, and runs the pin suite
(tests/test_oracle_gated_delta.py) against that build in a subprocess: the suite has to fail.
Nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gdn_oracle.c")

UPDATE = "S[i * dk + j] = alpha * (S[i * dk + j] - bt * w[i] * kt[j]) + bt * vi * kt[j];"
MUTATIONS = {
    "decay_sign": ("const double alpha = exp(gd_load(", "const double alpha = exp(-gd_load("),
    "write_decayed_too": (UPDATE, "S[i * dk + j] = alpha * (S[i * dk + j] - bt * w[i] * kt[j] + bt * vi * kt[j]);"),
    "erase_not_decayed": (UPDATE, "S[i * dk + j] = alpha * S[i * dk + j] - bt * w[i] * kt[j] + bt * vi * kt[j];"),
    "erase_without_beta": (UPDATE, "S[i * dk + j] = alpha * (S[i * dk + j] - w[i] * kt[j]) + bt * vi * kt[j];"),
    "erase_sign": (UPDATE, "S[i * dk + j] = alpha * (S[i * dk + j] + bt * w[i] * kt[j]) + bt * vi * kt[j];"),
    "scale_dropped": ("qt[j] = scale * gd_load(q, qk_row + j, dtype);",
                      "qt[j] = gd_load(q, qk_row + j, dtype);"),
    "head_modulo": ("hk = h / r;", "hk = h % Hk;"),
    "key_from_query": ("kt[j] = gd_load(k, qk_row + j, dtype);",
                       "kt[j] = gd_load(q, qk_row + j, dtype);"),
    "state_transposed_read": ("for (int64_t j = 0; j < dk; ++j) acc += S[i * dk + j] * qt[j];",
                              "for (int64_t j = 0; j < dk; ++j) acc += S[j * dv + i] * qt[j];"),
    "initial_state_ignored": ("S[i] = s0 ? s0[bh * dv * dk + i] : 0.0;", "S[i] = 0.0;"),
    "fp16_exponent_bias": ("ldexp((double)(1024 + f), e - 25)", "ldexp((double)(1024 + f), e - 24)"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found once"
    c_path = tmp_path / "gdn_oracle_mut.c"
    c_path.write_text(src.replace(old, new))
    so_path = tmp_path / "liboracle_gdn_mut.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", str(so_path),
                           str(c_path), "-lm"])
    env = dict(os.environ, GDN_ORACLE_LIB=str(so_path), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_gated_delta.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"pins did not catch mutation {name}:\n{r.stdout[-2000:]}"
