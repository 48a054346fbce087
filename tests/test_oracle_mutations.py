"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a private copy of oracle/fa_oracle.c (a dropped term, a
wrong sign, index or offset, a swapped operand), builds it with gcc, and runs the pin suite
(tests/test_oracle.py) against that build in a subprocess: the suite has to fail.  Nothing
here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "fa_oracle.c")

MUTATIONS = {
    "drop_scale": ("double sj = scale * dot;", "double sj = dot;"),
    "causal_top_left": ("j > i + (Lkv - Lq)", "j > i"),
    "gqa_modulo_mapping": ("int64_t hk = h / G;\n      int64_t qoff",
                           "int64_t hk = h % Hkv;\n      int64_t qoff"),
    "mask_sign": ("sj += load_elem(mask", "sj -= load_elem(mask"),
    "lse_base2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "paged_slot_index": ("int64_t row = (page * Hkv + hk) * page_size + (t % page_size);",
                         "int64_t row = (page * Hkv + hk) * page_size;"),
    "mla_drop_rope": ("          dot += load_elem(q_pe, flat * Dr + d, dtype) * load_elem(kpe, row * Dr + d, dtype);\n",
                      ""),
    "merge_weight": ("double w = exp(x - total);", "double w = exp(x - m);"),
    "fp16_exponent_bias": ("ldexp((double)(1024 + f), e - 25)", "ldexp((double)(1024 + f), e - 24)"),
    "k_v_swapped": ("load_elem(k, (kbase + j) * Dk + d, dtype)", "load_elem(v, (kbase + j) * Dk + d, dtype)"),
    "no_max_shift": ("double p = exp(s[j] - m);", "double p = exp(s[j]);"),
    "no_max_shift_consistent": ("double p = exp(s[j] - m);", "double p = exp(s[j]);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new)
    if name == "no_max_shift_consistent":
        # exp without the max shift, with the lse made consistent with it: exact for small
        # scores, so only the large-score closed form can notice (it overflows).
        mutated = mutated.replace("*lse = m + log(l);", "*lse = log(l);")
    c_path = tmp_path / "fa_oracle_mut.c"
    c_path.write_text(mutated)
    so_path = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", str(so_path),
                           str(c_path), "-lm"])
    env = dict(os.environ, FA_ORACLE_LIB=str(so_path), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"pins did not catch mutation {name}:\n{r.stdout[-2000:]}"
