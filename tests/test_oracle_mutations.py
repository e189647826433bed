"""Plant plausible mistakes in a temporary copy of the oracle and check that
the pin suite fails for every one of them (dropped term, wrong sign, wrong
index, transposed operand, wrong GQA map, wrong segment rounding)."""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "oracle.c")

MUTANTS = {
    "lse_drops_max": ("*lse = m + log(z);", "*lse = log(z);"),
    "no_scale": ("s[t] = acc * p->scale;", "s[t] = acc;"),
    "exp_sign": ("s[t] = exp(s[t] - m);", "s[t] = exp(m - s[t]);"),
    "gqa_modulo": ("const int kvh = h / (p->num_q_heads / p->num_kv_heads);",
                   "const int kvh = h % p->num_kv_heads;"),
    "k_v_swapped": ("pool_index(p, blk[t], 1, kvh, slot[t], e));\n    }\n    *lse",
                    "pool_index(p, blk[t], 0, kvh, slot[t], e));\n    }\n    *lse"),
    "segment_floor": ("col += (len + B - 1) / B;", "col += len / B;"),
    "slot_off_by_one": ("slot[t] = (int32_t)(j % B);", "slot[t] = (int32_t)((j + 1) % B);"),
    "chain_leaf_first": ("for (int i = 0; i < n; ++i) out[i] = tmp[n - 1 - i];",
                         "for (int i = 0; i < n; ++i) out[i] = tmp[i];"),
    "weight_unnormalised": ("double w = s[t] / z;", "double w = s[t];"),
    "causal_off_by_one": ("const long long nvis = ntok - q_len[r] + idx_of[row] + 1;",
                          "const long long nvis = ntok - q_len[r] + idx_of[row];"),
    "causal_no_mask": ("const long long nvis = ntok - q_len[r] + idx_of[row] + 1;",
                       "const long long nvis = ntok;"),
    "chunk_row_swap": ("attend_one(p, q, row, h, blk, slot, nvis,",
                       "attend_one(p, q, (row + 1) % Q, h, blk, slot, nvis,"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mut = tmp_path / "oracle.c"
    mut.write_text(src.replace(old, new))
    env = dict(os.environ, ORACLE_SRC_OVERRIDE=str(mut))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_pins.py")],
                       env=env, capture_output=True, text=True, timeout=600,
                       cwd=os.path.dirname(HERE))
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
