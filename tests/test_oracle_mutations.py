"""The oracle's pins must be able to fail: plant one plausible mistake at a
time (at every place the mutated line occurs) in a copy of the C oracle (a dropped term, a wrong index or operator, a
wrong rounding rule), build that copy, and check that the pin suite rejects it.
CPU only; nothing here touches the CUDA path."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MUTATIONS = {
    "rank_by_modulo": ("return (int)(e / m);", "return (int)(e % m);"),
    "prefix_drops_running_sum": ("rank_prefix[r + 1] = rank_prefix[r] + num_tokens_per_rank[r];",
                                 "rank_prefix[r + 1] = num_tokens_per_rank[r];"),
    "last_lane_owns_rank": ("for (int jj = 0; jj < j; ++jj)", "for (int jj = j + 1; jj < k; ++jj)"),
    "rows_not_in_token_order": ("token_dst_row[idx] = rank_prefix[r] + next[r];",
                                "token_dst_row[idx] = rank_prefix[r + 1] - 1 - next[r];"),
    "bf16_ties_away": ("if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))",
                       "if (dropped >= 0x8000u)"),
    "e4m3_exponent_off_by_one": ("code = (e + 6) * 8 + n;", "code = (e + 7) * 8 + n;"),
    "fp8_wrong_scale": ("float s = amax / 448.0f;", "float s = amax / 240.0f;"),
    "localised_index_wrong": ("e - (int64_t)r * m : -1;", "e - (int64_t)r : -1;"),
    "combine_descending": ("rows[b - 1] > rows[b]; --b)", "rows[b - 1] < rows[b]; --b)"),
    "weights_not_masked": ("(local && topk_weights) ?", "(topk_weights) ?"),
    "weighted_combine_unfused": ("acc = fmaf(w, oracle_bf16_to_float(partial[(int64_t)rows[i] * H + h]), acc);",
                                 "acc = acc + w * oracle_bf16_to_float(partial[(int64_t)rows[i] * H + h]);"),
    "combined_weights_wrong_lane": ("acc += recv_topk_weights[(int64_t)rows[i] * k + j];",
                                    "acc += recv_topk_weights[(int64_t)rows[i] * k + (k - 1 - j)];"),
    "expand_counter_from_zero": ("for (int e = 0; e < E; ++e) count[e] = expert_prefix[e];",
                                 "for (int e = 0; e < E; ++e) count[e] = 0;"),
    "expand_metadata_whole_rank": ("recv_topk_idx[row * k + jj] = (jj == j) ? e - (int64_t)r * m : -1;",
                                   "recv_topk_idx[row * k + jj] = (topk_idx[(int64_t)t * k + jj] >= 0 && "
                                   "topk_idx[(int64_t)t * k + jj] / m == r) ? topk_idx[(int64_t)t * k + jj] - "
                                   "(int64_t)r * m : -1;"),
    "expand_weight_of_other_entries": ("(jj == j && topk_weights) ? topk_weights[(int64_t)t * k + j] : 0.0f;",
                                       "(topk_weights) ? topk_weights[(int64_t)t * k + jj] : 0.0f;"),
    "fp8_combine_fused": ("                float v = oracle_e4m3_to_float(codes[(int64_t)rows[i] * H + h]) * s;\n                acc = acc + v;",
                          "                acc = fmaf(oracle_e4m3_to_float(codes[(int64_t)rows[i] * H + h]), s, acc);"),
    "fp8_combine_wrong_block_scale": ("float s = scales[(int64_t)rows[i] * nb + h / 128];",
                                      "float s = scales[(int64_t)rows[i] * nb + (h / 128 + 1) % nb];"),
    "expand_source_token_off_by_one": ("            recv_src_idx[row] = t;\n            for (int jj = 0;",
                                       "            recv_src_idx[row] = t + 1;\n            for (int jj = 0;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = tmp_path / "moe_oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-o", str(lib),
                    str(mutated), "-lm"], check=True)
    env = dict(os.environ, MOE_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutation {name}:\n{r.stdout[-2000:]}"
