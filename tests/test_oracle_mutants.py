"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of oracle/hq_oracle.c (on the CPU),
builds the copy, and runs tests/test_oracle.py against it in a subprocess:
at least one pin has to fail.  A mistake that changes only the rounding order
(not the exact arithmetic) is not a mistake the pins are meant to see and is
not listed.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "hq_oracle.c")

MUTANTS = {
    "butterfly_difference_sign": ("float d = a - b;", "float d = b - a;"),
    "hadamard_scale_off_by_one_ulp": ("0x3E3504F3u", "0x3E3504F4u"),
    "signs_ignored": ("return ((signs[k / 32] >> (k % 32)) & 1u) ? -1.0f : 1.0f;", "return 1.0f;"),
    "missing_overall_scale": ("out[b * OR_BLOCK + j] = u[j] * c;", "out[b * OR_BLOCK + j] = u[j];"),
    "round_half_away": ("float r = rintf(x);", "float r = roundf(x);"),
    "zero_point_sign_in_gemm": ("- (int64_t)zeros[(size_t)n * NG + g];", "+ (int64_t)zeros[(size_t)n * NG + g];"),
    "range_not_widened_to_zero": ("float lo = 0.0f, hi = 0.0f, scale, z;", "float lo = w[0], hi = w[0], scale, z;"),
    "zero_point_from_wrong_sign": ("z = or_round_clamp(-lo / scale, 0.0f, 15.0f);",
                                   "z = or_round_clamp(lo / scale, 0.0f, 15.0f);"),
    "asym_divisor_16": ("scale = (hi - lo) / 15.0f;", "scale = (hi - lo) / 16.0f;"),
    "sym_divisor_128": ("scale = a / 127.0f;", "scale = a / 128.0f;"),
    "act_absmax_signed": ("float t = fabsf(u[k]);", "float t = u[k];"),
    "group_sum_drops_last": ("for (k = g * G; k < (g + 1) * G; ++k) t += q[k];",
                             "for (k = g * G; k < (g + 1) * G - 1; ++k) t += q[k];"),
    "activation_transposed": ("int64_t a = qx[(size_t)m * K + k];", "int64_t a = qx[(size_t)k * M + m];"),
    "epilogue_drops_terms": ("acc = acc + t;", "acc = t;"),
    "epilogue_wrong_group_scale": ("float t = scales[(size_t)n * NG + g] * p;",
                                   "float t = scales[(size_t)n * NG + (g + 1) % NG] * p;"),
    "epilogue_drops_row_scale": ("Y[(size_t)m * N + n] = sx[m] * acc;", "Y[(size_t)m * N + n] = acc;"),
    "splitmix_gamma": ("0x9E3779B97F4A7C15ULL", "0x9E3779B97F4A7C16ULL"),
    "argmax_ties_last_index": ("if (isnan(a) || a > b) best = v;", "if (isnan(a) || a >= b) best = v;"),
    "tree_ignores_parent_validity": ("valid[i] = valid[p] && tokens[i] == g[p];", "valid[i] = tokens[i] == g[p];"),
    "tree_compares_own_greedy": ("valid[i] = valid[p] && tokens[i] == g[p];", "valid[i] = valid[p] && tokens[i] == g[i];"),
    "tree_ties_highest_index": ("if (valid[i] && depth[i] > depth[best]) best = i;",
                                "if (valid[i] && depth[i] >= depth[best]) best = i;"),
    "tree_bonus_from_parent": ("*bonus = g[best];", "*bonus = g[best > 0 ? parent[best] : 0];"),
    "half_exponent_bias": ("v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);"),
    "half_subnormal_scale": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    "attn_node_does_not_see_itself": ("vis[(size_t)i * M + i] = 1;", "vis[(size_t)i * M + i] = (i == 0);"),
    "attn_sees_every_tree_node": ("if (vis[(size_t)i * M + j]) pos[n++] = L + j;", "pos[n++] = L + j;"),
    "attn_walk_stops_at_parent": ("vis[(size_t)i * M + p] = 1;\n            cur = p;",
                                  "vis[(size_t)i * M + p] = 1;\n            break;"),
    "attn_cache_drops_last_position": ("for (int t = 0; t < L; ++t) pos[n++] = t;",
                                       "for (int t = 0; t + 1 < L; ++t) pos[n++] = t;"),
    "attn_ignores_scale": ("s[a] = scale * dot;", "s[a] = dot;"),
    "attn_kv_head_modulo": ("const int i = r / Hq, h = r % Hq, hk = h / G;",
                            "const int i = r / Hq, h = r % Hq, hk = h % Hkv;"),
    "delta_forgets_gate": ("S[(size_t)r * D + c] = alpha * (S[(size_t)r * D + c] - beta * u[r] * (double)k[c]) +",
                           "S[(size_t)r * D + c] = (S[(size_t)r * D + c] - beta * u[r] * (double)k[c]) +"),
    "delta_no_erase": ("- beta * u[r] * (double)k[c]) +", "- 0.0 * u[r] * (double)k[c]) +"),
    "delta_write_unscaled": ("beta * (double)v[r] * (double)k[c];", "(double)v[r] * (double)k[c];"),
    "delta_chain_skips_root": ("        while (cur > 0) {\n            const int p = parent[cur];\n            if (p < 0 || p >= cur) break;\n            chain[n++] = p;",
                               "        while (cur > 1) {\n            const int p = parent[cur];\n            if (p < 0 || p >= cur) break;\n            chain[n++] = p;"),
    "delta_output_transposed": ("for (int c = 0; c < D; ++c) t += S[(size_t)rr * D + c] * (double)qi[c];",
                                "for (int c = 0; c < D; ++c) t += S[(size_t)c * D + rr] * (double)qi[c];"),
    "delta_commit_skips_root": ("for (int a = -1; a < n_accept; ++a) {", "for (int a = 0; a < n_accept; ++a) {"),
    "commit_overwrites_root": ("memcpy(c + ((size_t)h * cap + L + 1 + d) * D,", "memcpy(c + ((size_t)h * cap + L + d) * D,"),
    "commit_reads_parent_row": ("c + ((size_t)h * cap + L + path[d]) * D, sizeof", "c + ((size_t)h * cap + L + path[d] - 1) * D, sizeof"),
    "attn_softmax_unnormalized": ("o[d] = num / den;", "o[d] = num;"),
    "attn_values_from_keys": ("num += s[a] * or_half_to_double(v[((size_t)hk * cap + pos[a]) * D + d]);",
                              "num += s[a] * or_half_to_double(k[((size_t)hk * cap + pos[a]) * D + d]);"),
    "attn_query_of_kv_head": ("const uint16_t *qr = q + ((size_t)i * Hq + h) * D;",
                              "const uint16_t *qr = q + ((size_t)i * Hq + hk) * D;"),
    "delta_chain_applied_leaf_first": ("for (int a = n - 1; a >= 0; --a) {", "for (int a = 0; a < n; ++a) {"),
    "delta_gate_scales_write": ("S[(size_t)r * D + c] = alpha * (S[(size_t)r * D + c] - beta * u[r] * (double)k[c]) +\n                                   beta * (double)v[r] * (double)k[c];",
                                "S[(size_t)r * D + c] = alpha * (S[(size_t)r * D + c] - beta * u[r] * (double)k[c] +\n                                   beta * (double)v[r] * (double)k[c]);"),
    "delta_commit_path_reversed": ("const int j = a < 0 ? 0 : path[a];", "const int j = a < 0 ? 0 : path[n_accept - 1 - a];"),
    "delta_commit_skips_last": ("for (int a = -1; a < n_accept; ++a) {", "for (int a = -1; a + 1 < n_accept; ++a) {"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "m.c")
        so = os.path.join(d, "m.so")
        open(c, "w").write(mutated)
        subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", c, "-o", so, "-lm"],
                       check=True)
        env = dict(os.environ, HQ_ORACLE_TEST_LIB=so)
        r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"), "-x",
                            "-q", "-p", "no:cacheprovider", "-k", "not openmp"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 1, f"{name}: pins did not fail (rc={r.returncode})\n{r.stdout[-2000:]}"
        assert "failed" in r.stdout
