"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a private copy of the oracle's C source (on
the CPU, in a temporary directory), builds it, and runs the pin suite against
that build in a subprocess: the suite has to fail.
"""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

# (name, exact text in the oracle, replacement)
MUTANTS = [
    ("silu_sign", "h = g[j] / (1.0 + exp(-g[j])) * u[j]", "h = g[j] / (1.0 + exp(g[j])) * u[j]"),
    ("drop_up", "h = g[j] / (1.0 + exp(-g[j])) * u[j]", "h = g[j] / (1.0 + exp(-g[j]))"),
    ("down_transposed", "elem(c->Wd, c->dtype, (size_t)j * c->d + q)",
     "elem(c->Wd, c->dtype, (size_t)q * c->f + j)"),
    ("gate_up_swapped", "g[j] += xi * elem(c->Wg", "g[j] += xi * elem(c->Wu"),
    ("router_transposed", "elem(c->Wg, c->dtype, (size_t)i * c->N + e)",
     "elem(c->Wg, c->dtype, (size_t)e * c->d + i)"),
    ("router_no_bias", "if (c->bias) acc += (double)c->bias[e];", ""),
    ("tie_break_reversed", "  return a < b;", "  return a > b;"),
    ("nan_ranks_high", "isnan(v) ? -INFINITY : v", "isnan(v) ? INFINITY : v"),
    ("softmax_wrong_index", "topk_w[(size_t)t * k + j] = exp(l[topk_idx[(size_t)t * k + j]] - lmax) / denom",
     "topk_w[(size_t)t * k + j] = exp(l[j] - lmax) / denom"),
    ("softmax_unnormalised", "- lmax) / denom;", "- lmax);"),
    ("capacity_off_by_one", "capacity > 0 && rank >= capacity", "capacity > 0 && rank > capacity"),
    ("capacity_floor", "return (int)ceil(cf", "return (int)floor(cf"),
    ("combine_keeps_dropped", "if (inv_pos_rows[(size_t)r * k + j] < 0) continue; /* dropped slot */", ""),
    ("combine_no_shared", "yr[q] += shared[(size_t)r * d + q];", ";"),
    ("combine_unweighted", "yr[q] += w * o[q];", "yr[q] += o[q];"),
    ("entropy_natural_log", "h -= freq[e] * log2(freq[e]);", "h -= freq[e] * log(freq[e]);"),
    ("cv_sample_std", "var /= N;", "var /= (N - 1);"),
    ("top3_tie_higher_id", "if (best < 0 || freq[e] > freq[best]) best = e;",
     "if (best < 0 || freq[e] >= freq[best]) best = e;"),
    ("balance_without_N", "stats[5] = N * bal;", "stats[5] = bal;"),
    ("prob_not_normalised", "p[e] += exp(l[e] - m) / s;", "p[e] += exp(l[e] - m);"),
    ("reroute_same_candidate", "if (!placed[a] && ptr[t] < kr) prop[a] = ptr[t]++;",
     "if (!placed[a] && ptr[t] < kr) prop[a] = ptr[t];"),
    ("reroute_capacity_off_by_one",
     "if (e >= 0 && e < N && used[e] < capacity) {\n          used[e]++;\n          placed[a] = 1;",
     "if (e >= 0 && e < N && used[e] <= capacity) {\n          used[e]++;\n          placed[a] = 1;"),
    ("reroute_weights_first_choice",
     "const int e = cand[(size_t)t * kr + final_cand[(size_t)t * k + j]];\n        final_w",
     "const int e = cand[(size_t)t * kr + j];\n        final_w"),
    ("e4m3_ties_to_odd", "else c = (lo & 1) == 0 ? lo : hi;", "else c = (lo & 1) == 0 ? hi : lo;"),
    ("e4m3_round_down", "if (dlo < dhi) c = lo;", "if (dlo <= 2 * dhi) c = lo;"),
    ("hidden_silu_sign", "h[j] = g / (1.0 + exp(-g)) * u;", "h[j] = g / (1.0 + exp(g)) * u;"),
    ("e4m3_subnormal_exponent", "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    ("e4m3_bias_8", "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    ("fp8_scale_inverted", "*scale = amax > 0.0f ? amax / 448.0f : 1.0f;",
     "*scale = amax > 0.0f ? 448.0f / amax : 1.0f;"),
    ("fp8_weights_input_axis",
     "quantize_vector(c->W, c->dtype, (size_t)e * c->d * c->f + j, (size_t)c->f, c->d,",
     "quantize_vector(c->W, c->dtype, (size_t)e * c->d * c->f + (size_t)j * c->d, 1, c->d,"),
    # the E4M3 down projection of the hidden rows
    ("fp8_h_row_scale_dropped", "(e4m3_tab[hq[j]] * (double)hs)", "(e4m3_tab[hq[j]])"),
    ("fp8_down_channel_scale_dropped", "(e4m3_tab[wq[j]] * (double)c->sd[m])",
     "(e4m3_tab[wq[j]])"),
    ("fp8_h_scale_of_row0",
     "quantize_vector(c->h, ORACLE_F64, (size_t)r * c->f, 1, c->f, hq, 1, &hs);",
     "quantize_vector(c->h, ORACLE_F64, 0, 1, c->f, hq, 1, &hs);"),
    ("fp8_down_transposed", "(e4m3_tab[wq[j]] * (double)c->sd[m])",
     "(e4m3_tab[c->qd[(size_t)j * c->d + m]] * (double)c->sd[m])"),
    ("fp8_h_rounded_to_bf16",
     "quantize_vector(c->h, ORACLE_F64, (size_t)r * c->f, 1, c->f, hq, 1, &hs);",
     "double *hb = (double *)malloc(sizeof(double) * (size_t)c->f);\n"
     "  for (int j = 0; j < c->f; ++j) {\n"
     "    float v = (float)c->h[(size_t)r * c->f + j];\n"
     "    uint32_t b;\n"
     "    memcpy(&b, &v, 4);\n"
     "    b = (b + 0x7FFFu + ((b >> 16) & 1u)) & 0xFFFF0000u;\n"
     "    memcpy(&v, &b, 4);\n"
     "    hb[j] = v;\n"
     "  }\n"
     "  quantize_vector(hb, ORACLE_F64, 0, 1, c->f, hq, 1, &hs);\n"
     "  free(hb);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mut = src.replace(old, new)
    csrc = tmp_path / "mut.c"
    csrc.write_text(mut)
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", str(lib), str(csrc),
                    "-lm"], check=True)
    env = dict(os.environ, MOE_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"planted mistake '{name}' went unnoticed by the pins"
