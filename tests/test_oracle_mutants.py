"""Plants plausible mistakes in a temporary copy of the oracle (CPU only) and
checks that the pins catch each one: a dropped term, a wrong sign, index or
base, a transposed operand.  The committed oracle is never modified."""

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# (name, text in dsa_oracle.c, replacement)
MUTANTS = [
    ("rope_direction_cos_row", "qh[h][2 * i] = x0 * c - x1 * s;", "qh[h][2 * i] = x0 * c + x1 * s;"),
    ("rope_direction_sin_row", "qh[h][2 * i + 1] = x0 * s + x1 * c;", "qh[h][2 * i + 1] = -x0 * s + x1 * c;"),
    ("rope_half_split",
     "double x0 = qh[h][2 * i], x1 = qh[h][2 * i + 1];\n                qh[h][2 * i] = x0 * c - x1 * s;\n"
     "                qh[h][2 * i + 1] = x0 * s + x1 * c;",
     "double x0 = qh[h][i], x1 = qh[h][i + 32];\n                qh[h][i] = x0 * c - x1 * s;\n"
     "                qh[h][i + 32] = x0 * s + x1 * c;"),
    ("rope_pos_plus_one", "double th = (double)pos * (double)inv_freq[i];",
     "double th = (double)(pos + 1) * (double)inv_freq[i];"),
    ("rope_pair_index", "double th = (double)pos * (double)inv_freq[i];",
     "double th = (double)pos * (double)inv_freq[(i + 1) % RP];"),
    ("rope_upper_dims", "double x0 = qh[h][2 * i], x1 = qh[h][2 * i + 1];\n                qh[h][2 * i] = x0 * c - x1 * s;\n"
     "                qh[h][2 * i + 1] = x0 * s + x1 * c;",
     "double x0 = qh[h][64 + 2 * i], x1 = qh[h][64 + 2 * i + 1];\n                qh[h][64 + 2 * i] = x0 * c - x1 * s;\n"
     "                qh[h][64 + 2 * i + 1] = x0 * s + x1 * c;"),
    ("ssmax_log10", "log((double)pos + 1.0)", "log10((double)pos + 1.0)"),
    ("ssmax_log_pos", "log((double)pos + 1.0)", "log((double)pos + 2.0)"),
    ("ssmax_s_b_swapped", "(double)ss[h] * log((double)pos + 1.0) + (double)sb[h]",
     "(double)sb[h] * log((double)pos + 1.0) + (double)ss[h]"),
    ("score_no_sqrt128", "double r = dot / sqrt(128.0);", "double r = dot;"),
    ("score_no_sqrt32", "total += (double)w[h] * r / sqrt(32.0);", "total += (double)w[h] * r;"),
    ("score_no_relu", "if (r < 0.0) r = 0.0;", ";"),
    ("score_relu_after_weight", "total += (double)w[h] * r / sqrt(32.0);",
     "total += fmax(0.0, (double)w[h] * dot / sqrt(128.0)) / sqrt(32.0);"),
    ("score_head_weight_index", "total += (double)w[h] * r / sqrt(32.0);",
     "total += (double)w[IH - 1 - h] * r / sqrt(32.0);"),
    ("query_transposed", "qh[h][d] = f * oracle_bf16_value(q[h * ID + d]);",
     "qh[h][d] = f * oracle_bf16_value(q[d * IH + h]);"),
    ("causal_exclusive", "for (int64_t j = 0; j <= pos; ++j) {", "for (int64_t j = 0; j < pos; ++j) {"),
    ("mask_zero_not_neg_inf", "row[j] = -INFINITY;", "row[j] = 0.0;"),
    ("page_offset", "row = page * s->page_size + j % s->page_size;",
     "row = page * s->page_size + (j + 1) % s->page_size;"),
    ("page_index", "int64_t page = s->page_table[(int64_t)b * s->max_pages + p];",
     "int64_t page = s->page_table[(int64_t)b * s->max_pages + (p + 1) % s->max_pages];"),
    ("e4m3_bias", "v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("e4m3_subnormal", "v = ldexp((double)m / 8.0, 1 - 7);", "v = ldexp((double)m / 8.0, -7);"),
    ("e4m3_nan", "if (e == 15 && m == 7) return NAN;", "if (e == 15 && m == 7) return 480.0;"),
    ("bf16_shift", "uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
    ("key_scale_dropped", "k[d] = oracle_e4m3_value(p[d]) * sc;", "k[d] = oracle_e4m3_value(p[d]);"),
    ("ds_mla_group", "oracle_e4m3_value(row[d]) * (double)scale[d / 128];",
     "oracle_e4m3_value(row[d]) * (double)scale[d % 4];"),
    ("ds_mla_rope_offset", "memcpy(&b, row + MV + 16 + 2 * r, 2);", "memcpy(&b, row + MV + 2 * r, 2);"),
    ("topk_tie_larger_index", "return (x->j > y->j) - (x->j < y->j);", "return (x->j < y->j) - (x->j > y->j);"),
    ("topk_smallest", "if (x->s > y->s) return -1;\n    if (x->s < y->s) return 1;",
     "if (x->s > y->s) return 1;\n    if (x->s < y->s) return -1;"),
    ("topk_pad_zero", "idx[i] = i < m ? v[i].j : -1;", "idx[i] = i < m ? v[i].j : 0;"),
    ("topk_one_short", "int32_t m = n < k ? n : k;", "int32_t m = n < k ? n : (k > 0 ? k - 1 : 0);"),
    ("mla_score_512_dims", "for (int d = 0; d < MD; ++d) dot += qd[d] * c[(int64_t)j * MD + d];",
     "for (int d = 0; d < MV; ++d) dot += qd[d] * c[(int64_t)j * MD + d];"),
    ("mla_no_sm_scale", "s[j] = sm_scale * dot;", "s[j] = dot;"),
    ("mla_lse_log2", "lse[h] = mx + log(l);", "lse[h] = mx + log2(l);"),
    ("mla_lse_no_max", "lse[h] = mx + log(l);", "lse[h] = log(l);"),
    ("mla_value_offset", "oh[d] += p * cj[d];", "oh[d] += p * cj[(d + 64) % MD];"),
    ("mla_keeps_minus_one", "if (j < 0) continue;", "if (j < 0) j = 0;"),
    ("mla_empty_lse_zero", "lse[h] = -INFINITY;", "lse[h] = 0.0;"),
    ("mla_unnormalised", "double p = exp(s[j] - mx) / l;", "double p = exp(s[j] - mx);"),
    ("mla_query_head", "qd[d] = oracle_bf16_value(q[h * MD + d]);", "qd[d] = oracle_bf16_value(q[((h + 1) % MH) * MD + d]);"),
    # the cache-write side
    ("e4m3_encode_round_half_up", "double val = rint(a / q) * q;", "double val = floor(a / q + 0.5) * q;"),
    ("e4m3_encode_no_saturation", "if (val > 448.0) val = 448.0; /* saturate */", ";"),
    ("e4m3_encode_subnormal_quantum", "if (lead < -6) lead = -6;     /* subnormals: the quantum stays 2^-9 */",
     "if (lead < -7) lead = -7;"),
    ("bf16_encode_truncate", "double r = rint(a / q);       /* exact division by a power of two; rint ties to even */",
     "double r = floor(a / q);"),
    ("bf16_encode_exponent_bias", "uint16_t ebits = (uint16_t)(be - 1 + 127);", "uint16_t ebits = (uint16_t)(be - 1 + 126);"),
    ("layer_norm_unbiased_variance", "        var /= ID;", "        var /= (ID - 1);"),
    ("layer_norm_no_eps", "double inv = 1.0 / sqrt(var + eps);", "double inv = 1.0 / sqrt(var);"),
    ("layer_norm_gamma_beta_swapped", "v[d] = (v[d] - mean) * inv * (double)gamma[d] + (double)beta[d];",
     "v[d] = (v[d] - mean) * inv * (double)beta[d] + (double)gamma[d];"),
    ("rope32_sign", "v[2 * i] = x0 * c - x1 * s;", "v[2 * i] = x0 * c + x1 * s;"),
    ("latent_rope_not_applied", "        if (inv_freq) rope32(o + MV, pos[t], inv_freq);\n    }\n    return 0;\n}\n\nint oracle_mla_q",
     "        (void)0;\n    }\n    return 0;\n}\n\nint oracle_mla_q"),
    ("mla_q_ssmax_skips_rope_dims", "for (int d = 0; d < MD; ++d) o[d] *= f;", "for (int d = 0; d < MV; ++d) o[d] *= f;"),
    ("mla_q_ssmax_head_index",
     "double f = (double)ssmax_s[h] * log((double)pos[t] + 1.0) + (double)ssmax_b[h];",
     "double f = (double)ssmax_s[(h + 1) % MH] * log((double)pos[t] + 1.0) + (double)ssmax_b[h];"),
    # DCP
    ("dcp_owner_ignores_interleave", "return (t / interleave) % world;", "return t % world;"),
    ("dcp_local_skips_turns", "return (turn / world) * interleave + t % interleave;",
     "return turn * interleave + t % interleave;"),
    ("dcp_global_rank_dropped", "return (own_turn * world + rank) * interleave + local % interleave;",
     "return (own_turn * world) * interleave + local % interleave;"),
    ("pack_negative_order", "return (b & 0x80000000u) ? ~b : (b | 0x80000000u);",
     "return (b & 0x80000000u) ? b : (b | 0x80000000u);"),
    ("pack_negative_zero", "if (score == 0.0f) score = 0.0f; /* -0 as +0 */", ";"),
    ("pack_id_not_inverted", "return ((uint64_t)score_code(score) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)id);",
     "return ((uint64_t)score_code(score) << 32) | (uint64_t)(uint32_t)id;"),
    ("merge_ids_unsorted", "qsort(ids, (size_t)m, sizeof(int32_t), by_id);", ";"),
    ("merge_duplicates_accepted", "dup |= all[i] == all[i - 1];", ";"),
    ("merge_takes_one_fewer", "int32_t m = n < k ? (int32_t)n : k;\n    for (int32_t i = 0; i < m; ++i) ids[i]",
     "int32_t m = n < k ? (int32_t)n : k - 1;\n    for (int32_t i = 0; i < m; ++i) ids[i]"),
    ("compact_ignores_owner", "if (t >= 0 && oracle_dcp_owner(t, world, interleave) == rank)", "if (t >= 0)"),
    ("lse_combine_max_not_logsumexp", "double L = m + log(sum);", "double L = m;"),
    # NVFP4
    ("e2m1_subnormal", "double v = e == 0 ? m * 0.5 : ldexp(1.0 + m * 0.5, e - 1);",
     "double v = e == 0 ? m * 1.0 : ldexp(1.0 + m * 0.5, e - 1);"),
    ("e2m1_bias", "double v = e == 0 ? m * 0.5 : ldexp(1.0 + m * 0.5, e - 1);",
     "double v = e == 0 ? m * 0.5 : ldexp(1.0 + m * 0.5, e - 2);"),
    ("e2m1_ties_to_odd", "if (d < best_d || (d == best_d && (c & 1) == 0)) {",
     "if (d < best_d || (d == best_d && (c & 1) == 1)) {"),
    ("e2m1_negative_zero_unsigned", "uint8_t sgn = signbit(v) ? 8 : 0;", "uint8_t sgn = v < 0.0 ? 8 : 0;"),
    ("nvfp4_scale_over_4", "scales[b] = oracle_e4m3_encode(amax / (6.0 * g));",
     "scales[b] = oracle_e4m3_encode(amax / (4.0 * g));"),
    ("nvfp4_nibble_order", "codes[8 * b + i / 2] = (uint8_t)(lo | (hi << 4));",
     "codes[8 * b + i / 2] = (uint8_t)(hi | (lo << 4));"),
    ("nvfp4_tensor_scale_dropped", "out[i] = g * oracle_e4m3_value(scales[i / 16]) * oracle_e2m1_value(nib);",
     "out[i] = oracle_e4m3_value(scales[i / 16]) * oracle_e2m1_value(nib);"),
    # block-sparse selection
    ("block_score_sum", "for (int32_t j = b * block; j < n && j < (b + 1) * block; ++j) m = fmax(m, scores[j]);",
     "for (int32_t j = b * block; j < n && j < (b + 1) * block; ++j) m = (m == -INFINITY ? 0.0 : m) + scores[j];"),
    ("block_recent_not_forced", "    chosen[last] = 1;\n", "\n"),
    ("block_recent_counted_twice", "if (v[i].j == last) continue;", ";"),
    ("block_score_spills_over", "for (int32_t j = b * block; j < n && j < (b + 1) * block; ++j) m = fmax(m, scores[j]);",
     "for (int32_t j = b * block; j < n && j <= (b + 1) * block; ++j) m = fmax(m, scores[j]);"),
    ("nvfp4_key_row_stride", "oracle_nvfp4_dequantize(ID, (const uint8_t*)ks->keys + row * (ID / 2),",
     "oracle_nvfp4_dequantize(ID, (const uint8_t*)ks->keys + row * (ID / 4),"),
    ("nvfp4_latent_scale_row", "ls->block_scale + row * (MD / 16),", "ls->block_scale + row * (MD / 32),"),
    ("nvfp4_latent_tensor_scale", "                                    ls->global, cj);",
     "                                    1.0, cj);"),
    ("lse_combine_weights_unnormalised",
     "double wgt = exp(lse_parts[(int64_t)r * rows + i] - L);", "double wgt = exp(lse_parts[(int64_t)r * rows + i] - m);"),
]

RUNNER = r"""
import sys
sys.path[:0] = [{root!r}, {here!r}]
import oracle, oracle_pins
L = oracle.load(sys.argv[1])
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(L)
    except Exception as e:
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
"""


def _run_mutant(tmp_path, name, old, new):
    src = open(os.path.join(ROOT, "oracle", "dsa_oracle.c")).read()
    assert src.count(old) == 1, f"{name}: anchor text not found exactly once"
    d = tmp_path / name
    d.mkdir()
    path = d / "dsa_oracle.c"
    path.write_text(src.replace(old, new))
    so = str(d / "libmutant.so")
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-w", "-ffp-contract=off", "-shared", "-fPIC",
                           "-I", os.path.join(ROOT, "oracle"), "-o", so, str(path), "-lm"])
    r = subprocess.run([sys.executable, "-c", RUNNER.format(root=ROOT, here=HERE), so], capture_output=True,
                       text=True, timeout=300)
    if r.returncode != 0:
        return name, ["<crashed>"]
    line = [x for x in r.stdout.splitlines() if x.startswith("FAILED:")][-1]
    return name, [x for x in line[len("FAILED:"):].split(",") if x]


def test_every_planted_mistake_fails_a_pin(tmp_path):
    oracle.build()
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        res = list(ex.map(lambda m: _run_mutant(tmp_path, *m), MUTANTS))
    survivors = [n for n, failed in res if not failed]
    assert not survivors, f"mistakes no pin catches: {survivors}"
