"""Mutation check of the oracle's CPU pins.

Each entry below plants one plausible mistake (a single-line change) in a copy
of the oracle's C source; the oracle pin tests (tests/test_oracle_*.py and
tests/test_rounding_claims.py) then run against the mutated copy.  A mutation
the tests do not catch means a missing pin.  Nothing here is collected by
pytest; run it by hand:

    python tests/oracle_mutations.py [--workdir DIR] [name ...]

It builds each mutated oracle with gcc inside the work directory (a fresh
temporary directory by default) and prints one line per mutation.
"""

import argparse
import os
import shutil
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
C = os.path.join("oracle", "nvfp4kv_oracle.c")

M = {
    "ties_away": [("if (a > mid * den) return hi;\n    return (lo % 2 == 0) ? lo : hi;",
                   "if (a > mid * den) return hi;\n    return hi;")],
    "scale_drops_g": [("round_quotient_to_table(amax, 6.0 * (double)g, e4m3_mags, 127)",
                       "round_quotient_to_table(amax, 6.0, e4m3_mags, 127)")],
    "code_drops_g": [("round_quotient_to_table(fabs(x[i]), sd * (double)g, e2m1_mags, 8)",
                      "round_quotient_to_table(fabs(x[i]), sd, e2m1_mags, 8)")],
    "zero_code_unsigned": [("codes16[i] = (uint8_t)(signbit(x[i]) ? (8 | c) : c);",
                            "codes16[i] = (uint8_t)(signbit(x[i]) && c ? (8 | c) : c);")],
    "zero_scale_codes_kept": [("int c = (sd == 0.0) ? 0 : round_quotient_to_table",
                               "int c = (sd == 0.0) ? 1 : round_quotient_to_table")],
    "dequant_drops_g": [("return oracle_e2m1_value(code) * oracle_e4m3_value(scale) * (double)g;",
                         "return oracle_e2m1_value(code) * oracle_e4m3_value(scale);")],
    "nibble_read_swapped": [("uint8_t code = (d % 2 == 0) ? (byte & 15) : (byte >> 4);",
                             "uint8_t code = (d % 2 == 1) ? (byte & 15) : (byte >> 4);")],
    "nibble_both_swapped": [("uint8_t code = (d % 2 == 0) ? (byte & 15) : (byte >> 4);",
                             "uint8_t code = (d % 2 == 1) ? (byte & 15) : (byte >> 4);"),
                            ("c[b * 8 + i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));",
                             "c[b * 8 + i] = (uint8_t)(codes[2 * i + 1] | (codes[2 * i] << 4));")],
    "v_scale_layout": [("return slab + grp * 2304 + 2176 + blk * 16 + r;", "return slab + grp * 2304 + 2176 + r * 8 + blk;")],
    "k_scale_layout": [("if (which == 0) return slab + grp * 2304 + 1024 + r * 8 + blk;",
                        "if (which == 0) return slab + grp * 2304 + 1024 + blk * 16 + r;")],
    "calib_no_448": [("return (float)amax / (largest_e2m1 * largest_e4m3);", "return (float)amax / largest_e2m1;")],
    "calib_keeps_inf": [("if (isfinite(a) && a > amax) amax = a;", "if (a > amax) amax = a;")],
    "no_sm_scale": [("            s *= sm_scale;\n", "            s *= 1.0;\n")],
    "gqa_interleaved": [("oracle_bf16_value(j->q[((int64_t)b * j->num_q_heads + kv * G + h) * HEAD_DIM + d]);",
                         "oracle_bf16_value(j->q[((int64_t)b * j->num_q_heads + h * Hkv + kv) * HEAD_DIM + d]);")],
    "extend_causal_short": [("int64_t n = n_prefix + i + 1;", "int64_t n = n_prefix + i + (i > 0 ? 0 : 1);")],
    "prefix_dst_no_cu": [("int64_t dst_row = (int64_t)cu_prefix_lens[r] + t;", "int64_t dst_row = (int64_t)r * 0 + t + cu_prefix_lens[0];")],
    "fp8_drops_g": [("int m = round_quotient_to_table(fabs(v), (double)g, e4m3_mags, 127);",
                     "int m = round_quotient_to_table(fabs(v), 1.0, e4m3_mags, 127);")],
    "fp8_fp32_quotient": [("int m = round_quotient_to_table(fabs(v), (double)g, e4m3_mags, 127);",
                           "int m = oracle_e4m3_encode((float)fabs(v) / g) & 0x7F;")],
    "scale_fp32_quotient": [("uint8_t s = (uint8_t)round_quotient_to_table(amax, 6.0 * (double)g, e4m3_mags, 127);",
                             "uint8_t s = oracle_e4m3_encode((float)amax / (6.0f * g));")],
    "code_fp32_quotient": [("int c = (sd == 0.0) ? 0 : round_quotient_to_table(fabs(x[i]), sd * (double)g, e2m1_mags, 8);",
                            "int c = (sd == 0.0) ? 0 : (oracle_e2m1_encode((float)fabs(x[i]) / ((float)sd * g)) & 7);")],
    "dequant_two_roundings": [("dst[d] = oracle_bf16_from_double(row[d]);",
                               "dst[d] = oracle_bf16_from_float((float)row[d]);")],
    "bf16_no_subnormal_step": [("int step_exp = (e - 1 >= -126) ? e - 8 : -133;", "int step_exp = e - 8;")],
    "bf16_ties_up": [("if (r > 0.5 || (r == 0.5 && fmod(f, 2.0) != 0.0)) f += 1.0;", "if (r >= 0.5) f += 1.0;")],
    "bf16_no_overflow": [("if (v >= ldexp(1.0, 128)) return sign | 0x7f80u;", "if (v > ldexp(1.0, 200)) return sign | 0x7f80u;")],
    "fp8_dequant_drops_g": [("for (int d = 0; d < HEAD_DIM; d++) out[d] = oracle_e4m3_value(c[d]) * (double)g;",
                             "for (int d = 0; d < HEAD_DIM; d++) out[d] = oracle_e4m3_value(c[d]);")],
    "e4m3_subnormal_step": [("ldexp((double)m, -9)", "ldexp((double)m, -10)")],
    "amax_signed": [("if (fabs(x[i]) > amax) amax = fabs(x[i]);", "if (x[i] > amax) amax = x[i];")],
    "bf16_truncates": [("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;", "(void)lower;")],
    "no_max_shift": [("double pt = exp(scores[h * n + t] - m[h]);", "double pt = exp(scores[h * n + t]);")],
    "extend_prefix_row_offset": [("src = (which ? c->v_pre : c->k_pre) + ((c->pre0 + t) * c->num_kv_heads + c->kv) * HEAD_DIM;",
                                  "src = (which ? c->v_pre : c->k_pre) + ((t) * c->num_kv_heads + c->kv) * HEAD_DIM;")],
    "extend_chunk_offset": [("src = (which ? c->v_new : c->k_new) + ((c->new0 + t - c->n_prefix) * c->num_kv_heads + c->kv) * HEAD_DIM;",
                             "src = (which ? c->v_new : c->k_new) + ((c->new0 + t - c->n_prefix + 1) * c->num_kv_heads + c->kv) * HEAD_DIM;")],
    "extend_gqa_interleaved": [("qd[h * HEAD_DIM + d] = oracle_bf16_value(j->q[(row * j->num_q_heads + kv * G + h) * HEAD_DIM + d]);",
                                "qd[h * HEAD_DIM + d] = oracle_bf16_value(j->q[(row * j->num_q_heads + h * Hkv + kv) * HEAD_DIM + d]);")],
    "paged_row_offset": [("dequant_row(c->p, page, c->kv, which, (int)(t % c->p->page_size), out);",
                          "dequant_row(c->p, page, c->kv, which, (int)((t + 1) % c->p->page_size), out);")],
    "slab_kv_order": [("return p->pool + (page * p->num_kv_heads + kv) * oracle_slab_bytes(p->dtype, p->page_size);",
                       "return p->pool + (kv * p->num_pages + page) * oracle_slab_bytes(p->dtype, p->page_size);")],
    "v_codes_offset": [("if (p->dtype == ORACLE_DTYPE_NVFP4) return slab + grp * 2304 + (which ? 1152 : 0) + r * 64;",
                        "if (p->dtype == ORACLE_DTYPE_NVFP4) return slab + grp * 2304 + (which ? 1088 : 0) + r * 64;")],
    "scale_nonsat_zero": [("int c = (sd == 0.0) ? 0 :", "int c = (sd == 0.0 && 0) ? 0 :")],
    "bf16_row_stride": [("int rc = store_row(&c->p, 0, 0, which, 0, (which ? c->v : c->k) + t * c->row_stride);",
                         "int rc = store_row(&c->p, 0, 0, which, 0, (which ? c->v : c->k) + t * 128);")],
    "prefix_kv_index": [("uint16_t *dst = (which ? v_ws : k_ws) + (dst_row * num_kv_heads + kv) * HEAD_DIM;",
                         "uint16_t *dst = (which ? v_ws : k_ws) + (dst_row * num_kv_heads + (num_kv_heads - 1 - kv)) * HEAD_DIM;")],
    "extend_req_map": [("while (r + 1 < j->num_reqs && j->cu_q[r + 1] <= row) r++;",
                        "while (r + 1 < j->num_reqs && j->cu_q[r + 1] < row) r++;")],
    "ties_low": [("if (a < mid) return lo;", "if (a <= mid) return lo;")],
    "calib_zero_gives_zero": [("if (amax == 0.0) return 1.0f;", "if (amax == 0.0) return 0.0f;")],
    "decode_out_offset": [("const int64_t o = ((int64_t)b * j->num_q_heads + (int64_t)kv * G) * HEAD_DIM;",
                           "const int64_t o = ((int64_t)b * j->num_q_heads + (int64_t)kv) * HEAD_DIM;")],
    "spread_signed": [("spread[h * HEAD_DIM + d] += wt * fabs(vrow[d] - out[h * HEAD_DIM + d]);",
                       "spread[h * HEAD_DIM + d] += wt * (vrow[d] - out[h * HEAD_DIM + d]);")],
    "spread_unnormalised": [("double wt = exp(scores[h * n + t] - m[h]) / l[h];",
                             "double wt = exp(scores[h * n + t] - m[h]);")],
}



def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--workdir", default=None, help="where the mutated copies are built (default: a temp dir)")
    ap.add_argument("names", nargs="*", help="mutations to run (default: all)")
    args = ap.parse_args()
    work = args.workdir or tempfile.mkdtemp(prefix="oracle_mutations_")
    tests = sorted(os.path.join("tests", f) for f in os.listdir(os.path.join(ROOT, "tests"))
                   if f.startswith("test_oracle_") or f == "test_rounding_claims.py")
    survivors = []
    for name, edits in M.items():
        if args.names and name not in args.names:
            continue
        tree = os.path.join(work, "tree")
        if os.path.exists(tree):
            shutil.rmtree(tree)
        os.makedirs(tree)
        for d in ("oracle", "tests", "workloads"):
            shutil.copytree(os.path.join(ROOT, d), os.path.join(tree, d),
                            ignore=shutil.ignore_patterns("*.so", "__pycache__"))
        shutil.copy(os.path.join(ROOT, "pytest.ini"), tree)
        path = os.path.join(tree, C)
        text = open(path).read()
        for old, new in edits:
            if text.count(old) != 1:
                raise SystemExit("mutation %s no longer applies: %r" % (name, old))
            text = text.replace(old, new)
        open(path, "w").write(text)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu"] + tests, cwd=tree,
                           capture_output=True, text=True, timeout=900)
        caught = r.returncode != 0
        if not caught:
            survivors.append(name)
        print("%-26s %s" % (name, "caught" if caught else "SURVIVED"), flush=True)
    shutil.rmtree(os.path.join(work, "tree"), ignore_errors=True)
    if survivors:
        raise SystemExit("not caught: " + ", ".join(survivors))


if __name__ == "__main__":
    main()
