"""The oracle pins must catch plausible mistakes in the oracle (CPU only).

Each case copies oracle.c, plants one plausible slip (a wrong index, a dropped
term, a wrong sign, a transposed axis), builds the copy into a temporary
library and runs the pin suite (test_oracle.py) against it in a child
process (test_oracle.py and test_oracle_fp8.py). The suite has to fail for
every mutant; the untouched copy has to pass, which shows that the harness
itself works.
"""
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "kv_head_modulo": ("int k = h / group;", "int k = h % s->num_kv_heads;"),
    "causal_off_by_one": ("int64_t n_vis = L - s->num_q + t + 1;",
                          "int64_t n_vis = L - s->num_q + t;"),
    "page_row_shift": ("int64_t row = ((int64_t)phys * s->num_kv_heads + k) * s->page_size + j % s->page_size;\n    return k_pages",
                       "int64_t row = ((int64_t)phys * s->num_kv_heads + k) * s->page_size + (j + 1) % s->page_size;\n    return k_pages"),
    "page_slot_index": ("int64_t slot = j / s->page_size;\n    if (slot >= s->max_pages_per_seq) return NULL;\n    int32_t phys = page_table[(int64_t)b * s->max_pages_per_seq + slot];\n    if (phys < 0 || phys >= s->num_pages) return NULL;\n    int64_t row = ((int64_t)phys * s->num_kv_heads + k) * s->page_size + j % s->page_size;\n    return k_pages",
                        "int64_t slot = j / s->page_size;\n    if (slot >= s->max_pages_per_seq) return NULL;\n    int32_t phys = page_table[(int64_t)b + slot * s->batch];\n    if (phys < 0 || phys >= s->num_pages) return NULL;\n    int64_t row = ((int64_t)phys * s->num_kv_heads + k) * s->page_size + j % s->page_size;\n    return k_pages"),
    "lse_drops_log_sum": ("if (lse_out) *lse_out = m + log(l);", "if (lse_out) *lse_out = m;"),
    "exp_sign": ("double e = exp(sbuf[j] - m);", "double e = exp(m - sbuf[j]);"),
    "value_row_stride": ("return v_pages + row * s->ov_depth;", "return v_pages + row * s->qk_depth;"),
    "q_axes_transposed": (
        "const uint16_t* qrow = J->q + (((int64_t)b * s->num_q + t) * s->num_q_heads + h) * s->qk_depth;\n    double m",
        "const uint16_t* qrow = J->q + (((int64_t)b * s->num_q_heads + h) * s->num_q + t) * s->qk_depth;\n    double m"),
    "combine_drops_partition_sum": ("double w = psum[p] * exp2((pmax[p] - gmax) * c) / gsum;",
                                    "double w = exp2((pmax[p] - gmax) * c) / gsum;"),
    "combine_missing_log2e": ("const double c = J->scale * (1.0 / log(2.0));",
                              "const double c = J->scale;"),
    "combine_lse_unscaled_max": ("*lse_out = J->scale * gmax + log(gsum);",
                                 "*lse_out = gmax + log(gsum);"),
    # the fp8 cache (oracle_decode_fp8)
    "e4m3_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3_subnormal_exponent": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "e4m3_sign_dropped": ("return sign ? -v : v;", "return v;"),
    "fp8_k_scale_dropped": ("for (int d = 0; d < d8; ++d) dst[d] = ks * e4m3_table[src[d]];",
                            "for (int d = 0; d < d8; ++d) dst[d] = e4m3_table[src[d]];"),
    "fp8_rope_column_rotated": ("dst[d8 + d] = widen_bf16(J->krope[r * J->rope_depth + d]);",
                                "dst[d8 + d] = widen_bf16(J->krope[r * J->rope_depth + (d + 1) % J->rope_depth]);"),
    "fp8_rope_scaled": ("dst[d8 + d] = widen_bf16(J->krope[r * J->rope_depth + d]);",
                        "dst[d8 + d] = ks * widen_bf16(J->krope[r * J->rope_depth + d]);"),
    "fp8_separate_v_scaled": ("for (int d = 0; d < s->ov_depth; ++d) dst[d] = e4m3_table[J->v8[r * s->ov_depth + d]];",
                              "for (int d = 0; d < s->ov_depth; ++d) dst[d] = (J->kscale ? (double)J->kscale[r] : 1.0) * e4m3_table[J->v8[r * s->ov_depth + d]];"),
    "fp8_latent_v_unscaled": ("for (int d = 0; d < s->ov_depth; ++d) dst[d] = ks * e4m3_table[J->k8[r * d8 + d]];",
                              "for (int d = 0; d < s->ov_depth; ++d) dst[d] = e4m3_table[J->k8[r * d8 + d]];"),
    "fp8_row_stride": ("const uint8_t* src = J->k8 + r * d8;", "const uint8_t* src = J->k8 + r * s->qk_depth;"),
}


def _build_and_run(name, tmpdir):
    src = open(SRC).read()
    if name != "identity":
        old, new = MUTANTS[name]
        assert src.count(old) >= 1, f"mutation site for {name} not found"
        src = src.replace(old, new, 1)
    d = os.path.join(tmpdir, name)
    os.makedirs(d)
    shutil.copy(os.path.join(ROOT, "oracle", "oracle.h"), d)
    c_path = os.path.join(d, "oracle.c")
    open(c_path, "w").write(src)
    so = os.path.join(d, "liboracle.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-o", so, c_path, "-lm",
                    "-lpthread"], check=True)
    env = dict(os.environ, SPD_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py"),
                        os.path.join(ROOT, "tests", "test_oracle_fp8.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode


def test_pins_catch_every_mutant():
    tmp = tempfile.mkdtemp(prefix="spd_mutants_")
    try:
        names = ["identity"] + sorted(MUTANTS)
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            codes = dict(zip(names, ex.map(lambda n: _build_and_run(n, tmp), names)))
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    assert codes["identity"] == 0, "the unmodified oracle must pass its pins"
    survivors = [n for n in MUTANTS if codes[n] == 0]
    assert not survivors, f"pins did not catch: {survivors}"
