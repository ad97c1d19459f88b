"""Plant plausible mistakes in a copy of the oracle's C source and check that the pins catch each.

Each planted variant is compiled into a temporary directory and the whole pin set runs against it
in a child process (a variant that crashes the child also counts as caught). This is what shows
the pins are strong enough to trust the oracle: a dropped term, a wrong index, a wrong sign or a
transposed operand anywhere in it makes at least one pin fail.
"""
import json
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle as oracle_pkg

TESTS = os.path.dirname(os.path.abspath(__file__))

MUTANTS = {
    "seq_side_drops_head_offset": [
        ("* N + head_off_r + h) * d + j;", "* N + h) * d + j;")],
    "head_side_drops_seq_offset": [
        ("(bb * S + seq_off_q + i) * n_r + h) * d + j;", "(bb * S + i) * n_r + h) * d + j;")],
    "head_side_wrong_batch_stride": [
        ("(bb * S + seq_off_q + i) * n_r + h) * d + j;",
         "(bb * s_q + seq_off_q + i) * n_r + h) * d + j;")],
    "seq_side_wrong_batch_stride": [
        ("((bb * s_q + i) * N + head_off_r + h) * d + j;",
         "((bb * S + i) * N + head_off_r + h) * d + j;")],
    "offsets_include_own_shard": [
        ("for (int p = 0; p < k; ++p) s += splits[p];",
         "for (int p = 0; p <= k && p < 8; ++p) s += splits[p];")],
    "mode1_reads_wrong_rank": [
        ("copy_elem(out[q] + seq_side * e, in[r] + head_side * e, e);",
         "copy_elem(out[q] + seq_side * e, in[q] + head_side * e, e);")],
    "mode1_same_as_mode0": [
        ("if (mode == 0)\n                                copy_elem",
         "if (mode == 0 || mode == 1)\n                                copy_elem")],
    "element_copy_truncated": [("case 2: memcpy(dst, src, 2); break;", "case 2: memcpy(dst, src, 1); break;")],
    "source_query_drops_head_offset": [
        ("N + offset_of(head_splits, r) + h) * d + j;", "N + h) * d + j;")],
    "rmsnorm_drops_eps": [("sqrt(mean_sq + eps)", "sqrt(mean_sq)")],
    "rmsnorm_sum_not_mean": [("mean_sq = sum_sq / (double)d", "mean_sq = sum_sq")],
    "rmsnorm_drops_weight": [("x[j] * inv_rms * w[j]", "x[j] * inv_rms")],
    "rmsnorm_eps_outside_sqrt": [("1.0 / sqrt(mean_sq + eps)", "1.0 / (sqrt(mean_sq) + eps)")],
    "rope_sin_sign": [("y[2 * j] = a * c - bq * s;", "y[2 * j] = a * c + bq * s;"),
                      ("y[2 * j + 1] = a * s + bq * c;", "y[2 * j + 1] = -a * s + bq * c;")],
    "rope_freq_exponent": [("-2.0 * (double)j / (double)d", "-1.0 * (double)j / (double)d")],
    "rope_rotate_half_pairs": [
        ("const double a = y[2 * j], bq = y[2 * j + 1];", "const double a = y[j], bq = y[j + d / 2];"),
        ("y[2 * j] = a * c - bq * s;", "y[j] = a * c - bq * s;"),
        ("y[2 * j + 1] = a * s + bq * c;", "y[j + d / 2] = a * s + bq * c;")],
    "fused_local_position": [
        ("transform_row(src, d, w, eps, (double)(seq_off_q + i), theta, dst);",
         "transform_row(src, d, w, eps, (double)i, theta, dst);")],
    "fused_row_local_position": [
        ("transform_row(src, d, w, eps, (double)s, theta, y);",
         "transform_row(src, d, w, eps, (double)i, theta, y);")],
    "qkv_planes_swapped": [("qrow = qkv_in[q] + (((bb * s_q + i) * 3 + 0)", "qrow = qkv_in[q] + (((bb * s_q + i) * 3 + 1)"),
                           ("krow = qkv_in[q] + (((bb * s_q + i) * 3 + 1)", "krow = qkv_in[q] + (((bb * s_q + i) * 3 + 0)")],
    "qkv_plane_stride": [("(((bb * s_q + i) * 3 + 2) * N + g) * d;", "((bb * s_q + i) * N + 2 * N + g) * d;")],
    "qkv_k_uses_q_weight": [("transform_row(krow, d, wk, eps, p, theta, k_out[r] + dst_row);",
                             "transform_row(krow, d, wq, eps, p, theta, k_out[r] + dst_row);")],
    "packed_planes_transposed": [("const uint16_t* row = token + (c * N + g) * d;",
                                  "const uint16_t* row = token + (g * planes + c) * d;")],
    "packed_pitch_ignored": [("const uint16_t* token = in[q] + (bb * s_q + i) * pitch;",
                              "const uint16_t* token = in[q] + (bb * s_q + i) * planes * N * d;")],
    "packed_k_uses_q_weight": [("transform_row(row, d, wk, eps, p, theta, k_out[r] + dst_row);",
                                "transform_row(row, d, wq, eps, p, theta, k_out[r] + dst_row);")],
    "packed_plain_to_wrong_plane": [("plain_out[c * W + r][dst_row + j] = row[j];",
                                     "plain_out[c * W + r][dst_row + j] = row[j - (c > 0 ? N * d : 0)];")],
    "packed_bwd_k_uses_q_weight": [("c == q_plane ? wq : wk, eps,", "wq, eps,")],
    "packed_bwd_dw_shared": [("c == q_plane ? dw : dw + d);", "dw);")],
    "packed_bwd_plain_from_wrong_plane": [("const uint16_t* gr = grads[c * W + r] + head_row;",
                                           "const uint16_t* gr = grads[(c == q_plane || c == k_plane ? c : q_plane) * W + r] + head_row;")],
    "bwd_rope_forward_direction": [("orc_rope(u, d, -p, theta);", "orc_rope(u, d, p, theta);")],
    "bwd_drops_norm_projection": [("dx[j] = inv_rms * (u[j] * w[j] - xh * dot / (double)d);",
                                   "dx[j] = inv_rms * u[j] * w[j];")],
    "bwd_eps_dropped": [("sqrt(sum_sq / (double)d + eps)", "sqrt(sum_sq / (double)d)")],
    "bwd_dot_misses_weight": [("dot += u[j] * w[j] * xh;", "dot += u[j] * xh;")],
    "bwd_dw_unnormalised": [("dw_acc[j] += u[j] * xh;", "dw_acc[j] += u[j] * x[j];")],
    "bwd_position_rank_local": [("(double)(seq_off_q + i), theta,\n                                      dx[q]", "(double)i, theta,\n                                      dx[q]")],
    "bwd_dw_not_cleared": [("for (int64_t j = 0; j < d; ++j) dw[j] = 0.0;", "")],
    "bwd_gradient_from_wrong_token": [("g[j] = orc_bf16_to_double(g_out[r][out_row + j]);",
                                       "g[j] = orc_bf16_to_double(g_out[r][out_row - (i > 0 ? n_r * d : 0) + j]);")],
    "f16_decode_bias": [("ldexp((double)(1024 + fraction), field - 25)",
                         "ldexp((double)(1024 + fraction), field - 24)")],
    "f16_decode_subnormal_scale": [("v = ldexp((double)fraction, -24);", "v = ldexp((double)fraction, -25);")],
    "f16_encode_one_bit_short": [("ldexp(1.0, ex - 10)", "ldexp(1.0, ex - 9)")],
    "f16_encode_truncates": [("nearbyint(a / step)", "floor(a / step)")],
    "f16_encode_normal_floor": [("if (ex < -14) ex = -14;", "if (ex < -15) ex = -15;")],
    "rope_half_sin_sign": [("y[j] = first * c - second * s;", "y[j] = first * c + second * s;")],
    "rope_half_wrong_partner": [("second = y[half + j];", "second = y[half + j - (j > 0)];")],
    "rope_half_freq_exponent": [("pow(theta, -(double)(2 * j) / (double)d)", "pow(theta, -(double)j / (double)d)")],
    "variant_ignores_half_pairs": [("    if (half_pairs)\n        orc_rope_half", "    if (0)\n        orc_rope_half")],
    "variant_ignores_f16": [("return f16 ? orc_f16_to_double(h) : orc_bf16_to_double(h);",
                             "return orc_bf16_to_double(h);")],
    "variant_local_position": [("eps,\n                                          (double)(seq_off_q + i), theta, dst);",
                                "eps,\n                                          (double)i, theta, dst);")],
    "variant_bwd_forward_rotation": [("rope_pairs(u, d, -p, theta, half_pairs);",
                                      "rope_pairs(u, d, p, theta, half_pairs);")],
    "variant_bwd_grad_drops_seq_offset": [("const int64_t grad_row = ((bb * S + seq_off_q + i) * n_r + h) * d;",
                                           "const int64_t grad_row = ((bb * S + i) * n_r + h) * d;")],
    "part_row_range_ignored": [("static int64_t part_row_end(int64_t s_q, int64_t i_hi) { return i_hi < s_q ? i_hi : s_q; }",
                                "static int64_t part_row_end(int64_t s_q, int64_t i_hi) { (void)i_hi; return s_q; }")],
    "bwd_part_starts_at_row_zero": [
        ("""            for (int64_t i = i_lo; i < part_row_end(s_q, i_hi); ++i)
                for (int64_t hg = 0; hg < N; ++hg) {""",
         """            for (int64_t i = 0; i < part_row_end(s_q, i_hi); ++i)
                for (int64_t hg = 0; hg < N; ++hg) {""")],
    "bf16_truncates": [("nearbyint(a / quantum)", "floor(a / quantum)")],
    "bf16_one_bit_too_many": [("ldexp(1.0, ex - 7)", "ldexp(1.0, ex - 8)")],
    "bf16_widening_drops_low_bits": [("uint32_t bits = (uint32_t)h << 16;",
                                      "uint32_t bits = ((uint32_t)h & 0xFFF0u) << 16;")],
}

CHILD = r"""
import json, sys
sys.path.insert(0, {tests!r}); sys.path.insert(0, {root!r})
import torch
torch.set_num_threads(1)
import oracle, oracle_pins
orc = oracle.Oracle({lib!r})
print(json.dumps(oracle_pins.run_all(orc, quick=True)))
"""


# the children run side by side: one thread each, so that they do not oversubscribe the cores
_CHILD_ENV = dict(os.environ, OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")


def _check(name, tmpdir):
    with open(oracle_pkg.SOURCE) as f:
        src = f.read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"{name}: pattern not found exactly once: {old!r}"
        src = src.replace(old, new)
    c_path = os.path.join(tmpdir, f"{name}.c")
    with open(c_path, "w") as f:
        f.write(src)
    lib = oracle_pkg.build(os.path.join(tmpdir, f"lib{name}.so"), c_path)
    code = CHILD.format(tests=TESTS, root=os.path.dirname(TESTS), lib=lib)
    try:
        proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                              timeout=1200, env=_CHILD_ENV)
    except subprocess.TimeoutExpired:
        return name, []  # not caught: reported by name below
    if proc.returncode != 0:
        return name, ["crashed"]
    return name, json.loads(proc.stdout.strip().splitlines()[-1])


def test_every_planted_mistake_is_caught(tmp_path):
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as pool:
        results = dict(pool.map(lambda n: _check(n, str(tmp_path)), MUTANTS))
    missed = [n for n, failed in results.items() if not failed]
    assert not missed, f"planted mistakes no pin caught: {missed}"


def test_unmutated_copy_passes(tmp_path):
    """The same child-process harness on an unmodified copy reports no failure."""
    lib = oracle_pkg.build(os.path.join(str(tmp_path), "libclean.so"))
    code = CHILD.format(tests=TESTS, root=os.path.dirname(TESTS), lib=lib)
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                          timeout=1200, env=_CHILD_ENV)
    assert proc.returncode == 0, proc.stderr[-2000:]
    assert json.loads(proc.stdout.strip().splitlines()[-1]) == []


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
