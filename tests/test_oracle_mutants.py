"""The pins must be able to fail: plant plausible mistakes in copies of the
oracle source, build each copy, and check that the pin suite rejects it.

Each mutant is compiled to a temporary library and exercised in a child
process (ORACLE_SO points the oracle package at it), so a broken copy can never
disturb this process.  Mistakes are planted only in the oracle, on the CPU.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "pad_sign": ("kp[i] * g->d[i] - g->p[i]", "kp[i] * g->d[i] + g->p[i]"),
    "stride_dilation_swapped": ("op[i] * g->s[i] + kp[i] * g->d[i]", "op[i] * g->d[i] + kp[i] * g->s[i]"),
    "bias_dropped": ("double acc = bias ? (double)bias[o] : 0.0;", "double acc = 0.0;"),
    "kernel_flipped": ("unflatten(t, g->ndim, g->k, kp);\n      int64_t off = tap_input_offset(g, op, kp);",
                       "unflatten(t, g->ndim, g->k, kp);\n      for (int z = 0; z < g->ndim; ++z) kp[z] = g->k[z] - 1 - kp[z];\n"
                       "      int64_t off = tap_input_offset(g, op, kp);"),
    "out_dims_off_by_one": ("d[i] * (k[i] - 1) - 1, s[i]) + 1", "d[i] * (k[i] - 1), s[i]) + 1"),
    "min_became_max": ("if (z < mn) mn = z;", "if (z > mn || mn == INFINITY) mn = z;"),
    "softmax_no_normalise": ("res[o * res_stride] = exp(m[o] - mx) / sum;", "res[o * res_stride] = exp(m[o] - mx);"),
    "tap_dim_order_reversed": ("off = off * g->in[i] + q;", "off = off + q * (i == 0 ? 1 : g->in[0]);"),
    "min_axis_always_depth": ("const int r = min_dim - 2,", "const int r = 0 * min_dim,"),
    "kept_axes_swapped": ("a = (r == 0) ? 1 : 0, b = (r == 2) ? 1 : 2;", "b = (r == 0) ? 1 : 0, a = (r == 2) ? 1 : 2;"),
    "group_offset_dropped": ("(n * g->G * g->C + grp * g->C + c)", "(n * g->G * g->C + c)"),
    "group_of_channel_wrong": ("const int64_t grp = o / (g->K / g->G);", "const int64_t grp = o % g->G;"),
}

CHILD = r"""
import sys, traceback
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import test_oracle as t
checks = [t.test_page_worked_shapes, t.test_out_dims_brute_force_count, t.test_read_once_conv1d_long_geometry,
          t.test_linearity_and_bias, t.test_fused_rows_sum_to_one_and_open_interval,
          t.test_fused_matches_torch_float64, t.test_fused_single_depth_is_softmax_of_conv]
checks += [lambda s=s: t.test_matches_torch_float64(s) for s in range(6)]
checks += [lambda m=m: t.test_fused_min_dim_matches_torch_float64(m) for m in (2, 3, 4)]
checks += [lambda a=a: t.test_grouped_matches_torch_float64(*a) for a in ((1, 2, 4, 6), (2, 3, 6, 3), (3, 4, 4, 8))]
checks += [lambda nd=nd: t.test_delta_kernel_selects_one_input(nd) for nd in (1, 2, 3)]
checks += [lambda nd=nd: t.test_all_ones_counts_in_bounds_taps(nd) for nd in (1, 3)]
failed = 0
for c in checks:
    try:
        c()
    except Exception:
        failed += 1
print("FAILED_PINS", failed)
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation site for {name} not found exactly once"
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "oracle_mut.c")
        so = os.path.join(td, "liboracle_mut.so")
        open(c, "w").write(src.replace(before, after))
        subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", so, c, "-lm"])
        env = dict(os.environ, ORACLE_SO=so)
        code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    # a crash of the child also counts as rejection
    if r.returncode != 0:
        return
    line = [l for l in r.stdout.splitlines() if l.startswith("FAILED_PINS")]
    assert line, r.stdout + r.stderr
    assert int(line[-1].split()[1]) > 0, f"mutant {name} passed every pin"
