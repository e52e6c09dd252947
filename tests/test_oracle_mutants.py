"""Mutation check of the oracle's pins.

Each case plants one plausible mistake in a copy of oracle/q4_oracle.c (a
swapped constant, a dropped term, a flipped sign or comparison, a wrong
operand order), builds it, and runs the pin tests that should notice, with
the oracle pointed at the mutant (Q4_ORACLE_LIB).  Every mutant must make
those pins fail; the unmodified source, built the same way, must pass them.
Nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "q4_oracle.c")

STEP = "tests/test_oracle_step.py"
ROUND = "tests/test_oracle_rounding.py"
PRIM = "tests/test_oracle_primitives.py"
CLIP = "tests/test_oracle_clip.py"
FACT = "tests/test_oracle_factored.py"

MUTANTS = {
    # AdamW recurrences and update
    "m_uses_beta2": ("float mm = fmaf(s.beta1, m, s.omb1 * g);", "float mm = fmaf(s.beta2, m, s.omb1 * g);", [STEP]),
    "v_drops_square": ("vv = fmaf(s.beta2, v, s.omb2 * (g * g));", "vv = fmaf(s.beta2, v, s.omb2 * g);", [STEP]),
    "no_bias_correction": ("return 1.0f / (sqrtf(x) * s->c2 + s->eps);", "return 1.0f / (sqrtf(x) + s->eps);",
                           [STEP]),
    "decay_sign": ("float th = T->param[e] * s.decay - s.step_size * (mm * rr);",
                   "float th = T->param[e] * s.decay + s.step_size * (mm * rr);", [STEP]),
    # block scale and EDEN
    "absmax_without_abs": ("float ax = fabsf(x[i]);", "float ax = x[i];", [STEP]),
    "eden_inverted": ("return s * (A / B);", "return s * (B / A);", [STEP]),
    # rounding rules
    "state_sr_direction": ("return (u * (a[k + 1] - a[k]) < (x - a[k])) ? k + 1 : k;",
                           "return (u * (a[k + 1] - a[k]) > (x - a[k])) ? k + 1 : k;", [ROUND]),
    "update_sr_gap_sign": ("return (u * (rk - rk1) < (rk - r)) ? k + 1 : k;",
                           "return (u * (rk - rk1) < (r - rk)) ? k + 1 : k;", [ROUND]),
    "rtn_tie_up": ("if (x > T[k]) c++;", "if (x >= T[k]) c++;", [ROUND]),
    # primitives
    "philox_multiplier": ("(uint64_t)0xD2511F53u * (uint64_t)c0", "(uint64_t)0xD2511F55u * (uint64_t)c0", [PRIM]),
    "bf16_truncates": ("return (uint16_t)((u + 0x7fffu + lsb) >> 16);", "return (uint16_t)(u >> 16);", [PRIM]),
    # factored statistics
    "row_mean_divisor": ("float mean = (float)(row_sums[i] / (double)cols);",
                         "float mean = (float)(row_sums[i] / (double)rows);",
                         [STEP]),
    # gradient-norm clipping
    "sqnorm_lane_order": ("q[l] = ((sq[0] + sq[1]) + (sq[2] + sq[3])) + ((sq[4] + sq[5]) + (sq[6] + sq[7]));",
                          "q[l] = ((sq[0] + sq[2]) + (sq[1] + sq[3])) + ((sq[4] + sq[6]) + (sq[5] + sq[7]));",
                          [CLIP]),
    "clip_not_clamped": ("return (c >= 1.0f) ? 1.0f : c;", "return (c >= 1.0f) ? c : 1.0f;", [CLIP]),
    "factored_stats_ignore_clip": ("double g = clipped(grad[e], clip);", "double g = clipped(grad[e], 1.0f);",
                                   [CLIP]),
    # draws, phases and variants
    "draw_purpose_bit": ("(uint32_t)(idx >> 34) | (purpose << 28)", "(uint32_t)(idx >> 34) | (purpose << 27)", [PRIM]),
    "lm_head_sr_in_every_phase": ("(T->flags & OT_LM_HEAD) && (call_flags & OS_LM_HEAD_SR_ACTIVE) && recipe != OR_TORCHAO",
                                  "(T->flags & OT_LM_HEAD) && recipe != OR_TORCHAO", [STEP]),
    "torchao_head_sr": ("(call_flags & OS_LM_HEAD_SR_ACTIVE) && recipe != OR_TORCHAO)",
                        "(call_flags & OS_LM_HEAD_SR_ACTIVE))", [STEP]),
    "next_r_same_step_c2": ("s.rc = hn[1];", "s.rc = s.c2;", [STEP]),
    "update_rtn_direction": ("return ((r - rk1) < (rk - r)) ? k + 1 : k;", "return ((r - rk1) > (rk - r)) ? k + 1 : k;",
                             [ROUND, STEP]),
    "column_mean_divisor": ("float mean = (float)(col_sums[j] / (double)rows);",
                            "float mean = (float)(col_sums[j] / (double)cols);",
                            [STEP]),
    # factored second moment in the step
    "factored_vhat_times_rbar": ("(T->v_row[ri] * T->v_col[cj]) / rbar;", "(T->v_row[ri] * T->v_col[cj]) * rbar;",
                                 [FACT]),
    "factored_row_column_swap": ("int64_t ri = (fbase + e) / cols, cj = (fbase + e) % cols;",
                                 "int64_t ri = (fbase + e) % cols, cj = (fbase + e) / cols;", [FACT]),
    # data-parallel shards of a factored parameter
    "shard_step_ignores_offset": ("int64_t ri = (fbase + e) / cols, cj = (fbase + e) % cols;",
                                  "int64_t ri = e / cols, cj = e % cols;", [FACT]),
    "shard_partials_ignore_offset": ("int64_t ge = fbase + e;", "int64_t ge = e;", [FACT]),
    "factored_zero_rbar_gives_one": ("vv = (rbar == 0.0f) ? 0.0f :", "vv = (rbar == 0.0f) ? 1.0f :", [FACT]),
    "factored_rbar_from_columns": ("for (int64_t i = 0; i < rows; ++i) acc += R[i];",
                                   "for (int64_t i = 0; i < rows; ++i) acc += C[i % cols];", [FACT]),
    "factored_1d_v_in_dyn4": (
        "const float* Lv = (recipe == OR_ZIP_SR) ? cb->dyn4 : (recipe == OR_TORCHAO) ? cb->lin4nz : cb->dyn4nz;\n"
        "    const float* tv = (recipe == OR_ZIP_SR) ? cb->dyn4_t : (recipe == OR_TORCHAO) ? cb->lin4nz_t : cb->dyn4nz_t;",
        "const float* Lv = (recipe == OR_ZIP_SR || recipe == OR_FACTORED) ? cb->dyn4 : (recipe == OR_TORCHAO) ? "
        "cb->lin4nz : cb->dyn4nz;\n"
        "    const float* tv = (recipe == OR_ZIP_SR || recipe == OR_FACTORED) ? cb->dyn4_t : (recipe == OR_TORCHAO) ? "
        "cb->lin4nz_t : cb->dyn4nz_t;", [FACT]),
}


# Mistakes in the Python half of the oracle (the codebook constructions):
# the pins run from a copy of oracle/ and tests/ with the mistake planted.
PY_MUTANTS = {
    "nf4_delta": ("delta = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0)", "delta = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 31.0)"),
    "dyn4_fraction_index": ("vals.append(10.0 ** (-e) * (0.1 + 0.9 * (j + 1) / 2 ** f))",
                            "vals.append(10.0 ** (-e) * (0.1 + 0.9 * j / 2 ** f))"),
    "sdyn4_left_endpoints": ("mags.append(10.0 ** (i - 2) * (lo + hi) / 2.0)", "mags.append(10.0 ** (i - 2) * lo)"),
}


def _build(src_text: str, out_dir) -> str:
    c = os.path.join(out_dir, "q4_oracle_mut.c")
    so = os.path.join(out_dir, "liboracle_mut.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-o", so,
                    c, "-lm"], check=True)
    return so


def _run_pins(so: str, files):
    env = dict(os.environ, Q4_ORACLE_LIB=so)
    return subprocess.run([sys.executable, "-m", "pytest", *files, "-x", "-q", "-m", "not gpu",
                           "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True)


def test_unmodified_oracle_passes_the_pins_through_the_override(tmp_path):
    with open(SRC) as f:
        so = _build(f.read(), str(tmp_path))
    r = _run_pins(so, [CLIP, PRIM, FACT])
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name, tmp_path):
    old, new, files = MUTANTS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    so = _build(src.replace(old, new), str(tmp_path))
    r = _run_pins(so, files)
    assert r.returncode == 1, f"{name} survived the pins:\n{r.stdout[-1500:]}"


@pytest.mark.parametrize("name", sorted(PY_MUTANTS) + ["unmodified"])
def test_planted_codebook_mistake_fails_a_pin(name, tmp_path):
    import shutil
    old, new = PY_MUTANTS.get(name, ("delta = 1.0 - 0.5", "delta = 1.0 - 0.5"))
    for d in ("oracle", "tests"):
        shutil.copytree(os.path.join(ROOT, d), os.path.join(tmp_path, d),
                        ignore=shutil.ignore_patterns("_build", "__pycache__", "*.so"))
    cb = os.path.join(tmp_path, "oracle", "codebooks.py")
    with open(cb) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found"
    with open(cb, "w") as f:
        f.write(src.replace(old, new))
    with open(SRC) as f:
        so = _build(f.read(), str(tmp_path))      # the C half unchanged
    env = dict(os.environ, Q4_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_primitives.py", "-x", "-q",
                        "-m", "not gpu", "-p", "no:cacheprovider", "--rootdir", str(tmp_path)],
                       cwd=str(tmp_path), env=env, capture_output=True, text=True)
    if name == "unmodified":                     # the copied tree itself passes
        assert r.returncode == 0, r.stdout[-1500:]
    else:
        assert r.returncode == 1, f"{name} survived the pins:\n{r.stdout[-1500:]}"
