"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/hs_oracle.c (a flipped comparison, a
dropped update, an off-by-one), builds it with gcc into a temporary library, and runs the
pin suite against it in a child process. The child must report at least one failing pin.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "hs_oracle.c")

MUTANTS = [
    ("tie_to_highest_slot", "if (x->slot != y->slot) return x->slot < y->slot ? -1 : 1;",
     "if (x->slot != y->slot) return x->slot < y->slot ? 1 : -1;"),
    ("evict_newest_stamp", "if (x->stamp != y->stamp) return x->stamp < y->stamp ? -1 : 1;",
     "if (x->stamp != y->stamp) return x->stamp < y->stamp ? 1 : -1;"),
    ("free_slots_last", "if (x->occupied != y->occupied) return x->occupied < y->occupied ? -1 : 1;",
     "if (x->occupied != y->occupied) return x->occupied < y->occupied ? 1 : -1;"),
    ("clock_not_stored", "    lru_clock[r] = c;\n", "\n"),
    ("hit_not_refreshed", "        stamps[s] = c;\n        used[s] = 1;", "        used[s] = 1;"),
    ("newest_not_reserved", "if (cls[i] == E_VALID && tk[i] >= base) {", "if (cls[i] == E_VALID && tk[i] > base) {"),
    ("fast_path_off_by_one", "  if (S <= H) {\n      for", "  if (S < H) {\n      for"),
    ("victims_reversed", "int32_t v = cand[j].slot;", "int32_t v = cand[m - 1 - j].slot;"),
    ("token_as_host_row", "int64_t h = hcl[t];", "int64_t h = t;"),
    ("hit_wrong_row", "out[i] = checked_row(dbl[s], g->device_rows, err);\n        cls[i] = E_DONE;",
     "out[i] = checked_row(dbl[s + 1], g->device_rows, err);\n        cls[i] = E_DONE;"),
    ("resident_offset_wrong", "return (int64_t)p * g->page_size + t % g->page_size;",
     "return (int64_t)p * g->page_size + (t + 1) % g->page_size;"),
    ("sanitize_too_loose", "tokens[s] < -1 || tokens[s] >= base)", "tokens[s] < -1 || tokens[s] >= base + 1)"),
    ("backup_always_reserved", "if (row < 0) row = S <= H ? dbl[t] : dbl[H];", "if (row < 0) row = dbl[H];"),
    ("duplicates_not_rejected", "else if (first_at[t] >= 0)", "else if (first_at[t] >= 2000000000)"),
    ("misses_not_zero_filled", "else memset(dst, 0, (size_t)B);", "else (void)dst;"),
    ("invalidate_keeps_stamp", "  tokens[s] = -1;\n  stamps[s] = 0;\n}", "  tokens[s] = -1;\n}"),
    ("invalidate_fast_path_too", "  return S > g->hot_slots;\n}", "  return 1;\n}"),
    ("invalidate_skips_first_token", "for (int32_t k = offsets[r]; k < offsets[r + 1]; ++k)",
     "for (int32_t k = offsets[r] + 1; k < offsets[r + 1]; ++k)"),
    ("invalidate_row_is_token", "if (rows[j] == hcl[t]) {", "if (rows[j] == t) {"),
    ("gather_drops_last_layer", "for (int32_t l = first_layer; l < first_layer + num_layers; ++l) {",
     "for (int32_t l = first_layer; l < first_layer + num_layers - 1; ++l) {"),
    ("plan_drops_first_miss", "plan_dst[(int64_t)r * K + j] = d;", "plan_dst[(int64_t)r * K + j] = j == 0 ? -1 : d;"),
    ("leader_copies_every_layer", "for (int32_t l = 0; l < copy_layers; ++l) {",
     "for (int32_t l = 0; l < g->num_layers; ++l) {"),
    ("spec_one_reserved_row", "out[i] = checked_row(dbl[H + (tk[i] - base)], g->device_rows, err);",
     "out[i] = checked_row(dbl[H], g->device_rows, err);"),
    ("spec_marks_before_s0_only", "t <= base; ++t) tokens[t] = t;", "t < base; ++t) tokens[t] = t;"),
    ("spec_backup_first_reserved_row", "if (row < 0) row = t + 1 <= H ? dbl[t] : dbl[H + j];",
     "if (row < 0) row = t + 1 <= H ? dbl[t] : dbl[H];"),
    ("host_stride_ignored", "const int64_t stride = g->host_row_stride > 0 ? g->host_row_stride : g->row_bytes;",
     "const int64_t stride = g->row_bytes;"),
    ("duplicate_holder_highest_slot", "      if (holders[t] == 0) lowest_slot[t] = s;\n",
     "      lowest_slot[t] = s;\n"),
    ("spec_plans_share_one_slice", "copy_layers, plan_tokens ? plan_tokens + q * RK : NULL, plan_dst ? plan_dst + q * RK : NULL,",
     "copy_layers, plan_tokens, plan_dst,"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    csrc = tmp_path / "mutant.c"
    csrc.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", str(csrc), "-o", str(lib)])
    code = ("import sys; sys.path[:0] = [%r, %r]; import test_oracle_pins as t; "
            "n = t.run_all_pins(); print('failed pins:', n); sys.exit(0 if n else 3)"
            % (ROOT, os.path.join(ROOT, "tests")))
    env = dict(os.environ, HS_ORACLE_LIB=str(lib))
    p = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode != 3, f"mutant {name} survived every pin:\n{p.stdout}\n{p.stderr}"
    assert p.returncode == 0, f"mutant {name}: pin run crashed (rc {p.returncode}):\n{p.stderr[-2000:]}"


# Planted mistakes in the sparse-MLA decode oracle (oracle/sparse_mla.py). Each copy is loaded
# as a module of its own and the consumer's pins (tests/test_oracle_sparse_mla.py) run against
# it in this process; at least one must fail.
MLA_SRC = os.path.join(ROOT, "oracle", "sparse_mla.py")
MLA_MUTANTS = [
    ("e4m3_bias_8", "np.exp2(e.astype(np.float64) - 7.0)", "np.exp2(e.astype(np.float64) - 8.0)"),
    ("e4m3_subnormal_scale", "m / 8.0 * 2.0 ** -6", "m / 8.0 * 2.0 ** -7"),
    ("e4m3_nan_missed", "(e == 0xF) & (m == 7)", "(e == 0xF) & (m == 8)"),
    ("scales_interleaved", "np.repeat(scales, SCALE_BLOCK, axis=1)", "np.tile(scales, SCALE_BLOCK)"),
    ("rope_left_out", " + q[r, :, D_LATENT:] @ rope.T)", ")"),
    ("scores_unscaled", "s = sm_scale * (", "s = 1.0 * ("),
    ("lse_without_max", "lse[r] = (smax + np.log(z))[:, 0]", "lse[r] = np.log(z)[:, 0]"),
    ("masked_rows_kept", "rows = out_rows[r][out_rows[r] >= 0]", "rows = out_rows[r][out_rows[r] >= -1]"),
    ("softmax_over_heads", "z = e.sum(axis=1, keepdims=True)", "z = e.sum(axis=0, keepdims=True)"),
    ("rope_low_half", "(bits.astype(np.uint32) << 16)", "(bits.astype(np.uint32) << 0)"),
]


@pytest.mark.parametrize("name,old,new", MLA_MUTANTS, ids=[m[0] for m in MLA_MUTANTS])
def test_mla_mutant_is_caught(name, old, new):
    import types

    import test_oracle_sparse_mla as pins

    src = open(MLA_SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mod = types.ModuleType("sparse_mla_mutant")
    exec(compile(src.replace(old, new), f"<{name}>", "exec"), mod.__dict__)
    failed = 0
    saved = pins.M
    try:
        pins.M = mod
        for fn in [getattr(pins, k) for k in dir(pins) if k.startswith("test_")]:
            try:
                with np.errstate(all="ignore"):
                    fn()
            except Exception:  # an assertion, or the mistake breaking a shape
                failed += 1
    finally:
        pins.M = saved
    assert failed, f"mutant {name} survived every pin"
