"""Planted mistakes in the fp64 oracle, for checking that its pins catch them.

Each entry of ``MUTANTS`` is (name, original text, replacement) for one
plausible slip in ``oracle/bsfa_oracle.py``: a flipped comparison, a dropped
term, a wrong index, a swapped visiting order.  The original text must occur
exactly once in the oracle's source, so a mutant that no longer applies is an
error rather than a silent pass.

``GUARD_MUTANTS`` does the same for ``oracle/guard.py``, the guard band that
keeps generated thresholds clear of ties; its pins are
``tests/test_oracle_guard.py``.

Loaded as a pytest plugin (``-p tests.oracle_mutants``) with the environment
variable ``BSFA_ORACLE_MUTANT`` naming one entry, it builds that mutant of the
module on the CPU and installs it in place of ``oracle.bsfa_oracle`` (or
``oracle.guard``) for the test session; the files are not touched.  Without
the variable it does nothing.
"""
import os
import sys
import types

ENV = "BSFA_ORACLE_MUTANT"

MUTANTS = [
    # block geometry and the score matrix
    ("partial_blocks_as_candidates", "if (j + 1) * Bk <= first_row:",
     "if j * Bk <= first_row:"),
    ("candidate_when_fully_visible", "if (j + 1) * Bk <= first_row:",
     "if (j + 1) * Bk - 1 <= first_row:"),
    ("last_row_window_shrinks", "if first_key <= last_row:", "if first_key < last_row:"),
    ("causal_mask_excludes_self", "s = np.where(cols[None, :] <= rows[:, None], s, NEG_INF)",
     "s = np.where(cols[None, :] < rows[:, None], s, NEG_INF)"),
    ("no_softmax_scale", "s = sigma * (q_h[r0:r1] @ k_h[:r1].T)", "s = q_h[r0:r1] @ k_h[:r1].T"),
    ("tile_mean_not_max", "return float(np.max(s[:, j * Bk:(j + 1) * Bk]))",
     "return float(np.mean(s[:, j * Bk:(j + 1) * Bk]))"),
    ("tile_max_first_row_only", "return float(np.max(s[:, j * Bk:(j + 1) * Bk]))",
     "return float(np.max(s[0, j * Bk:(j + 1) * Bk]))"),
    # threshold gate
    ("gt_instead_of_ge", "keep[j] = tile_max(s, j, Bk) >= T_hi",
     "keep[j] = tile_max(s, j, Bk) > T_hi"),
    ("diagonal_gated",
     "            keep[j] = True\n        else:\n            keep[j] = tile_max(s, j, Bk) >= T_hi",
     "            keep[j] = tile_max(s, j, Bk) >= T_hi\n        else:\n"
     "            keep[j] = tile_max(s, j, Bk) >= T_hi"),
    ("gqa_modulo", "return h // (Hq // Hkv)", "return h % Hkv"),
    ("threshold_by_kv_head",
     "T_hi = float(thresholds[h][threshold_index(i, len(thresholds[h]))])",
     "T_hi = float(thresholds[kh][threshold_index(i, len(thresholds[kh]))])"),
    ("threshold_index_wraps", "return min(i, nT - 1)", "return i % nT"),
    # renormalised attention
    ("lse_drops_max", "lse = (M + np.log(Z))[:, 0]", "lse = np.log(Z)[:, 0]"),
    ("skipped_keys_in_denominator", "Z = np.sum(e, axis=1, keepdims=True)",
     "Z = np.sum(np.exp(s - M), axis=1, keepdims=True)"),
    ("output_not_normalised", "out = (e @ vals) / Z", "out = e @ vals"),
    # calibration
    ("kth_plus_one", "return float(sorted(values, reverse=True)[k - 1])",
     "return float(sorted(values, reverse=True)[min(k, len(values) - 1)])"),
    ("kth_smallest", "return float(sorted(values, reverse=True)[k - 1])",
     "return float(sorted(values)[k - 1])"),
    ("short_history_not_minus_inf",
     "    if len(values) < k:\n        return NEG_INF\n"
     "    return float(sorted(values, reverse=True)[k - 1])",
     "    if not values:\n        return NEG_INF\n"
     "    return float(sorted(values, reverse=True)[min(k, len(values)) - 1])"),
    ("calibration_sums_samples", "T[:, h, i] = acc / N", "T[:, h, i] = acc"),
    # lambda gate
    ("lambda_running_max_frozen", "            m = np.maximum(m, rowmax)",
     "            m = np.where(np.isinf(m), rowmax, m)"),
    ("lambda_one_row_skips", "kept = not bool(np.all(stat < log_lambda))",
     "kept = not bool(np.any(stat < log_lambda))"),
    ("lambda_skip_at_bound", "kept = not bool(np.all(stat < log_lambda))",
     "kept = not bool(np.all(stat <= log_lambda))"),
    ("lambda_log2_bound", "kept = not bool(np.all(stat < log_lambda))",
     "kept = not bool(np.all(stat < log_lambda / math.log(2.0)))"),
    ("lambda_tile_max_statistic", "rowmax = np.max(s[:, j * Bk:(j + 1) * Bk], axis=1)",
     "rowmax = np.full(s.shape[0], np.max(s[:, j * Bk:(j + 1) * Bk]))"),
    ("lambda_descending", "return cands + diags", "return cands[::-1] + diags"),
    ("lambda_max_raised_by_skipped_block",
     "        keep[j] = kept\n        if kept:\n            m = np.maximum(m, rowmax)",
     "        keep[j] = kept\n        m = np.maximum(m, rowmax)"),
    ("lambda_statistic_after_update",
     "        if trace is not None:\n            trace.append((j, m.copy(), rowmax.copy(), kept))\n"
     "        keep[j] = kept\n        if kept:\n            m = np.maximum(m, rowmax)",
     "        keep[j] = kept\n        if kept:\n            m = np.maximum(m, rowmax)\n"
     "        if trace is not None:\n            trace.append((j, m.copy(), rowmax.copy(), kept))"),
    ("lambda_statistic_min_over_rows", "out.append((j, float(np.max(rowmax - m_before))))",
     "out.append((j, float(np.min(rowmax - m_before))))"),
    ("lambda_statistic_tile_wide", "out.append((j, float(np.max(rowmax - m_before))))",
     "out.append((j, float(np.max(rowmax) - np.max(m_before))))"),
    ("lambda_diagonal_first", "return cands + diags", "return diags + cands"),
    # whole-head forms
    ("block_maxima_partial_candidates", "        ncand = (i * Bq) // Bk  # key blocks j with",
     "        ncand = (i * Bq + Bk - 1) // Bk  # key blocks j with"),
    ("block_maxima_first_row",
     "out[i, :ncand] = torch.amax(sT.reshape(ncand, Bk * (r1 - r0)), dim=1).numpy()",
     "out[i, :ncand] = torch.amax(sT.reshape(ncand, Bk, r1 - r0), dim=1)[:, 0].numpy()"),
    ("whole_head_threshold_gt", "keep[i, j] = smax[i, j] >= t", "keep[i, j] = smax[i, j] > t"),
    ("whole_head_diagonal_gated", "            elif cls == DIAGONAL:\n                keep[i, j] = True",
     "            elif cls == DIAGONAL:\n                keep[i, j] = smax[i, j] >= t"),
    ("whole_head_lambda_gt", "            if st >= log_lambda:", "            if st > log_lambda:"),
    ("whole_head_lambda_max_on_skip",
     "                keep[i, j] = True\n                m = np.maximum(m, rowmax[j])",
     "                keep[i, j] = True\n            m = np.maximum(m, rowmax[j])"),
    # mean correction
    ("stand_in_without_count", "logits[:, n] = sigma * (q_rows @ kbar) + math.log(c1 - c0)",
     "logits[:, n] = sigma * (q_rows @ kbar)"),
    ("stand_in_without_scale", "logits[:, n] = sigma * (q_rows @ kbar) + math.log(c1 - c0)",
     "logits[:, n] = q_rows @ kbar + math.log(c1 - c0)"),
    ("stand_ins_for_kept_blocks", "if not kept and block_class(i, j, Bq, Bk, L) == CANDIDATE]",
     "if block_class(i, j, Bq, Bk, L) == CANDIDATE]"),
    ("stand_in_value_first_row", "vbar[n] = v_h[c0:c1].mean(axis=0)", "vbar[n] = v_h[c0]"),
    ("stand_in_key_first_row", "kbar = k_h[c0:c1].mean(axis=0)", "kbar = k_h[c0]"),
    # packing and accounting
    ("varlen_drops_last_sequence", "for b in range(len(cu_seqlens) - 1):",
     "for b in range(len(cu_seqlens) - 2):"),
    ("flops_without_pv",
     "return F * (float(np.count_nonzero(visible)) + float(np.count_nonzero(keep)))",
     "return F * float(np.count_nonzero(visible))"),
]

GUARD_MUTANTS = [
    ("guard_gqa_modulo", "c = orc.candidate_maxima(qs[h], ks_[h // g], i, Bq, Bk, sigma)",
     "c = orc.candidate_maxima(qs[h], ks_[h % Hkv], i, Bq, Bk, sigma)"),
    ("guard_keys_without_reuse",
     "out.setdefault((h, orc.threshold_index(i, nT)), []).extend(c)",
     "out.setdefault((h, i), []).extend(c)"),
    ("guard_any_gap", "idx = np.nonzero(gaps >= min_gap)[0]", "idx = np.nonzero(gaps > 0)[0]"),
    ("guard_no_low_end", "cands = [vals[0] - margin, vals[-1] + margin]",
     "cands = [vals[-1] + margin]"),
    ("guard_moves_clear_values",
     "if vals.size == 0 or not np.any(np.abs(vals - x) < band):", "if vals.size == 0:"),
]

_ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")
ORACLE_PATH = os.path.join(_ORACLE_DIR, "bsfa_oracle.py")
GUARD_PATH = os.path.join(_ORACLE_DIR, "guard.py")


def target(name: str):
    """(module name under ``oracle``, source path, pin file) of mutant ``name``."""
    if any(m[0] == name for m in MUTANTS):
        return "bsfa_oracle", ORACLE_PATH, "tests/test_oracle_pins.py"
    if any(m[0] == name for m in GUARD_MUTANTS):
        return "guard", GUARD_PATH, "tests/test_oracle_guard.py"
    raise KeyError(name)


def mutated_source(name: str) -> str:
    """The target module's source with mutant ``name`` applied."""
    entry = [m for m in MUTANTS + GUARD_MUTANTS if m[0] == name]
    if len(entry) != 1:
        raise KeyError(name)
    _, old, new = entry[0]
    with open(target(name)[1]) as f:
        src = f.read()
    if src.count(old) != 1:
        raise ValueError(f"mutant {name}: the original text occurs {src.count(old)} times")
    return src.replace(old, new)


def _install(name: str) -> None:
    import oracle
    mod_name, path, _ = target(name)
    mod = types.ModuleType(f"oracle.{mod_name}")
    mod.__file__ = path
    mod.__package__ = "oracle"
    sys.modules[f"oracle.{mod_name}"] = mod
    exec(compile(mutated_source(name), path, "exec"), mod.__dict__)
    setattr(oracle, mod_name, mod)


if os.environ.get(ENV):
    _install(os.environ[ENV])
