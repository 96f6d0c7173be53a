"""Plant plausible mistakes in a copy of the oracle and check the pins catch them.

Each mutation edits one spot of a *copy* of the oracle's C source (a flipped
comparison, a dropped term, a wrong index or sign), compiles it on the CPU and
runs the pin tests against it in a child process.  A mutation survives only if
every pin still passes; none may.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moonep_oracle.c")

MUTATIONS = {
    "receiver_not_lowest": ("for (int j = 0; j < R; j++) if (rem[j] < C) { recv = j; break; }",
                            "for (int j = R - 1; j >= 0; j--) if (rem[j] < C) { recv = j; break; }"),
    "donor_not_lowest": ("for (int j = 0; j < R; j++) if (rem[j] > C) { donor = j; break; }",
                         "for (int j = R - 1; j >= 0; j--) if (rem[j] > C) { donor = j; break; }"),
    "keep_drops_donations": ("for (int j = 0; j < R; j++) keep[j] = G[j] - donated[j];",
                             "for (int j = 0; j < R; j++) keep[j] = (G[j] < C ? G[j] : C);"),
    "padding_overcounts": ("int64_t padded = (n + tp - 1) / tp * tp;",
                           "int64_t padded = (n + tp) / tp * tp;"),
    "zero_fill_off_by_one": ("zfr[((int64_t)j * EB + x) * 2 + 0] = (int32_t)(end + n);",
                             "zfr[((int64_t)j * EB + x) * 2 + 0] = (int32_t)(end + n - (n > 0));"),
    "dup_sign_encoding": ("dst[base + k] = primary ? (int32_t)g : (int32_t)(-(g + 1));",
                          "dst[base + k] = primary ? (int32_t)g : (int32_t)(-g);"),
    "dup_rule_any_rank": ("if (route_rank[base + k2] == j) primary = 0;",
                          "if (route_rank[base + k2] == j && k2 == k - 1) primary = 0;"),
    "q_order_s_before_r": ("  for (int r = 0; r < R; r++)\n    for (int s = 0; s < S; s++)\n      for (int k = 0; k < K; k++) {\n        int64_t id = (int64_t)r * C + (int64_t)s * K + k;\n        int e = topk[id];\n        int h",
                           "  for (int s = 0; s < S; s++)\n    for (int r = 0; r < R; r++)\n      for (int k = 0; k < K; k++) {\n        int64_t id = (int64_t)r * C + (int64_t)s * K + k;\n        int e = topk[id];\n        int h"),
    "slot_index_transposed": ("int64_t slot = (int64_t)E + (int64_t)j * B + b;",
                              "int64_t slot = (int64_t)E + (int64_t)b * R + j;"),
    "combine_double_counts_k0": ("for (int k = 1; k < K; k++) acc = acc + bf16_to_f32(y[decode_row(d[k]) * H + c]);",
                                 "for (int k = 0; k < K; k++) acc = acc + bf16_to_f32(y[decode_row(d[k]) * H + c]);"),
    "combine_decodes_minus_d": ("for (int k = 1; k < K; k++) acc = acc + bf16_to_f32(y[decode_row(d[k]) * H + c]);",
                                "for (int k = 1; k < K; k++) acc = acc + bf16_to_f32(y[(d[k] < 0 ? -d[k] : d[k]) * H + c]);"),
    "bf16_truncates": ("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;",
                       "if (lower > 0x8000u) upper += 1u;"),
    "reduce_drops_seed": ("float acc = Gh[(int64_t)e * HHp + c];", "float acc = 0.0f;"),
    "reduce_keeps_slots": ("for (int64_t c = c0; c < c1; c++) Gs[(int64_t)i * HHp + c] = 0.0f;",
                           "for (int64_t c = c0; c < c1; c++) Gs[(int64_t)i * HHp + c] = Gs[(int64_t)i * HHp + c];"),
    "prefetch_skips_check": ("if (e < 0) continue;\n      int64_t slot", "if (e < 0) e = 0;\n      int64_t slot"),
    "prefetch_bytes_wrong_slot": ("const int64_t dst_row = (int64_t)E + (int64_t)j * B + b;",
                                  "const int64_t dst_row = (int64_t)E + (int64_t)b * R + j;"),
    "prefetch_bytes_copies_unused": ("      if (e < 0) continue;\n      const int64_t dst_row",
                                     "      if (e < 0) e = 0;\n      const int64_t dst_row"),
    "prepare_pad_off_by_one": ("      if (s >= n) {\n        if (hidden)", "      if (s > n) {\n        if (hidden)"),
    "prepare_keeps_invalid_weight": ("          topk[i] = 0;\n          if (w) w[i] = 0.0f;", "          topk[i] = 0;"),
    "prepare_counts_before_padding": ("    if (tpe) {\n      for (int e = 0; e < E; e++) tpe[(int64_t)r * E + e] = 0;",
                                      "    if (tpe) {\n      for (int e = 0; e < E; e++) tpe[(int64_t)r * E + e] = (e == 0) ? -(S - n) * K : 0;"),
    "fold_takes_other_ranks": ("          if (d[k2] < 0 && decode_row(d[k2]) / NvS == j)\n            acc = acc",
                               "          if (1)\n            acc = acc"),
    "primaries_combine_adds_duplicates": ("        if (d[k] >= 0) acc = acc + bf16_to_f32(y[(int64_t)d[k] * H + c]);",
                                          "        acc = acc + bf16_to_f32(y[decode_row(d[k]) * H + c]);"),
    "dispatch_no_weight_zero": ("if (w_out) w_out[g] = 0.0f;", "if (w_out) w_out[g] = w_out[g];"),
    "cu_exclusive": ("cu[(int64_t)j * EB + x] = (int32_t)end;", "cu[(int64_t)j * EB + x] = (int32_t)(end - padded);"),
    "slots_filled_from_end": ("etc[(int64_t)j * B + nslots] = e;", "etc[(int64_t)j * B + (B - 1 - nslots)] = e;"),
    # summation orders
    "combine_reversed_k": ("float acc = bf16_to_f32(y[decode_row(d[0]) * H + c]);\n      for (int k = 1; k < K; k++) acc = acc + bf16_to_f32(y[decode_row(d[k]) * H + c]);",
                           "float acc = bf16_to_f32(y[decode_row(d[K - 1]) * H + c]);\n      for (int k = K - 2; k >= 0; k--) acc = acc + bf16_to_f32(y[decode_row(d[k]) * H + c]);"),
    "combine_pairwise": ("float acc = bf16_to_f32(y[decode_row(d[0]) * H + c]);\n      for (int k = 1; k < K; k++) acc = acc + bf16_to_f32(y[decode_row(d[k]) * H + c]);",
                         "float v[64];\n      for (int k = 0; k < K; k++) v[k] = bf16_to_f32(y[decode_row(d[k]) * H + c]);\n"
                         "      for (int w = 1; w < K; w *= 2) for (int k = 0; k + w < K; k += 2 * w) v[k] = v[k] + v[k + w];\n"
                         "      float acc = v[0];"),
    "combine_fp64_accumulate": ("float acc = bf16_to_f32(y[decode_row(d[0]) * H + c]);\n      for (int k = 1; k < K; k++) acc = acc + bf16_to_f32(y[decode_row(d[k]) * H + c]);",
                                "double acc = bf16_to_f32(y[decode_row(d[0]) * H + c]);\n      for (int k = 1; k < K; k++) acc = acc + bf16_to_f32(y[decode_row(d[k]) * H + c]);"),
    "reduce_reversed_rank_slot": ("      for (int j = 0; j < R; j++)\n        for (int b = 0; b < B; b++)\n          if (etc[j * B + b] == e)",
                                  "      for (int j = R - 1; j >= 0; j--)\n        for (int b = B - 1; b >= 0; b--)\n          if (etc[j * B + b] == e)"),
    "reduce_slot_major": ("      for (int j = 0; j < R; j++)\n        for (int b = 0; b < B; b++)\n          if (etc[j * B + b] == e)",
                          "      for (int b = 0; b < B; b++)\n        for (int j = 0; j < R; j++)\n          if (etc[j * B + b] == e)"),
    "reduce_seed_last": ("float acc = Gh[(int64_t)e * HHp + c];\n      for (int j = 0; j < R; j++)\n        for (int b = 0; b < B; b++)\n          if (etc[j * B + b] == e) acc = acc + Gs[((int64_t)j * B + b) * HHp + c];",
                         "float acc = 0.0f;\n      for (int j = 0; j < R; j++)\n        for (int b = 0; b < B; b++)\n          if (etc[j * B + b] == e) acc = acc + Gs[((int64_t)j * B + b) * HHp + c];\n      acc = acc + Gh[(int64_t)e * HHp + c];"),
    "fold_reversed_duplicates": ("        for (int k2 = k + 1; k2 < K; k2++)\n          if (d[k2] < 0 && decode_row(d[k2]) / NvS == j)\n            acc = acc",
                                 "        for (int k2 = K - 1; k2 > k; k2--)\n          if (d[k2] < 0 && decode_row(d[k2]) / NvS == j)\n            acc = acc"),
    "primaries_combine_reversed": ("      float acc = bf16_to_f32(y[(int64_t)d[0] * H + c]);  /* route 0 is always primary */\n      for (int k = 1; k < K; k++)\n        if (d[k] >= 0)",
                                   "      float acc = 0.0f;\n      for (int k = K - 1; k >= 0; k--)\n        if (d[k] >= 0)"),
}

CHILD = r'''
import json, sys, traceback
sys.path.insert(0, {root!r})
import numpy as np
import oracle
from tests import test_oracle_pins as P
from combine_moonep_plan_gb300 import workloads as wl
o = oracle.Oracle({lib!r})
pins = [
    ("golden_dup", lambda: P.test_golden_plan(o, "plan_two_ranks_dup.json")),
    ("golden_chain", lambda: P.test_golden_plan(o, "plan_chain_donor_turns_receiver.json")),
    ("invariants_tiny_zipf", lambda: P.test_oracle_plan_invariants(o, "tiny", wl.SHAPES["tiny"], "zipf3")),
    ("invariants_kimi_hot", lambda: P.test_oracle_plan_invariants(o, "kimi", wl.Shape("k", R=8, E=384, K=8, S=64, H=8, Hp=8, B=48, tp=128, weights="sigmoid"), "hot")),
    ("stable_sort", lambda: P.test_balanced_routing_is_a_stable_sort(o, "tiny")),
    ("restate_kimi", lambda: P.test_oracle_matches_sort_based_restatement(o, "kimi_k2", "hot30")),
    ("restate_mixtral", lambda: P.test_oracle_matches_sort_based_restatement(o, "mixtral", 3.0)),
    ("restate_small", lambda: [P.test_oracle_matches_restatement_random_small(o, i) for i in range(8)]),
    ("slots_error", lambda: P.test_slots_error_when_b_below_group_size(o)),
    ("dispatch_scatter", lambda: P.test_dispatch_is_a_scatter(o)),
    ("k_times_x", lambda: P.test_identity_expert_combine_is_k_times_x(o)),
    ("combine_bound", lambda: P.test_combine_within_one_ulp_of_exact_sum(o)),
    ("bf16_torch", lambda: P.test_bf16_rounding_matches_torch(o)),
    ("prefetch_copy", lambda: P.test_prefetch_copies_home_rows(o)),
    ("prefetch_bytes", lambda: P.test_prefetch_bytes_copies_packed_rows(o)),
    ("prefetch_bytes_window", lambda: P.test_prefetch_bytes_of_bf16_rows_is_the_bf16_prefetch(o)),
    ("folded_hand", lambda: P.test_folded_combine_hand_example(o)),
    ("folded_nodup", lambda: P.test_folded_combine_equals_direct_without_duplicates(o)),
    ("folded_top2", lambda: P.test_folded_identity_combine_is_k_times_x_for_top2(o)),
    ("folded_bound", lambda: P.test_folded_combine_error_bound(o)),
    ("prepare_hand", lambda: P.test_prepare_hand_example(o)),
    ("prepare_random", lambda: P.test_prepare_random_properties(o)),
    ("reduce_const", lambda: P.test_reduce_constant_fill_counts_copies(o)),
    ("reduce_int", lambda: P.test_reduce_integer_values_exact(o)),
    ("combine_k_order", lambda: [P.test_combine_sums_in_k_order(o, v, w) for v, w in P.COMBINE_ORDER_CASES]),
    ("combine_k_order_ranks", lambda: P.test_combine_k_order_across_ranks(o)),
    ("fold_k_order", lambda: P.test_fold_sums_duplicates_in_k_order(o)),
    ("fold_two_groups", lambda: P.test_fold_k_order_with_two_groups(o)),
    ("primaries_k_order", lambda: P.test_primaries_combine_sums_in_k_order(o)),
    ("reduce_order", lambda: [P.test_reduce_sums_in_rank_slot_order(o, *c) for c in P.REDUCE_ORDER_CASES]),
]
failed = []
for name, fn in pins:
    try:
        fn()
    except Exception:
        failed.append(name)
print(json.dumps(failed))
'''


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, name):
    import oracle
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = str(tmp_path / "libmutant.so")
    oracle.compile_c(str(mutated), lib, include_dir=os.path.dirname(SRC))
    res = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, lib=lib)],
                         capture_output=True, text=True, timeout=300)
    if res.returncode != 0:
        # a crash of the mutant also exposes it
        return
    failed = json.loads(res.stdout.strip().splitlines()[-1])
    assert failed, f"mutation {name} survived every pin"


def test_unmutated_oracle_passes_every_pin(tmp_path):
    import oracle
    lib = oracle.build()
    res = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, lib=lib)],
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    assert json.loads(res.stdout.strip().splitlines()[-1]) == []
