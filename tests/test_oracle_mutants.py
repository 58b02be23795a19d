"""Planted mistakes in the oracle must fail at least one pin (no GPU).

Each mutant is a copy of oracle.c with one plausible slip -- a dropped term,
a wrong index or sign, a transposed operand, a wrong rounding tie -- compiled
into a scratch directory.  A mutant that passes every pin would mean the pins
cannot tell that slip from the real oracle.
"""
import os

import pytest

import oracle
import pins

MUTANTS = {
    "ring_direction": ("x[(c + k) % P]", "x[(c + P - k) % P]"),
    "ring_start_rank": ("int c = (int)(e / L);", "int c = (int)((e / L + 1) % (size_t)P);"),
    "ring_dropped_rank": ("for (int k = 1; k < P; ++k) acc = combine(acc, x[(c + k) % P]",
                          "for (int k = 1; k < P - 1; ++k) acc = combine(acc, x[(c + k) % P]"),
    "chunk_not_16B": ("return round_up(per, vec_elems(dtype));", "return per;"),
    "sum_sign": ("acc.f = acc.f + x.f;", "acc.f = acc.f - x.f;"),
    "min_flipped": ("acc.f = (x.f < acc.f) ? x.f : acc.f;", "acc.f = (x.f > acc.f) ? x.f : acc.f;"),
    "int_min_unsigned": ("acc.u = (uint32_t)((b < a) ? b : a);",
                         "acc.u = (x.u < acc.u) ? x.u : acc.u;"),
    "tree_children_swapped": (
        "    if (l) acc = combine(acc, tree_value(x, l, P, t, dtype, op), dtype, op);\n"
        "    if (r) acc = combine(acc, tree_value(x, r, P, t, dtype, op), dtype, op);",
        "    if (r) acc = combine(acc, tree_value(x, r, P, t, dtype, op), dtype, op);\n"
        "    if (l) acc = combine(acc, tree_value(x, l, P, t, dtype, op), dtype, op);"),
    "tree_own_last": (
        "    acc_t acc = x[tree_owner(v, P, t)];\n    int l = tree_left(v), r = tree_right(v, P);\n"
        "    if (l) acc = combine(acc, tree_value(x, l, P, t, dtype, op), dtype, op);",
        "    int l = tree_left(v), r = tree_right(v, P);\n"
        "    acc_t acc = l ? tree_value(x, l, P, t, dtype, op) : x[tree_owner(v, P, t)];\n"
        "    if (l) acc = combine(acc, x[tree_owner(v, P, t)], dtype, op);"),
    "tree1_shift_wrong": ("return t == 0 ? v - 1 : v % P;", "return t == 0 ? v - 1 : (v + 1) % P;"),
    "tree_right_dropped": ("if (r) acc = combine(acc, tree_value(x, r, P, t, dtype, op), dtype, op);",
                           "(void)r;"),
    "tree_split_floor": ("size_t h = round_up((count + 1) / 2, vec_elems(dtype));",
                         "size_t h = round_up(count / 2, vec_elems(dtype));"),
    "rne_ties_away": ("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;",
                      "if (lower >= 0x8000u) upper += 1;"),
    "scale_dropped": ("    if (dtype != OR_I32 && scale != 1.0f) acc.f = acc.f * scale;\n    return acc;",
                      "    return acc;"),
    "only_rank0_written": ("algo, scale);\n        for (int r = 0; r < P; ++r) store_narrowed(recv[r], e, y, dtype);",
                           "algo, scale);\n        store_narrowed(recv[0], e, y, dtype);"),
    "bf16_widen_shift": ("uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h << 15;"),
    "rs_shard_start": ("            acc_t acc = x[s];\n            for (int k = 1; k < P; ++k) acc = combine(acc, x[(s + k) % P], dtype, op);",
                       "            acc_t acc = x[(s + 1) % P];\n            for (int k = 2; k <= P; ++k) acc = combine(acc, x[(s + k) % P], dtype, op);"),
    "rs_wrong_shard": ("            size_t e = (size_t)s * recvcount + i;", "            size_t e = (size_t)((s + 1) % P) * recvcount + i;"),
    "rs_scale_dropped": ("            if (dtype != OR_I32 && scale != 1.0f) acc.f = acc.f * scale;\n            store_narrowed(recv[s], i, acc, dtype);",
                         "            store_narrowed(recv[s], i, acc, dtype);"),
    "hier_group_start": ("        int g = (int)((c2 + (size_t)j) % (size_t)G);",
                         "        int g = (int)((c2 + (size_t)j + 1) % (size_t)G);"),
    "hier_local_start": ("        acc_t part = x[g * Q + (int)(c1 % (size_t)Q)];",
                         "        acc_t part = x[g * Q];"),
    "hier_subchunk_len": ("    size_t L2 = round_up((len1 + (size_t)G - 1) / (size_t)G, V);",
                          "    size_t L2 = round_up((count + (size_t)G - 1) / (size_t)G, V);"),
    "ag_wrong_offset": ("memcpy((char*)recv[r] + ((size_t)s * sendcount + i) * es,",
                        "memcpy((char*)recv[r] + ((size_t)((s + r) % P) * sendcount + i) * es,"),
    "scale_before_fold": ("    acc_t acc;\n    if (algo == OR_ALGO_TREE) {",
                          "    acc_t xs[OR_MAX_RANKS];\n"
                          "    for (int r = 0; r < P; ++r) {\n"
                          "        xs[r] = x[r];\n"
                          "        if (dtype != OR_I32 && scale != 1.0f) xs[r].f = xs[r].f * scale;\n"
                          "    }\n"
                          "    x = xs;\n    scale = 1.0f;\n"
                          "    acc_t acc;\n    if (algo == OR_ALGO_TREE) {"),
    "bf16_truncate": ("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;", "(void)lower;"),
    "int_sum_saturates": ("if (op == OR_SUM) acc.u = acc.u + x.u; /* wraps modulo 2^32 */",
                          "if (op == OR_SUM) {\n"
                          "            int64_t s = (int64_t)(int32_t)acc.u + (int64_t)(int32_t)x.u;\n"
                          "            acc.u = (uint32_t)(int32_t)(s > INT32_MAX ? INT32_MAX : s < INT32_MIN ? INT32_MIN : s);\n"
                          "        }"),
    "tree_root_below_p": ("    while (r * 2 <= P) r *= 2;", "    while (r * 2 < P) r *= 2;"),
    "hier_groups_reversed": ("        int g = (int)((c2 + (size_t)j) % (size_t)G);",
                             "        int g = (int)((c2 + (size_t)(G - j)) % (size_t)G);"),
    "hier_group_size_swapped": ("    int G = P / Q;", "    int G = Q;\n    Q = P / G;"),
    "hier_scale_per_group": ("        total = j == 0 ? part : combine(total, part, dtype, op);\n    }\n"
                             "    if (dtype != OR_I32 && scale != 1.0f) total.f = total.f * scale;\n",
                             "        if (dtype != OR_I32 && scale != 1.0f) part.f = part.f * scale;\n"
                             "        total = j == 0 ? part : combine(total, part, dtype, op);\n    }\n"),
    "float_min_on_bits": ("else if (op == OR_MIN) acc.f = (x.f < acc.f) ? x.f : acc.f;",
                          "else if (op == OR_MIN) acc.u = (x.u < acc.u) ? x.u : acc.u;"),
    "ll_folds_as_tree": ("    if (algo == OR_ALGO_TREE) {\n        int t = e",
                         "    if (algo != OR_ALGO_RING) {\n        int t = e"),
    "sampled_ignores_idx": ("acc_t y = reduce_element(x, P, count, idx[i], dtype, op, algo, scale);",
                            "acc_t y = reduce_element(x, P, count, i, dtype, op, algo, scale);"),
    "hier_sampled_ignores_idx": ("reduce_element_hier(x, P, Q, count, idx[i], dtype, op, scale)",
                                 "reduce_element_hier(x, P, Q, count, i, dtype, op, scale)"),
    "rs_scale_before_fold": ("            for (int r = 0; r < P; ++r) x[r] = load_widened(send[r], e, dtype);\n"
                             "            acc_t acc = x[s];",
                             "            for (int r = 0; r < P; ++r) {\n"
                             "                x[r] = load_widened(send[r], e, dtype);\n"
                             "                if (dtype != OR_I32 && scale != 1.0f) x[r].f = x[r].f * scale;\n"
                             "            }\n"
                             "            scale = 1.0f;\n"
                             "            acc_t acc = x[s];"),
    "ag_rank0_piece_only": ("(const char*)send[s] + i * es, es);", "(const char*)send[0] + i * es, es);"),
    "vector_of_4_elements": ("static size_t vec_elems(int dtype) { return 16 / elem_size(dtype); }",
                             "static size_t vec_elems(int dtype) { (void)dtype; return 4; }"),
    "hier_chunks_by_group_count": ("    size_t L1 = round_up((count + (size_t)Q - 1) / (size_t)Q, V);",
                                   "    size_t L1 = round_up((count + (size_t)G - 1) / (size_t)G, V);"),
    "hier_subchunk_from_zero": ("    size_t c2 = (e - c1 * L1) / L2;", "    size_t c2 = (e / L2) % (size_t)G;"),
    "tree_right_one_try": ("    for (int h = b / 2; h >= 1; h /= 2)\n        if (v + h <= P) return v + h;\n    return 0;",
                           "    return v + b / 2 <= P ? v + b / 2 : 0;"),
    "tree_right_two_tries": ("    for (int h = b / 2; h >= 1; h /= 2)\n        if (v + h <= P) return v + h;\n    return 0;",
                             "    for (int h = b / 2; h >= 1 && h >= b / 4; h /= 2)\n        if (v + h <= P) return v + h;\n    return 0;"),
    "rne_ties_down": ("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;",
                      "if (lower > 0x8000u) upper += 1;"),
    "tree_halves_swapped": ("int t = e < oracle_tree_split(count, dtype) ? 0 : 1;",
                            "int t = e < oracle_tree_split(count, dtype) ? 1 : 0;"),
    "tree1_maps_like_tree0": ("return t == 0 ? v - 1 : v % P;", "return v - 1;"),
    "float_min_ties_take_later": ("else if (op == OR_MIN) acc.f = (x.f < acc.f) ? x.f : acc.f;",
                                  "else if (op == OR_MIN) acc.f = (x.f <= acc.f) ? x.f : acc.f;"),
    "float_max_ties_take_later": ("else acc.f = (x.f > acc.f) ? x.f : acc.f;",
                                  "else acc.f = (x.f >= acc.f) ? x.f : acc.f;"),
    # 32-bit slips that only show at counts past 2^32 elements
    "chunk_index_32bit": ("int c = (int)(e / L);", "int c = (int)((uint32_t)e / L);"),
    "tree_split_32bit": ("size_t h = round_up((count + 1) / 2, vec_elems(dtype));",
                         "size_t h = round_up((size_t)(uint32_t)(count + 1) / 2, vec_elems(dtype));"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    mutant_c = tmp_path / f"{name}.c"
    mutant_c.write_text(src.replace(before, after))
    lib = oracle.compile_source(str(mutant_c), str(tmp_path / f"lib{name}.so"))
    O = oracle.Oracle(lib)
    failures = []
    for pin in pins.ALL_PINS:
        try:
            if pin in (pins.pin_ring_simulation, pins.pin_hierarchical_steps):
                pin(O, quick=True)
            else:
                pin(O)
        except (AssertionError, oracle.OracleError) as exc:
            failures.append(f"{pin.__name__}: {str(exc)[:80]}")
    assert failures, f"mutant {name} passed every pin"
    os.remove(lib)
