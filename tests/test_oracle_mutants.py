"""Planted mistakes in the oracle: do its pins catch them?

Each mutant is a copy of the oracle package, in a temporary folder, with one
plausible mistake written into its source: a dropped term, a wrong sign or
comparison, a wrong index, an off-by-one, a wrong tie rule.  The pin suite
(test_oracle_pins.py) then runs in a child process against that copy and must
fail; a mutant it let through would mark a gap in the pins.  The unchanged
copy must pass (the control).  Nothing here touches the GPU or the product
library, and the oracle in the repository is never modified.

Left out on purpose: the promotion counter layout (token | level << 32 |
head << 40 | seq << 52) is a convention of this implementation, not a value
the pages fix, so only the GPU parity tests (which implement it independently)
hold it in place."""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

C, PY = "oracle.c", "__init__.py"

# (name, file, [(text, replacement), ...]); every text occurs exactly once in the file
MUTANTS = [
    # the hash and the promotion
    ("splitmix64_gamma_typo", C, [("0x9E3779B97F4A7C15ULL", "0x9E3779B97F4A7C17ULL")]),
    ("promotion_fallback_takes_largest_draw", C, [("if (u < bu) { bu = u; best = j; }",
                                                   "if (u > bu) { bu = u; best = j; }")]),
    ("promotion_draws_at_level_2", C, [("        uint32_t u = orc_promote_draw(seed, layer, seq, head, j, 1);\n        if",
                                        "        uint32_t u = orc_promote_draw(seed, layer, seq, head, j, 2);\n        if")]),
    # step a1, the lift
    ("lift_without_sqrt", C, [("e_out[j] = sqrt(r > 0.0 ? r : 0.0);", "e_out[j] = r > 0.0 ? r : 0.0;")]),
    ("lift_adds_the_norm", C, [("double r = M2 - n_out[j];", "double r = M2 + n_out[j];")]),
    ("lift_takes_the_smallest_norm", C, [("if (s > M2) M2 = s;", "if (j == 0 || s < M2) M2 = s;")]),
    ("lifted_coordinate_dropped_from_the_distance", C, [("    return s + t * t;\n}", "    return s;\n}")]),
    # step a3, the assignment
    ("assign_ties_to_the_highest_parent", C, [("if (best < 0 || D < bd) { bd = D; best = m; }",
                                               "if (best < 0 || D <= bd) { bd = D; best = m; }")]),
    ("promoted_token_not_its_own_parent", C, [("        token_parent[parent_tok[m]] = m;\n",
                                               "        (void)token_parent;\n")]),
    # step a4, the pages
    ("pack_reverses_the_token_order", C, [("members[start[m] + fill[m]++] = (int32_t)j;",
                                           "members[start[m] + count[m] - 1 - fill[m]++] = (int32_t)j;")]),
    ("pack_pages_one_token_short", C, [("for (int64_t r = 0; r < count[m]; r += S) {",
                                        "for (int64_t r = 0; r < count[m]; r += S - 1) {"),
                                       ("(count[m] - r) < S ? (count[m] - r) : S)",
                                        "(count[m] - r) < S - 1 ? (count[m] - r) : S - 1)")]),
    ("pack_every_page_full_length", C, [("page_len[P] = len;", "page_len[P] = S;")]),
    # step a5, the pool
    ("pool_pad_slots_not_zero", C, [("dk[i] = j >= 0 ? K[(int64_t)j * d + i] : 0.0;",
                                     "dk[i] = K[(int64_t)(j >= 0 ? j : 0) * d + i];")]),
    # steps a6-a8, the selection
    ("select_ascending_scores", C, [("if (x->s > y->s) return -1;\n    if (x->s < y->s) return 1;",
                                     "if (x->s < y->s) return -1;\n    if (x->s > y->s) return 1;")]),
    ("select_ties_to_the_highest_page", C, [("return (x->id > y->id) - (x->id < y->id);",
                                             "return (x->id < y->id) - (x->id > y->id);")]),
    ("select_every_head_scores_with_head_0", C, [("s += q[(int64_t)h * d + i] * parent_keys[(int64_t)m * d + i];",
                                                  "s += q[i] * parent_keys[(int64_t)m * d + i];")]),
    ("union_of_the_first_head_only", C, [("if (r < k) in_union[order[r].id] = 1;",
                                          "if (r < k && h == 0) in_union[order[r].id] = 1;")]),
    # step a9, the gather
    ("gather_full_length_pages", C, [("buf_len[u] = page_len[p];", "buf_len[u] = S;")]),
    # step a10, the attention
    ("attention_without_scale", C, [("logit[t] = dot * scale;", "logit[t] = dot;")]),
    ("attention_over_padded_slots", C, [("if (s >= buf_len[u]) { logit[t] = -INFINITY; continue; }",
                                         "if (s >= S) { logit[t] = -INFINITY; continue; }")]),
    ("attention_not_normalised", C, [("double w = exp(logit[t] - mx) / den;", "double w = exp(logit[t] - mx);")]),
    # step a11, the insert
    ("insert_splits_at_16", C, [("if (page >= 0 && page_len[page] >= S) page = -1;",
                                 "if (page >= 0 && page_len[page] >= S - 1) page = -1;")]),
    ("insert_without_the_lifted_coordinate", C, [("    double e = sqrt(r > 0.0 ? r : 0.0);\n    int32_t Np",
                                                  "    double e = 0.0 * r;\n    int32_t Np")]),
    # sink / window pages
    ("window_not_cut_at_the_sink", PY, [("return se, max(se, N - max(n_window, 0))",
                                         "return se, N - max(n_window, 0)")]),
    ("sink_pages_run_past_the_sink", PY, [("[(a, min(a + S, se)) for a in range(0, se, S)]",
                                           "[(a, a + S) for a in range(0, se, S)]")]),
    ("window_pages_before_sink_pages", PY, [
        ("ranges = [(a, min(a + S, se)) for a in range(0, se, S)] + [(a, min(a + S, N)) for a in range(ws, N, S)]",
         "ranges = [(a, min(a + S, N)) for a in range(ws, N, S)] + [(a, min(a + S, se)) for a in range(0, se, S)]")]),
    ("positional_pages_owned_by_parent_0", PY, [("np.full(len(ranges), -1, np.int32)", "np.full(len(ranges), 0, np.int32)")]),
    ("middle_promotion_ids_not_absolute", PY, [("return (out + lo).astype(np.int32)", "return out.astype(np.int32)")]),
    ("positional_pages_not_attended", PY, [("    if n_pos:\n        sel = np.concatenate",
                                            "    if n_pos < 0:\n        sel = np.concatenate")]),
    ("budget_counts_the_positional_pages", PY, [("    k_pages = -(-budget_tokens // S)\n",
                                                 "    k_pages = max(0, -(-budget_tokens // S) - int(idx.get(\"n_pos\", 0)))\n")]),
    # inter-layer reuse
    ("reuse_keeps_the_previous_layers_keys", PY, [
        ("parent_keys=K[parent_tok] if N else K[:0],\n                parent_e=e[parent_tok] if N else e[:0], "
         "token_parent=token_parent,\n                pool_k=pool_k, pool_v=pool_v, S=S, **pk, **extra)",
         "parent_keys=_f64(prev[\"parent_keys\"]) if N else K[:0],\n                parent_e=e[parent_tok] if N "
         "else e[:0], token_parent=token_parent,\n                pool_k=pool_k, pool_v=pool_v, S=S, **pk, **extra)")]),
    # third level and descent
    ("level2_draws_at_level_1", PY, [("promote_draw(seed, layer, seq, head, int(t), 2)",
                                      "promote_draw(seed, layer, seq, head, int(t), 1)")]),
    ("level2_fallback_takes_largest_draw", PY, [("node2 = np.array([int(np.argmin(d2))])",
                                                 "node2 = np.array([int(np.argmax(d2))])")]),
    ("descent_keeps_the_lowest_level2_scores", PY, [("key=lambda i: (-s2[i], i))[:k_pages]",
                                                     "key=lambda i: (s2[i], i))[:k_pages]")]),
    ("descent_pages_not_limited_to_k", PY, [("                if len(pages) < k_pages:", "                if True:")]),
    ("descent_children_by_ascending_score", PY, [("sorted(cand, key=lambda m: (-s1[m], m))",
                                                  "sorted(cand, key=lambda m: (s1[m], m))")]),
]


def _run_pins_against(tmp_path, fname=None, subs=()):
    dst = tmp_path / "oracle"
    shutil.copytree(os.path.join(ROOT, "oracle"), dst,
                    ignore=shutil.ignore_patterns("*.so", "*.tmp*", "__pycache__"))
    if fname:
        path = dst / fname
        src = path.read_text()
        for old, new in subs:
            assert src.count(old) == 1, old
            src = src.replace(old, new)
        path.write_text(src)
    # the copy first on the path: `import oracle` in the pins resolves to it
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([str(tmp_path), ROOT]))
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=str(tmp_path), env=env, capture_output=True, text=True, timeout=900)
    return r.returncode, r.stdout[-3000:] + r.stderr[-1000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """(return code, output tail) of the pin suite against the unchanged copy
    and against every mutant, the child processes run side by side."""
    jobs = {"control": (None, ())}
    jobs.update({name: (fname, subs) for name, fname, subs in MUTANTS})
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        futs = {name: ex.submit(_run_pins_against, tmp_path_factory.mktemp(name), fname, subs)
                for name, (fname, subs) in jobs.items()}
        return {name: f.result() for name, f in futs.items()}


def test_unchanged_copy_passes_the_pins(outcomes):
    rc, out = outcomes["control"]
    assert rc == 0, out


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, outcomes):
    rc, out = outcomes[name]
    assert rc == 1, f"{name}: the pins let this mistake through (rc {rc})\n{out}"
