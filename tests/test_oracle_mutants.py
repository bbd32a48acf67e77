"""Plausible mistakes planted in copies of the CPU oracle are caught by the pins.

Each mutant is one textual edit of oracle/wf_oracle.c, compiled to a scratch
directory on the CPU; the test asserts that at least one of the named pin
checks fails against it (and, as a control, that all of them pass on the
unmodified oracle)."""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "wf_oracle.c")

MUTANTS = [
    ("argmax keeps the last of equal maxima", "if (L > best) {", "if (L >= best) {",
     [pins.check_argmax_ties]),
    ("weight row stride dropped (operand misindexed)", "logit(h + p * d, W + v * d, d)", "logit(h + p * d, W + v, d)",
     [pins.check_argmax_bruteforce]),
    ("second-best not updated when the best moves", "second = best;\n                best = L;",
     "best = L;", [pins.check_argmax_bruteforce]),
    ("tree ignores the parent's acceptance", "int parent_acc = (p < 0) ? 1 : acc[p];", "int parent_acc = 1;",
     [pins.check_tree_golden, pins.check_tree_bruteforce]),
    ("tree compares against the node's own row", "int prow = (p < 0) ? root : root + 1 + p;",
     "int prow = root + 1 + i;", [pins.check_tree_golden, pins.check_tree_bruteforce]),
    ("tree keeps the highest index on equal depth", "depth[i] > best_depth", "depth[i] >= best_depth",
     [pins.check_tree_golden, pins.check_tree_bruteforce]),
    ("chain bonus taken one row early", "bonus[b] = g[root + n];", "bonus[b] = g[root + (n > 0 ? n - 1 : 0)];",
     [pins.check_chain_golden]),
    ("chain compares draft j with row j+1", "dr[n] == g[root + n]", "dr[n] == g[root + n + 1]",
     [pins.check_chain_golden, pins.check_chain_is_linear_tree]),
    ("router drops the first-layer bias", "double z = b1[j];", "double z = 0.0;",
     [pins.check_router_closed_forms]),
    ("router drops the second-layer bias", "double out = b2;", "double out = 0.0;",
     [pins.check_router_closed_forms, pins.check_route_strict]),
    ("tanh approximation of GELU", "return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));",
     "return 0.5 * x * (1.0 + tanh(0.7978845608028654 * (x + 0.044715 * x * x * x)));",
     [pins.check_gelu_values]),
    ("route on >= instead of >", "route[b] = out > tau ? 1 : 0;", "route[b] = out >= tau ? 1 : 0;",
     [pins.check_route_strict]),
    ("top-k ties keep the higher id", "return (x->id > y->id) - (x->id < y->id);",
     "return (x->id < y->id) - (x->id > y->id);", [pins.check_topk_ties]),
    ("log-sum-exp without the max shift", "lse[b] = mx + log(acc);", "lse[b] = log(acc);",
     [pins.check_topk_bruteforce]),
    ("entropy without the max shift", "for (int64_t v = 0; v < V; ++v) S += exp(L[v] - M);",
     "M = 0.0;\n        for (int64_t v = 0; v < V; ++v) S += exp(L[v] - M);", [pins.check_entropy]),
    ("entropy in bits", "if (p > 0.0) ent -= p * log(p);", "if (p > 0.0) ent -= p * log2(p);",
     [pins.check_entropy]),
    ("entropy route on >=", "route[b] = ent > tau ? 1 : 0;", "route[b] = ent >= tau ? 1 : 0;",
     [pins.check_entropy_route_strict]),
    ("kept rows use the node index as the row", "out[j] = pos_off[b] + 1 + path[(int64_t)b * path_stride + j - 1];",
     "out[j] = pos_off[b] + path[(int64_t)b * path_stride + j - 1];", [pins.check_accepted_rows]),
    ("kept-row offsets forget the root", "acc_off[b + 1] = acc_off[b] + n + 1;", "acc_off[b + 1] = acc_off[b] + n;",
     [pins.check_accepted_rows]),
    ("tree frontier ranked by log-probability alone", "ps[made] = (par < 0 ? 0.0f : ps[par]) + l;",
     "ps[made] = l;", [pins.check_build_tree]),
    ("tree listed in score order, not depth by depth", "if (pd[r[i].idx] == dd) new_of[r[i].idx] = out++;",
     "if (dd == 1) new_of[r[i].idx] = out++;", [pins.check_build_tree]),
    ("tree ties keep the later node", "return (x->idx > y->idx) - (x->idx < y->idx);\n}\n\nint oracle_build_tree",
     "return (x->idx < y->idx) - (x->idx > y->idx);\n}\n\nint oracle_build_tree", [pins.check_build_tree]),
    ("top-k maps through the wrong id", "tids[(int64_t)b * k + j] = d2t[s[j].id];",
     "tids[(int64_t)b * k + j] = s[j].id;", [pins.check_topk_bruteforce]),
    ("RMSNorm with eps outside the root", "const double r = 1.0 / sqrt(ss / (double)din + eps);",
     "const double r = 1.0 / (sqrt(ss / (double)din) + eps);", [pins.check_rmsnorm]),
    ("RMSNorm over the sum, not the mean", "const double r = 1.0 / sqrt(ss / (double)din + eps);",
     "const double r = 1.0 / sqrt(ss + eps);", [pins.check_rmsnorm]),
    ("rotation turns the wrong way", "y[i] = x1 * c - x2 * s;\n        y[i + half] = x2 * c + x1 * s;",
     "y[i] = x1 * c + x2 * s;\n        y[i + half] = x2 * c - x1 * s;", [pins.check_rope]),
    ("rotation frequencies theta^(-i/D)", "pow(theta, -2.0 * (double)i / (double)D)",
     "pow(theta, -(double)i / (double)D)", [pins.check_rope]),
    ("rotation pairs neighbours (2i, 2i+1)", "const double x1 = x[i], x2 = x[i + half];\n        y[i] = x1 * c - x2 * s;\n        y[i + half] = x2 * c + x1 * s;",
     "const double x1 = x[2 * i], x2 = x[2 * i + 1];\n        y[2 * i] = x1 * c - x2 * s;\n        y[2 * i + 1] = x2 * c + x1 * s;",
     [pins.check_rope]),
    ("query head h reads KV head h mod G", "const int g = h / (H / G);", "const int g = h % G;",
     [pins.check_catchup_head_groups, pins.check_catchup_single_entry]),
    ("scores not scaled by 1/sqrt(D)", "sc[t] = s / sqrt((double)D);", "sc[t] = s;",
     [pins.check_catchup_two_entries]),
    ("backlog positions ignore the cached length", "const int64_t pos = cache_len[b] + (r - bl_off[b]);",
     "const int64_t pos = r - bl_off[b];", [pins.check_catchup_lazy_equals_eager]),
    ("final query rotated one position late", "const double pos = (double)(T - 1);", "const double pos = (double)T;",
     [pins.check_catchup_final_query]),
    ("final token taken from the start of the backlog", "const int64_t f = bl_off[b + 1] - 1;",
     "const int64_t f = bl_off[b];", [pins.check_catchup_final_query, pins.check_catchup_lazy_equals_eager]),
    ("final token does not attend to itself",
     "const int64_t T = cache_len[b] + (bl_off[b + 1] - bl_off[b]);",
     "const int64_t T = cache_len[b] + (bl_off[b + 1] - bl_off[b]) - 1;",
     [pins.check_catchup_two_entries, pins.check_catchup_single_entry]),
    ("residual dropped", "out[(int64_t)b * din + i] = bf16_value(u[f * din + i]) + row_dot(Wo + i * HD, ob, HD);",
     "out[(int64_t)b * din + i] = row_dot(Wo + i * HD, ob, HD);", [pins.check_catchup_single_entry]),
    ("output projection reads Wo transposed", "row_dot(Wo + i * HD, ob, HD)", "row_dot(Wo + i, ob, HD)",
     [pins.check_catchup_output_projection]),
    ("value projection applied without the norm",
     "vrow[(int64_t)g * D + e] = bf16_round(row_dot(Wv + ((int64_t)g * D + e) * din, a, din));",
     "vrow[(int64_t)g * D + e] = bf16_round(row_dot(Wv + ((int64_t)g * D + e) * din, a, din) / bf16_value(gamma[0]));",
     [pins.check_catchup_final_query]),
]


@pytest.mark.parametrize("desc,old,new,checks", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, desc, old, new, checks):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    mo = oracle.Oracle(oracle.compile_c(str(mpath), str(tmp_path / "libmutant.so")))
    caught = []
    for chk in checks:
        try:
            chk(mo)
        except AssertionError:
            caught.append(chk.__name__)
    assert caught, f"no pin caught: {desc}"
