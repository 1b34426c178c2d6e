"""Plant plausible mistakes in copies of the oracle and check that the pins
catch every one of them (CPU only).

Each mutant is a single textual edit of sv_oracle.c (a flipped comparison, a
wrong sign, an off-by-one index, a transposed operand ...).  The copy is
compiled into a temporary directory; the real oracle is never touched.
"""
import os

import pytest

import oracle
import pins

MUTANTS = [
    ("accept test not strict", "accept = ui < thresh;", "accept = ui <= thresh;"),
    ("accept margin ignores ratios at or above 1", "margin = fabs(ui - ratio);",
     "margin = ratio < 1.0 ? fabs(ui - ratio) : INFINITY;"),
    ("accept margin measured against the clamped threshold", "margin = fabs(ui - ratio);",
     "margin = fabs(ui - thresh);"),
    ("ratio inverted", "ratio = qd / pd;", "ratio = pd / qd;"),
    ("zero draft probability rejects",
     "if (pd == 0.0) {\n            accept = 1;", "if (pd == 0.0) {\n            accept = 0;"),
    ("residual sign flipped", "double diff = qk - pk;", "double diff = pk - qk;"),
    ("residual not clamped", "r[k] = diff > 0.0 ? diff : 0.0;", "r[k] = diff;"),
    ("residual from the next position",
     "size_t toff = (trow0 + j) * (size_t)V, doff = (drow0 + j) * (size_t)V;",
     "size_t toff = (trow0 + j + 1) * (size_t)V, doff = (drow0 + j) * (size_t)V;"),
    ("bonus from the last draft position",
     "size_t toff = (trow0 + N) * (size_t)V;", "size_t toff = (trow0 + N - 1) * (size_t)V;"),
    ("temperature multiplies",
     "return exp((z - m) / T) / S;", "return exp((z - m) * T) / S;"),
    ("normaliser without the max shift", "S += exp((z - m) / T);", "S += exp(z / T);"),
    ("accept uniform off by one", "double ui = a->u[trow0 + i];", "double ui = a->u[trow0 + i + 1];"),
    ("sample uses the first uniform",
     "out[j] = orc_inverse_cdf(r, V, a->u[trow0 + N], &smargin);",
     "out[j] = orc_inverse_cdf(r, V, a->u[trow0 + 0], &smargin);"),
    ("inverse CDF not strict", "if (x < C) {", "if (x <= C) {"),
    ("greedy ties to the highest index", "if (z > best_z) {", "if (z >= best_z) {"),
    ("scan does not stop at the first rejection",
     "if (!accept) {\n            j = i;\n            break;\n        }",
     "if (!accept) {\n            j = i;\n        }"),
    ("num_accepted counts the correction token",
     "a->sample_margin[b] = smargin;\n    a->num_accepted[b] = j;",
     "a->sample_margin[b] = smargin;\n    a->num_accepted[b] = j + 1;"),
    ("draft probability read from the target row",
     "double ui = a->u[trow0 + i];",
     "double ui = a->u[trow0 + i]; pd = orc_prob(orc_logit(a->target, a->dtype, (trow0 + i) * (size_t)V + d), mq[i], Sq[i], T);"),
    ("greedy emits the draft at a mismatch",
     "j = i;\n                out[i] = ai;", "j = i;\n                out[i] = a->draft_tokens[drow0 + i];"),
    ("R == 0 reading dropped (samples the empty residual)",
     "if (R == 0.0) /* q_j == p_j: the rejection had probability 0 */",
     "if (0) /* q_j == p_j: the rejection had probability 0 */"),
    ("invalid rows not detected", "if (isnan(z) || z == INFINITY)\n            return 0;",
     "if (0)\n            return 0;"),
    ("bad draft tokens not detected", "if (d < 0 || d >= V)", "if (d < 0 || d > V)"),
    ("kv commits one row too many", "for (int k = 0; k < a; ++k) {", "for (int k = 0; k <= a && k < N; ++k) {"),
    ("kv destination ignores the cache length",
     "* max_len + len + k) * row_bytes;", "* max_len + k) * row_bytes;"),
    ("kv length not advanced", "cache_len[b] = len + a;", "cache_len[b] = len;"),
    ("kv overflow check off by one", "(long long)len + a > max_len", "(long long)len + a >= max_len"),
    ("kv plane and sequence transposed in the scratch",
     "src = (((size_t)p * B + b) * N + k) * row_bytes;", "src = (((size_t)b * P + p) * N + k) * row_bytes;"),
    ("kv bad count not reported", "if (a > N) {", "if (a > N + 1) {"),
    ("kv invalid verify commits", "if (a < 0)\n            continue;", "if (a < -1)\n            continue;"),
    ("tree: sibling residual skipped", "if (R > 0.0)\n                for (int k = 0; k < V; k++) {",
     "if (0)\n                for (int k = 0; k < V; k++) {"),
    ("tree: residual not normalised", "r[k] = (diff > 0.0 ? diff : 0.0) / R;", "r[k] = (diff > 0.0 ? diff : 0.0);"),
    ("tree: siblings tried in reverse order",
     "for (int c = n + 1; c <= M && next < 0; c++) {\n            if (par[c] != n)\n                continue;\n            const int x",
     "for (int c = M; c > n && next < 0; c--) {\n            if (par[c] != n)\n                continue;\n            const int x"),
    ("tree: final sample reuses the first child's uniform",
     "out[depth] = orc_inverse_cdf(r, V, a->u[row0], &smargin);",
     "out[depth] = orc_inverse_cdf(r, V, a->u[row0 + (M > 0)], &smargin);"),
    ("tree: a node may be its own parent", "if (par[n] < 0 || par[n] >= n)", "if (par[n] < 0 || par[n] > n)"),
    ("tree: leaves' draft rows validated", "if (!greedy && has_child && !(status & ORC_SEQ_BAD_TREE) &&",
     "if (!greedy && !(status & ORC_SEQ_BAD_TREE) &&"),
    ("tree: margin ignores ratios at or above 1", "margin = fabs(a->u[row0 + c] - ratio);",
     "margin = ratio < 1.0 ? fabs(a->u[row0 + c] - ratio) : INFINITY;"),
    ("tree: zero draft probability rejects", "if (p[x] == 0.0) {\n                accept = 1;",
     "if (p[x] == 0.0) {\n                accept = 0;"),
    ("tree: greedy takes the last matching child",
     "for (int c = n + 1; c <= M && next < 0; c++) {\n                if (par[c] != n)",
     "for (int c = n + 1; c <= M; c++) {\n                if (par[c] != n)"),
    ("tree: bonus from the parent's row at a leaf", "r[k] = orc_prob(orc_logit(a->target, a->dtype, (row0 + n) * (size_t)V + k), mq, Sq, T);",
     "r[k] = orc_prob(orc_logit(a->target, a->dtype, (row0 + (n ? par[n] : 0)) * (size_t)V + k), mq, Sq, T);"),
]


def _mutant_source(old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"anchor must occur exactly once: {old!r}"
    return src.replace(old, new)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src = tmp_path / "mutant.c"
    src.write_text(_mutant_source(old, new))
    lib = oracle.compile_library(str(src), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except Exception as e:  # an assertion, or a crash of the mutant's logic
            caught.append(f"{pin.__name__}: {type(e).__name__}")
    assert caught, f"no pin caught the mutant '{name}'"
    print(f"{name}: caught by {len(caught)} pins, e.g. {caught[0]}")


def test_anchors_are_unique():
    for _, old, _ in MUTANTS:
        _mutant_source(old, old)
    assert os.path.exists(oracle.SOURCE)
