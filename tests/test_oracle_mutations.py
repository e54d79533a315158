"""Planted mistakes in the oracles, on the CPU: each must fail a pin.

The pins of ``test_oracle_pins.py`` (linear pass) and
``test_softmax_oracle_pins.py`` (softmax layer) are run against mutated
copies of the oracles: the C recurrence rebuilt from an edited copy of its
source, the numpy softmax oracle loaded from an edited copy of its module.
Each mutant is a plausible slip (a dropped term, a wrong sign, index or
transpose, an exclusive diagonal, a branch that loses or widens its prefix,
one head's values for every head) and must fail at least one pin; an
unedited copy built the same way must pass all of them.  The mutants live in
temporary files only.
"""
import importlib.util
import os
import subprocess

import numpy as np
import pytest

import oracle.oracle as la_oracle
import test_oracle_pins as la_pins
import test_softmax_oracle_pins as sm_pins

ORACLE_DIR = os.path.dirname(la_oracle.__file__)

# (name, text in the C source, replacement)
C_MUTANTS = [
    ("exclusive diagonal (o_t from S_{t-1})",
     "ot[j] += Si[j] * qi;", "ot[j] += (Si[j] - kt[i] * vt[j]) * qi;"),
    ("S q in place of S^T q",
     "ot[j] += Si[j] * qi;", "ot[j] += S[j * D + i] * qi;"),
    ("state not accumulated (S_{t-1} dropped)",
     "Si[j] += ki * vt[j];", "Si[j] = ki * vt[j];"),
    ("wrong sign of the state update",
     "Si[j] += ki * vt[j];", "Si[j] -= ki * vt[j];"),
    ("branch from a zero state",
     "memcpy(S, S0, sizeof(double) * D * D);", "memset(S, 0, sizeof(double) * D * D);"),
    ("branch from another view's state",
     "init_states + ((int64_t)parent[b] * H + h)",
     "init_states + ((int64_t)(num_states - 1 - parent[b]) * H + h)"),
    ("head 0's values for every head",
     "const double *vt = v + (t * H + h) * D;", "const double *vt = v + (t * H) * D;"),
    ("last row of a view dropped",
     "run_rows(q, k, v, H, D, h, view_cu[vi], view_cu[vi + 1], S, out);",
     "run_rows(q, k, v, H, D, h, view_cu[vi], view_cu[vi + 1] - (view_cu[vi + 1] > view_cu[vi]), S, out);"),
]

# (name, text in softmax_oracle.py, replacement)
SOFTMAX_MUTANTS = [
    ("exclusive diagonal",
     "causal = np.tril(np.ones((n, n), dtype=bool))",
     "causal = np.tril(np.ones((n, n), dtype=bool), -1)"),
    ("branch without its parent view",
     "_segment(q[a:b], k[a:b], v[a:b], k[pa:pb], v[pa:pb], scale)",
     "_segment(q[a:b], k[a:b], v[a:b], empty, empty, scale)"),
    ("branch prefix runs up to the branch (siblings visible)",
     "_segment(q[a:b], k[a:b], v[a:b], k[pa:pb], v[pa:pb], scale)",
     "_segment(q[a:b], k[a:b], v[a:b], k[pa:a], v[pa:a], scale)"),
    ("scale 1/d in place of 1/sqrt(d)",
     "scale = 1.0 / math.sqrt(D)", "scale = 1.0 / D"),
    ("lse without the row maximum",
     "(m + np.log(l))[..., 0]", "(np.log(l))[..., 0]"),
    ("head 0's values for every head",
     "vv = np.concatenate([vp[:, h], vs[:, h]], axis=0)",
     "vv = np.concatenate([vp[:, 0], vs[:, 0]], axis=0)"),
]


def _la_pins():
    p = la_pins
    return [
        ("hand-worked example", p.test_hand_worked_example),
        ("recurrent = quadratic = chunked",
         lambda: [p.test_recurrent_equals_quadratic_and_chunked(L) for L in (1, 65, 129)]),
        ("tiny workload = quadratic form", p.test_tiny_workload_matches_quadratic_form),
        ("final state = K^T V", p.test_final_state_is_kt_v),
        ("d = 1 cumulative sum", p.test_d1_is_a_cumulative_sum),
        ("one-hot exact counts", p.test_one_hot_inputs_give_exact_counts),
        ("branch = tail of view ++ branch", p.test_branch_equals_tail_of_view_plus_branch),
        ("siblings do not matter", p.test_siblings_do_not_change_a_branch),
        ("packed = per-view runs", p.test_packed_pass_equals_per_view_runs),
        ("branches from cached state", p.test_branches_from_cached_state_equal_in_pass_branches),
        ("linearity", p.test_linear_in_v_and_in_q),
        ("heads independent", p.test_heads_are_independent_and_threads_do_not_matter),
        ("random passes = quadratic forms",
         lambda: [p.test_random_packed_passes_equal_quadratic_forms(s) for s in range(2)]),
    ]


def _softmax_pins():
    p = sm_pins
    return [
        ("views = library causal attention",
         lambda: [p.test_view_equals_library_causal_attention(L) for L in (1, 65, 129)]),
        ("branches = library attention with a mask",
         lambda: [p.test_branches_equal_library_attention_with_visibility_mask(s) for s in (None, 0.3)]),
        ("zero queries: running means", p.test_zero_queries_give_running_means),
        ("first view row", p.test_first_view_row_returns_its_value_and_score),
        ("huge scale: hard attention", p.test_huge_scale_is_hard_attention),
        ("branch = tail of view ++ branch", p.test_branch_equals_tail_of_view_plus_branch),
        ("siblings and packing", p.test_siblings_do_not_change_a_branch_and_packing_equals_separate_runs),
        ("common score shift", p.test_a_common_score_shift_leaves_output_and_shifts_lse),
        ("sampled rows = whole pass", p.test_sampled_rows_equal_whole_pass),
        ("random passes = library attention",
         lambda: [p.test_random_packed_passes_equal_library_attention(s) for s in range(2)]),
    ]


def _failing(pins):
    failed = []
    for name, run in pins:
        try:
            run()
        except Exception:   # an assertion, or a rejected or non-finite result
            failed.append(name)
    return failed


def _edit(text, old, new):
    assert text.count(old) >= 1, "mutation site not found: %r" % old
    return text.replace(old, new, 1)


def _build_c(tmp_path, tag, source):
    src = tmp_path / ("oracle_%s.c" % tag)
    lib = tmp_path / ("liboracle_%s.so" % tag)
    src.write_text(source)
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-o", str(lib), str(src)],
                   check=True)
    return la_oracle.bind_library(str(lib))


def _c_source():
    with open(os.path.join(ORACLE_DIR, "spanla_oracle.c")) as f:
        return f.read()


def test_unedited_c_oracle_copy_passes_every_pin(tmp_path, monkeypatch):
    monkeypatch.setattr(la_oracle, "_lib", _build_c(tmp_path, "control", _c_source()))
    assert _failing(_la_pins()) == []


@pytest.mark.parametrize("mutant", C_MUTANTS, ids=[m[0] for m in C_MUTANTS])
def test_c_oracle_mutant_fails_a_pin(tmp_path, monkeypatch, mutant):
    name, old, new = mutant
    lib = _build_c(tmp_path, "m", _edit(_c_source(), old, new))
    monkeypatch.setattr(la_oracle, "_lib", lib)
    failed = _failing(_la_pins())
    print("%s: caught by %s" % (name, failed))
    assert failed, "no pin caught the planted mistake: %s" % name


def _load_softmax(tmp_path, tag, source):
    path = tmp_path / ("softmax_oracle_%s.py" % tag)
    path.write_text(source)
    spec = importlib.util.spec_from_file_location("softmax_oracle_%s" % tag, str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _softmax_source():
    with open(os.path.join(ORACLE_DIR, "softmax_oracle.py")) as f:
        return f.read()


def _use_softmax(monkeypatch, mod):
    monkeypatch.setattr(sm_pins, "oracle_softmax_pass", mod.oracle_softmax_pass)
    monkeypatch.setattr(sm_pins, "oracle_softmax_rows", mod.oracle_softmax_rows)


def test_unedited_softmax_oracle_copy_passes_every_pin(tmp_path, monkeypatch):
    _use_softmax(monkeypatch, _load_softmax(tmp_path, "control", _softmax_source()))
    assert _failing(_softmax_pins()) == []


@pytest.mark.parametrize("mutant", SOFTMAX_MUTANTS, ids=[m[0] for m in SOFTMAX_MUTANTS])
def test_softmax_oracle_mutant_fails_a_pin(tmp_path, monkeypatch, mutant):
    name, old, new = mutant
    with np.errstate(all="ignore"):
        _use_softmax(monkeypatch, _load_softmax(tmp_path, "m", _edit(_softmax_source(), old, new)))
        failed = _failing(_softmax_pins())
    print("%s: caught by %s" % (name, failed))
    assert failed, "no pin caught the planted mistake: %s" % name
