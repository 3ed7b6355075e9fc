"""The oracle against its pins (no GPU).

Besides running every pin on the oracle, this plants one mistake at a time in
a copy of ``oracle/oracle.c`` (a dropped term, a wrong sign, a shifted index,
a reversed tie order ...) and requires that some pin fails on each copy.
"""

import os

import numpy as np
import pytest

import oracle
import oracle_pins

pytestmark = pytest.mark.filterwarnings("ignore")


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.default())


# (name, text in oracle.c, replacement): each is a plausible slip
MUTANTS = [
    ("core_excludes_self", "dist[i * min_samples + (min_samples - 1)]",
     "dist[i * min_samples + (min_samples > 1 ? min_samples - 2 : 0)]"),
    ("tie_lo_reversed", "if (a->lo != b->lo) return a->lo < b->lo;",
     "if (a->lo != b->lo) return a->lo > b->lo;"),
    ("tie_hi_reversed", "return a->hi < b->hi;", "return a->hi > b->hi;"),
    ("weight_drops_core_b", "if (core[b] > w) w = core[b];", ""),
    ("weight_drops_core_a", "if (core[a] > w) w = core[a];", ""),
    ("distance_drops_last_feature",
     "    double s = 0.0;\n    for (int f = 0; f < d; ++f) {\n        double t = (double)a[f]",
     "    double s = 0.0;\n    for (int f = 0; f < d - 1; ++f) {\n        double t = (double)a[f]"),
    ("distance_sign", "double t = (double)a[f] - (double)b[f];",
     "double t = (double)a[f] + (double)b[f];"),
    ("knn_tie_reversed", "(da == db && ja < jb)", "(da == db && ja > jb)"),
    ("knn_skips_first_column", "for (int64_t j = 0; j < m; ++j) {", "for (int64_t j = 1; j < m; ++j) {"),
    ("prim_relax_inverted", "if (key_less(&kv, &best[u])) best[u] = kv;",
     "if (key_less(&best[u], &kv)) best[u] = kv;"),
    ("prim_picks_max", "if (bi < 0 || key_less(&best[rem[r]], &best[rem[bi]])) bi = r;",
     "if (bi < 0 || key_less(&best[rem[bi]], &best[rem[r]])) bi = r;"),
    ("no_sqrt", "    return sqrt(s);\n}", "    return s;\n}"),
    ("transposed_operand", "P[i * d + f] = X[(int64_t)f * ld + i];",
     "P[i * d + f] = X[(int64_t)i * d + f];"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = oracle.compile_c(str(path), str(tmp_path / f"lib{name}.so"))
    mutant = oracle.Oracle(so)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"


def test_oracle_rejects_bad_arguments():
    X = np.zeros((2, 3), dtype=np.float32)
    with pytest.raises(ValueError):
        oracle.knn(X, X, 4)
    with pytest.raises(ValueError):
        oracle.core_distances(X, 4)


# ---------------------------------------------------------------------------
# the back half (oracle/hierarchy.py)

def _hierarchy_from_source(src: str):
    import types
    mod = types.ModuleType("hierarchy_mutant")
    exec(compile(src, "hierarchy_mutant.py", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("pin", oracle_pins.HIERARCHY_PINS, ids=lambda f: f.__name__)
def test_hierarchy_pin(pin):
    from oracle import hierarchy
    pin(oracle.default(), hierarchy)


HIERARCHY_MUTANTS = [
    ("birth_at_zero", "            birth[child] = lam", "            birth[child] = 0.0"),
    ("size_rule_strict", "if sa >= min_cluster_size and sb >= min_cluster_size:",
     "if sa > min_cluster_size and sb > min_cluster_size:"),
    ("root_selectable", "        if node == n:\n            continue\n", ""),
    ("eom_inverted", "if below > stab[node]:", "if below < stab[node]:"),
    ("lambda_is_distance", "return 1.0 / d if d > 0.0 else math.inf", "return d"),
    ("small_side_continues", "            relabel[b] = me\n            queue.append(b)",
     "            relabel[a] = me\n            queue.append(a)"),
    ("root_points_not_noise", "while c is not None and c not in chosen:",
     "while c is not None and c not in chosen and c != n:"),
]


@pytest.mark.parametrize("name,old,new", HIERARCHY_MUTANTS, ids=[m[0] for m in HIERARCHY_MUTANTS])
def test_hierarchy_pins_catch_planted_mistake(name, old, new):
    from oracle import hierarchy
    src = open(hierarchy.__file__).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutant = _hierarchy_from_source(src.replace(old, new))
    failed = []
    for pin in oracle_pins.HIERARCHY_PINS:
        try:
            pin(oracle.default(), mutant)
        except Exception:  # an assertion, or the mutant breaking outright
            failed.append(pin.__name__)
    assert failed, f"no pin catches {name}"
