"""Pins of the oracle's tolerance diagnostics: the accept-margin and race flip
indices, the race's relative gap, the top-p edge flag, and the sampler's race
flip index, each against a hand-worked value (tests/golden/tolerance_examples.txt),
plus planted mistakes in each that those pins catch.  These diagnostics choose
which logits-entry requests the GPU parity tests may exempt from exact token
comparison, so each one is checked on its own."""
import subprocess

import numpy as np
import pytest

import oracle
from conftest import hand_workload, load_golden

G = None


def _g():
    global G
    if G is None:
        G = load_golden("tolerance_examples.txt")
    return G


def _f(key):
    return [float(x) for x in _g()[key]]


def _accept_case(c):
    p = np.array(_f(f"{c}_p"), np.float32)
    q = np.array(_f(f"{c}_q"), np.float32)
    t = np.stack([p, np.array([1.0, 0.0], np.float32)])  # position 0, then the bonus row
    w = hand_workload(t, q[None, :], [0], u=[0.5], E=np.ones((1, 2)), temperature=[1.0])
    return oracle.verify(w)


def test_accept_margin_values():
    for c in ("a1", "a2", "a3"):
        o = _accept_case(c)
        assert o["status"] == 0
        got = o["diag"][0, oracle.DIAG_ACCEPT_MARGIN]
        assert got == pytest.approx(float(_g()[f"{c}_margin"][0]), rel=1e-9), c
    # a1 and a2 accept (u q = 0.25 < p); a1 sits inside the band, a2 and a3 outside
    assert _accept_case("a1")["num_accepted"][0] == 1


def _race_case(c):
    p = np.array(_f(f"{c}_p" if f"{c}_p" in _g() else "r_p"), np.float32)
    q = np.array(_f(f"{c}_q" if f"{c}_q" in _g() else "r_q"), np.float32)
    u = _f(f"{c}_u")[0] if f"{c}_u" in _g() else 0.5
    t = np.stack([p, np.full(3, 1.0 / 3.0, np.float32)])
    w = hand_workload(t, q[None, :], [2], u=[u], E=np.array([_f(f"{c}_E")], np.float32), temperature=[1.0])
    return oracle.verify(w)


def test_race_flip_and_relgap_values():
    for c in ("r1", "r2", "r3"):
        o = _race_case(c)
        assert o["status"] == 0 and o["num_accepted"][0] == 0
        assert o["out_tokens"][0, 0] == 0  # key 0.25 beats 0.25 - d
        d = o["diag"][0]
        assert d[oracle.DIAG_RACE_FLIP] == pytest.approx(float(_g()[f"{c}_flip"][0]), rel=1e-9), c
        assert d[oracle.DIAG_RACE_RELGAP] == pytest.approx(float(_g()[f"{c}_relgap"][0]), rel=1e-9), c
        assert d[oracle.DIAG_ACCEPT_MARGIN] > 1e3  # u q(y) far above p(y): no flip
        assert d[oracle.DIAG_FALLBACK] == 0 and d[oracle.DIAG_PATH] == 0


def test_top_p_edge_flags():
    for rk, tk, fk in (("edge_row", "edge_topp", "edge_flag"), ("tie_row", "tie_topp", "tie_flag")):
        row = np.array(_f(rk), np.float32)
        V = row.shape[0]
        for tp, flag in zip(_f(tk), _g()[fk]):
            tp32 = float(np.float32(tp))
            _, edge, rc = oracle.logits_to_probs(row, 1.0, 0, tp32)
            assert rc == 0 and edge == int(flag), (rk, tp)
            # the same flag through the verifier's diagnostics (logits entry)
            t = np.stack([row, np.zeros(V, np.float32)])
            w = hand_workload(t, row[None, :], [0], entry="logits", u=[0.25], E=np.ones((1, V)), temperature=[1.0],
                              top_p=[tp32])
            o = oracle.verify(w)
            assert o["diag"][0, oracle.DIAG_TOPP_EDGE] == int(flag), (rk, tp)


def test_sampler_race_flip_value():
    row = np.zeros((1, 2), np.float32)
    s = oracle.sample_rows(row, temperature=[1.0], exponentials=np.array([_f("s_E")], np.float32))
    assert s["status"] == 0 and s["tokens"][0] == 0
    assert s["diag"][0, 0] == pytest.approx(float(_g()["s_flip"][0]), rel=1e-9)
    assert s["diag"][0, 1] == 0


def test_planted_mistakes_are_caught(oracle_mod, tmp_path):
    src = oracle_mod._SRC.read_text()
    tests = (test_accept_margin_values, test_race_flip_and_relgap_values, test_top_p_edge_flags,
             test_sampler_race_flip_value)
    mutants = {
        "flip index takes the smaller bound": ("return a > r ? a : r;", "return a < r ? a : r;"),
        "absolute bound 1e-5": ("double a = needed_abs / 1e-6, r = needed_rel / 1e-5;",
                                "double a = needed_abs / 1e-5, r = needed_rel / 1e-5;"),
        "relative bound 1e-6": ("double a = needed_abs / 1e-6, r = needed_rel / 1e-5;",
                                "double a = needed_abs / 1e-6, r = needed_rel / 1e-6;"),
        "accept margin scaled by p alone": ("scale = uq + (double)py;", "scale = (double)py;"),
        "race flip drops the runner-up's draw": ("double f = flip_index(d / (1.0 / e1 + 1.0 / ex),",
                                                 "double f = flip_index(d / (1.0 / e1),"),
        "race flip drops q from the relative scale": (
            "double m1 = (double)pa[win] + (qa ? (double)qa[win] : 0.0);", "double m1 = (double)pa[win];"),
        "relgap not relative": ("double r = k1 > 0 ? d / k1 : 0.0;", "double r = k1 > 0 ? d : 0.0;"),
        "top-p edge band 1e-5": ("fabs(above - (double)top_p) < 1e-6 || fabs(through - (double)top_p) < 1e-6",
                                 "fabs(above - (double)top_p) < 1e-5 || fabs(through - (double)top_p) < 1e-5"),
        "top-p edge ignores the sum above the cut": (
            "fabs(above - (double)top_p) < 1e-6 || fabs(through - (double)top_p) < 1e-6",
            "fabs(through - (double)top_p) < 1e-6"),
        "top-p edge on single entries, not value groups": ("if (kept[r] > cut) above += e;",
                                                          "if (kept[r] > cut || (r == 0 && kept[1] >= cut)) above += e;"),
        "sampler flip drops the runner-up's draw": ("double f = flip_index(d / (1.0 / e1 + 1.0 / (double)E[x]),",
                                                    "double f = flip_index(d / (1.0 / e1),"),
    }
    for name, (old, new) in mutants.items():
        assert src.count(old) == 1, name
        msrc = tmp_path / f"t_{abs(hash(name))}.c"
        msrc.write_text(src.replace(old, new, 1))
        so = tmp_path / f"t_{abs(hash(name))}.so"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", str(so),
                        str(msrc), "-lm"], check=True)
        saved, orig_build = oracle_mod._LIB, oracle_mod.build
        try:
            oracle_mod._LIB = None
            oracle_mod.build = lambda force=False, _so=so: _so
            caught = False
            for t in tests:
                try:
                    t()
                except AssertionError:
                    caught = True
                    break
        finally:
            oracle_mod.build, oracle_mod._LIB = orig_build, saved
        assert caught, name
