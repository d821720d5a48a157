"""Distributional pins of the CPU oracle.

Page 2, section 04: accepting y with min(1, p(y)/q(y)) and replacing a
rejection with the renormalised residual max(0, p - q) makes every committed
token follow the target p ("the accepted branch contributes min(p, q), the
rejected branch adds (p - q)+, together exactly p").  For fixed per-position
rows p_j, q_j and drafts y_j ~ q_j this gives the closed form

    P(commit x_0..x_{a-1}, t; A = a) = prod_{j<a} min(p_j(x_j), q_j(x_j))
                                       * ((p_a - q_a)+(t)   if a < gamma
                                          p_gamma(t)        if a = gamma)

and P(A >= k) = prod_{j<k} beta_j with beta_j = sum_x min(p_j, q_j) (the
"a^k" tail of section 10 made exact).  The closed form is first checked
against a brute-force enumeration in exact rationals of the per-position
algorithm of section 06; the oracle's sampled outcomes are then compared with
it by chi-square (page 2, section 13 asks for exactly this kind of test).
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest
import scipy.stats

from conftest import hand_workload

V, GAMMA = 3, 2
# rows with dyadic entries (exact in fp32 and as fractions); one row per position
P_ROWS = [[6, 7, 3], [2, 10, 4], [9, 1, 6]]  # /16
Q_ROWS = [[10, 4, 2], [5, 5, 6]]             # /16
P16 = [[Fraction(v, 16) for v in r] for r in P_ROWS]
Q16 = [[Fraction(v, 16) for v in r] for r in Q_ROWS]


def closed_form():
    out = {}
    for a in range(GAMMA + 1):
        for xs in itertools.product(range(V), repeat=a + 1):
            pr = Fraction(1)
            for j in range(a):
                pr *= min(P16[j][xs[j]], Q16[j][xs[j]])
            t = xs[a]
            pr *= (max(P16[a][t] - Q16[a][t], 0) if a < GAMMA else P16[GAMMA][t])
            out[xs] = pr
    return out


def brute_force():
    """Enumerate drafts y ~ q and the section-06 algorithm's branch probabilities."""
    out = {}

    def rec(j, prefix, pr):
        if j == GAMMA:
            for t in range(V):
                key = tuple(prefix) + (t,)
                out[key] = out.get(key, 0) + pr * P16[GAMMA][t]
            return
        res = [max(P16[j][x] - Q16[j][x], 0) for x in range(V)]
        zres = sum(res)
        for y in range(V):
            if Q16[j][y] == 0:
                continue
            alpha = min(Fraction(1), P16[j][y] / Q16[j][y])
            rec(j + 1, prefix + [y], pr * Q16[j][y] * alpha)
            if alpha < 1:
                for t in range(V):
                    if res[t]:
                        key = tuple(prefix) + (t,)
                        out[key] = out.get(key, 0) + pr * Q16[j][y] * (1 - alpha) * res[t] / zres

    rec(0, [], Fraction(1))
    return out


def test_closed_form_equals_brute_force():
    cf, bf = closed_form(), brute_force()
    assert sum(cf.values()) == 1
    for k in set(cf) | set(bf):
        assert cf.get(k, 0) == bf.get(k, 0), k


def _sample_workload(n, rng):
    p = np.array(P_ROWS, np.float32) / 16
    q = np.array(Q_ROWS, np.float32) / 16
    ids = np.stack([rng.choice(V, size=n, p=q[j].astype(np.float64)) for j in range(GAMMA)], axis=1).reshape(-1)
    target = np.tile(p, (n, 1))
    draft = np.tile(q, (n, 1))
    return hand_workload(target, draft, ids, u=rng.random(n * GAMMA, dtype=np.float32),
                         E=rng.standard_exponential((n, V), dtype=np.float32))


def _chi2_outcomes(out_tokens, nacc, n):
    cf = closed_form()
    keys = sorted(cf, key=lambda k: (len(k), k))
    index = {k: i for i, k in enumerate(keys)}
    codes = np.zeros(n, dtype=np.int64)
    # encode each committed sequence
    lens = nacc + 1
    for L in range(1, GAMMA + 2):
        sel = lens == L
        sub = out_tokens[sel, :L]
        for row_idx, row in zip(np.nonzero(sel)[0], sub):
            codes[row_idx] = index[tuple(int(v) for v in row)]
    obs = np.bincount(codes, minlength=len(keys)).astype(np.float64)
    exp = np.array([float(cf[k]) for k in keys]) * n
    keep = exp > 0
    assert obs[~keep].sum() == 0  # impossible outcomes never happen
    obs, exp = obs[keep], exp[keep]
    small = exp < 5  # merge bins with expectation < 5
    if small.any():
        obs = np.append(obs[~small], obs[small].sum())
        exp = np.append(exp[~small], exp[small].sum())
    return scipy.stats.chisquare(obs, exp).pvalue


@pytest.mark.parametrize("mode", ["test", "production"])
def test_oracle_outcomes_follow_closed_form(oracle_mod, mode):
    n = 400_000
    rng = np.random.default_rng(2024)
    w = _sample_workload(n, rng)
    r = oracle_mod.verify(w, production=(mode == "production"), seed=17, offset=5, with_diag=False)
    assert r["status"] == 0
    pval = _chi2_outcomes(r["out_tokens"], r["num_accepted"], n)
    assert pval > 0.01
    # first committed token ~ p_0 exactly
    first = np.bincount(r["out_tokens"][:, 0], minlength=V)
    assert scipy.stats.chisquare(first, n * np.array(P_ROWS[0]) / 16).pvalue > 0.01
    # P(A >= k) = prod beta_j ; histogram of A
    beta = [sum(min(a, b) for a, b in zip(P16[j], Q16[j])) for j in range(GAMMA)]
    pa = [1 - beta[0], beta[0] * (1 - beta[1]), beta[0] * beta[1]]
    hist = np.bincount(r["num_accepted"], minlength=GAMMA + 1)
    assert scipy.stats.chisquare(hist, n * np.array([float(x) for x in pa])).pvalue > 0.01
    # bonus given A = gamma follows p_gamma
    bon = r["out_tokens"][r["num_accepted"] == GAMMA, GAMMA]
    cnt = np.bincount(bon, minlength=V)
    assert scipy.stats.chisquare(cnt, len(bon) * np.array(P_ROWS[GAMMA]) / 16).pvalue > 0.01


def test_fixed_draft_branch_probabilities(oracle_mod):
    """Given a fixed draft y: P(out=y) = min(1, p(y)/q(y)) and
    P(out=x) = (1 - alpha) * r(x) / sum r for x != y (page 2, section 04)."""
    n = 300_000
    rng = np.random.default_rng(77)
    p = np.array([0.1, 0.2, 0.3, 0.15, 0.25], np.float32)
    q = np.array([0.4, 0.1, 0.2, 0.2, 0.1], np.float32)
    y = 0
    w = hand_workload(np.tile(np.stack([p, p]), (n, 1)), np.tile(q, (n, 1)), [y] * n, [1] * n,
                      u=rng.random(n, dtype=np.float32), E=rng.standard_exponential((n, 5), dtype=np.float32))
    r = oracle_mod.verify(w, with_diag=False)
    first = r["out_tokens"][:, 0]
    alpha = min(1.0, float(p[y]) / float(q[y]))
    res = np.maximum(p.astype(np.float64) - q, 0)
    expect = (1 - alpha) * res / res.sum()
    expect[y] += alpha
    obs = np.bincount(first, minlength=5)
    assert np.all(obs[expect == 0] == 0)  # (p - q)+ = 0 and x != y: never emitted
    nz = expect > 0
    assert scipy.stats.chisquare(obs[nz], n * expect[nz]).pvalue > 0.01


def test_planted_mistakes_are_caught(oracle_mod, tmp_path):
    """Each plausible slip in the oracle's arithmetic (a swapped operand, a
    non-strict comparison, a wrong row index, a dropped rollback term, a
    highest-index tie break) fails at least one of the pins above.  The
    mistakes are planted in copies of the oracle source, compiled on the CPU."""
    import ctypes
    import subprocess
    assert not _run_pins_against_current(oracle_mod)  # the unmodified oracle passes them all
    src = (oracle_mod._SRC).read_text()
    mutants = {
        "accept <= ": ("if (!a->synthetic_rates && uq < py) {", "if (!a->synthetic_rates && uq <= py) {"),
        "residual q-p": ("float d = p[x] - q[x];", "float d = q[x] - p[x];"),
        "target row s_i": ("const int64_t tb = s + i;", "const int64_t tb = s;"),
        "race highest index": ("if (best < 0 || key > bk) {", "if (best < 0 || key >= bk) {"),
        "rollback gamma": ("a->num_computed_tokens[i] -= (g - A);", "a->num_computed_tokens[i] -= (g - A - 1);"),
        "slots from A": ("for (int j = A + 1; j <= g; ++j)", "for (int j = A; j <= g; ++j)"),
        "bonus row g-1": ("if (prob_row(a, 1, tb + g, temp,", "if (prob_row(a, 1, tb + g - 1, temp,"),
        "u times p": ("float uq = u * qy;", "float uq = u * py;"),
        "greedy keeps y": ("toks[j] = gj;", "toks[j] = (j < g) ? a->draft_ids[s + j] : gj;"),
        "topk strict": ("(double)l[x] >= tau && (double)l[x] >= cut", "(double)l[x] > tau && (double)l[x] >= cut"),
        "subnormal temperature accepted": ("return t == 0.0f || (t >= FLT_MIN && !isinf(t));",
                                           "return t == 0.0f || (t > 0.0f && !isinf(t));"),
    }
    failures = {}
    for name, (old, new) in mutants.items():
        assert src.count(old) >= 1, name
        msrc = tmp_path / f"m_{abs(hash(name))}.c"
        msrc.write_text(src.replace(old, new))
        so = tmp_path / f"m_{abs(hash(name))}.so"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", str(so),
                        str(msrc), "-lm"], check=True)
        saved = oracle_mod._LIB
        try:
            lib = ctypes.CDLL(str(so))
            oracle_mod._LIB = None
            orig_build = oracle_mod.build
            oracle_mod.build = lambda force=False, _so=so: _so
            caught = _run_pins_against_current(oracle_mod)
        finally:
            oracle_mod.build = orig_build
            oracle_mod._LIB = saved
        failures[name] = caught
    missed = [k for k, v in failures.items() if not v]
    assert not missed, f"planted mistakes not caught: {missed}"


def _run_pins_against_current(oracle_mod):
    """Run the deterministic pins; return True if any of them fails."""
    import inspect
    import test_oracle_pins as pins
    names = [n for n, f in inspect.getmembers(pins, inspect.isfunction) if n.startswith("test_")]
    skip = {"test_production_draws_have_the_stated_laws", "test_philox_known_answers"}
    for n in names:
        if n in skip:
            continue
        f = getattr(pins, n)
        params = inspect.signature(f).parameters
        cases = [{}]
        marks = getattr(f, "pytestmark", [])
        for m in marks:
            if m.name == "parametrize":
                argnames = [a.strip() for a in (m.args[0].split(",") if isinstance(m.args[0], str) else m.args[0])]
                cases = [dict(zip(argnames, v if isinstance(v, tuple) else (v,))) for v in m.args[1]]
        for c in cases:
            kw = dict(c)
            if "oracle_mod" in params:
                kw["oracle_mod"] = oracle_mod
            try:
                f(**kw)
            except Exception:
                return True
    return False
