"""Pins of the oracle's n-gram proposer ("vLLM source walk-through (10)",
section "NgramProposer") against hand-worked cases, a brute-force search in
another formulation, and a KMP scan written from the page's description."""
import ctypes
import subprocess

import numpy as np
import pytest

from conftest import load_golden


def brute_force(t, min_n, max_n, k, max_model_len):
    """Longest n in [min_n, max_n] whose tail occurs earlier with a token after
    it; the most recent such occurrence; the tokens that followed it."""
    L = len(t)
    if L < min_n:
        return []
    kk = min(k, max_model_len - L)
    if kk <= 0:
        return []
    for n in range(max_n, min_n - 1, -1):
        if n > L - 1:
            continue
        tail = list(t[L - n:])
        for p in range(L - 1 - n, -1, -1):  # latest start first, the occurrence ends before L - 1
            if list(t[p:p + n]) == tail:
                start = p + n
                return list(t[start:start + min(kk, L - start)])
    return []


def kmp_reversed(t, min_n, max_n, k, max_model_len):
    """The page's method: read the history backwards, keep a prefix-function
    table of at most max_n entries, scan for the longest prefix match (capped
    at max_n), keep the first position where a strictly longer match appears."""
    L = len(t)
    if L < min_n:
        return []
    kk = min(k, max_model_len - L)
    if kk <= 0:
        return []
    r = list(t[::-1])
    pi = [0] * max_n  # prefix function of the pattern r[0:max_n]
    m = 0
    best, at = 0, -1
    for i in range(1, L):
        while m > 0 and (m == max_n or r[i] != r[m]):
            m = pi[m - 1]
        if r[i] == r[m]:
            m += 1
        if i < max_n:
            pi[i] = m
        if m > best:
            best, at = m, i
    if best < min_n:
        return []
    start = L - 1 - at + best
    return list(t[start:start + min(kk, L - start)])


def run_oracle(oracle_mod, t, min_n, max_n, k, mml):
    o = oracle_mod.ngram_propose(np.asarray(t, np.int32), [len(t)], min_ngram=min_n, max_ngram=max_n, k=k,
                                 max_model_len=mml)
    n = int(o["num_draft_tokens"][0])
    assert np.all(o["draft_token_ids"][0, n:] == -1)
    return list(o["draft_token_ids"][0, :n])


def test_golden_cases(oracle_mod):
    g = load_golden("ngram_examples.txt")
    for c in range(1, 7):
        t = [int(x) for x in g[f"c{c}_tokens"]]
        min_n, max_n, k, mml = (int(x) for x in g[f"c{c}_params"])
        expect = [int(x) for x in g[f"c{c}_expect"]]
        assert run_oracle(oracle_mod, t, min_n, max_n, k, mml) == expect, c
        assert brute_force(t, min_n, max_n, k, mml) == expect, c
        assert kmp_reversed(t, min_n, max_n, k, mml) == expect, c


@pytest.mark.parametrize("alphabet", [2, 3, 6])
def test_random_histories_match_both_formulations(oracle_mod, alphabet):
    rng = np.random.default_rng(alphabet)
    for _ in range(400):
        L = int(rng.integers(0, 40))
        t = rng.integers(0, alphabet, size=L).tolist()
        min_n = int(rng.integers(1, 5))
        max_n = int(rng.integers(min_n, 8))
        k = int(rng.integers(0, 6))
        mml = int(rng.integers(max(L - 2, 1), L + 8))
        got = run_oracle(oracle_mod, t, min_n, max_n, k, mml)
        assert got == brute_force(t, min_n, max_n, k, mml), (t, min_n, max_n, k, mml)
        assert got == kmp_reversed(t, min_n, max_n, k, mml), (t, min_n, max_n, k, mml)


def test_ragged_batch_and_bad_ranges(oracle_mod):
    rng = np.random.default_rng(5)
    hist = [rng.integers(0, 3, size=n).tolist() for n in (0, 1, 9, 30, 4)]
    flat = sum(hist, [])
    cu = np.cumsum([len(h) for h in hist])
    o = oracle_mod.ngram_propose(flat, cu, min_ngram=2, max_ngram=3, k=4, max_model_len=64)
    assert o["status"] == 0
    for q, h in enumerate(hist):
        n = int(o["num_draft_tokens"][q])
        assert list(o["draft_token_ids"][q, :n]) == brute_force(h, 2, 3, 4, 64)
    bad = cu.copy()
    bad[2] = bad[1] - 1  # a request ending before it starts
    o = oracle_mod.ngram_propose(flat, bad, min_ngram=2, max_ngram=3, k=4, max_model_len=64)
    assert o["status"] == oracle_mod.BAD_CU
    assert o["num_draft_tokens"][2] == 0 and np.all(o["draft_token_ids"][2] == -1)


def test_planted_mistakes_are_caught(oracle_mod, tmp_path):
    """Each plausible slip in the oracle's n-gram search fails the pins above."""
    src = oracle_mod._SRC.read_text()
    mutants = {
        "tie keeps the latest end": ("if (m > best_m) {", "if (m >= best_m) {"),
        "cap ignores i": ("int64_t cap = i < max_ngram ? i : max_ngram;", "int64_t cap = max_ngram;"),
        "start off by one": ("const int64_t start = L - 1 - best_i + best_m;",
                             "const int64_t start = L - best_i + best_m;"),
        "no room check": ("if (L - start < kk) kk = L - start;", "(void)0;"),
        "min_ngram ignored": ("if (best_m < min_ngram) continue;", "if (best_m < 1) continue;"),
    }
    for name, (old, new) in mutants.items():
        assert src.count(old) == 1, name
        msrc = tmp_path / f"n_{abs(hash(name))}.c"
        msrc.write_text(src.replace(old, new))
        so = tmp_path / f"n_{abs(hash(name))}.so"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", str(so),
                        str(msrc), "-lm"], check=True)
        saved = oracle_mod._LIB
        orig_build = oracle_mod.build
        try:
            oracle_mod._LIB = None
            oracle_mod.build = lambda force=False, _so=so: _so
            caught = False
            for test in (test_golden_cases, lambda m: test_random_histories_match_both_formulations(m, 2),
                         lambda m: test_random_histories_match_both_formulations(m, 3)):
                try:
                    test(oracle_mod)
                except (AssertionError, IndexError, ValueError):
                    caught = True
                    break
        finally:
            oracle_mod.build = orig_build
            oracle_mod._LIB = saved
        assert caught, name
