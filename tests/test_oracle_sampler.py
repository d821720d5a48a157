"""Pins of the oracle's draft-side sampler ("vLLM source walk-through (10)",
section "propose() multi-step loop": each draft token is drawn from the draft
distribution).  The transform is the one pinned in test_oracle_pins; here the
draw itself is checked: over many rows with the same logits, token
frequencies follow the transformed probabilities (chi-square, test mode and
the oracle's own Philox), greedy rows take the argmax, and the probability
row written out is the transform's output."""
import numpy as np
import pytest
import scipy.stats

import oracle


@pytest.mark.parametrize("production", [False, True])
@pytest.mark.parametrize("temp,k,p", [(1.0, 0, 1.0), (0.7, 4, 0.9), (1.5, 0, 0.8)])
def test_sampler_frequencies_follow_transformed_row(production, temp, k, p):
    rng = np.random.default_rng(4)
    V, R = 7, 200_000
    l = rng.standard_normal(V).astype(np.float32) * 1.5
    probs, _, rc = oracle.logits_to_probs(l, temp, k, p)
    assert rc == 0
    rows = np.tile(l, (R, 1))
    E = None if production else rng.standard_exponential((R, V), dtype=np.float32)
    r = oracle.sample_rows(rows, temperature=np.full(R, temp), top_k=np.full(R, k), top_p=np.full(R, p),
                           exponentials=E, seed=3, offset=1, with_probs=False)
    assert r["status"] == 0
    cnt = np.bincount(r["tokens"], minlength=V)
    expect = probs.astype(np.float64)
    assert np.all(cnt[expect == 0] == 0)
    nz = expect > 0
    assert scipy.stats.chisquare(cnt[nz], R * expect[nz] / expect[nz].sum()).pvalue > 0.01


def test_sampler_greedy_and_probs_output():
    rng = np.random.default_rng(5)
    l = rng.standard_normal((6, 50)).astype(np.float32)
    l[2, 7] = l[2, 9] = l[2].max() + 1  # tie: lowest index
    temps = np.array([0, 1, 0, 0.5, 1, 2], np.float32)
    r = oracle.sample_rows(l, temperature=temps, top_k=np.full(6, 10), top_p=np.full(6, 0.95),
                           exponentials=rng.standard_exponential((6, 50), dtype=np.float32))
    for i in (0, 2):
        assert r["tokens"][i] == int(np.argmax(l[i]))
    assert r["tokens"][2] == 7
    for i in (1, 3, 4, 5):
        expect, _, _ = oracle.logits_to_probs(l[i], temps[i], 10, 0.95)
        np.testing.assert_array_equal(r["probs"][i], expect)
        assert expect[r["tokens"][i]] > 0


def test_sampler_streams_differ_from_the_verifier():
    """Same seed and offset: the sampler's draws for row r are not the
    verifier's E draws for request r (different Philox key)."""
    V = 64
    l = np.zeros((256, V), np.float32)  # uniform rows: the token is the argmin of E
    r = oracle.sample_rows(l, seed=11, offset=0, with_probs=False)
    ver_argmin = [int(np.argmin([oracle.exponential(11, 0, i, x) for x in range(V)])) for i in range(256)]
    assert np.mean(np.array(ver_argmin) == r["tokens"]) < 0.2


def test_sampler_invalid_rows():
    l = np.zeros((3, 8), np.float32)
    l[1, 3] = np.nan
    r = oracle.sample_rows(l, temperature=np.array([-1.0, 1.0, 1.0], np.float32),
                           exponentials=np.ones((3, 8), np.float32))
    assert r["tokens"][0] == -1 and r["tokens"][1] == -1 and r["tokens"][2] == 0
    assert r["status"] == oracle.BAD_PARAM | oracle.BAD_VALUES
