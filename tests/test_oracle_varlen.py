"""Pins of the oracle's chain round with a per-request number of verified drafts
(SD 20.5, "Choosing how much to verify at every step").

The output law is integrated exactly over the uniforms (tests/exact_integration.py), so
the values are properties of the oracle's decisions: the box "Trimming a draft can break
exactness" prints (0.5, 0.18, 0.32) for a trim that looks at the draft, while a count of
drafts chosen without looking at them (always, never, or by an independent coin) keeps the
output law equal to p.
"""
import numpy as np
import pytest

from oracle import specdec_oracle as so
from exact_integration import round_outcome_law
from golden import read_fixture


def _first_token_law(p, q, choose_gamma):
    """Law of the first emitted token for one drafted token x ~ q whose verification count
    is choose_gamma(x) (0 or 1)."""
    V = len(p)
    logits = np.vstack([np.log(p), np.log(p)])
    law = np.zeros(V)
    for x in range(V):
        gb = choose_gamma(x)

        def verify(d, u, gb=gb):
            uu = list(u) + [0.5] * (2 - len(u))
            r = so.verify_chain_varlen_sequence(logits, q[None, :], d, 1.0, uu, gb)
            assert r["status"] & so.STATUS_ERROR_MASK == 0
            t = r["tokens"]
            return tuple(int(v) for v in t[t >= 0])

        for out, m in round_outcome_law(verify, [x], gb).items():
            law[out[0]] += q[x] * m
    return law


def test_draft_dependent_trim_gives_the_page_counterexample():
    fx = read_fixture("trim_counterexample.txt")
    p = np.array([float(v) for v in fx["p"]])
    q = np.array([float(v) for v in fx["q"]])
    got = _first_token_law(p, q, lambda x: 0 if x == 1 else 1)
    np.testing.assert_allclose(got, [float(v) for v in fx["trimmed_output"]], atol=1e-12)


@pytest.mark.parametrize("rule", ["always", "never"])
def test_draft_independent_counts_keep_the_target_law(rule):
    fx = read_fixture("trim_counterexample.txt")
    p = np.array([float(v) for v in fx["p"]])
    q = np.array([float(v) for v in fx["q"]])
    got = _first_token_law(p, q, (lambda x: 1) if rule == "always" else (lambda x: 0))
    np.testing.assert_allclose(got, p, atol=1e-12)


def test_independent_coin_keeps_the_target_law():
    """gamma_b from a coin that does not see the draft: the law mixes two exact laws."""
    rng = np.random.default_rng(2)
    p, q = rng.dirichlet(np.ones(4)), rng.dirichlet(np.ones(4))
    mix = 0.3 * _first_token_law(p, q, lambda x: 1) + 0.7 * _first_token_law(p, q, lambda x: 0)
    np.testing.assert_allclose(mix, p, atol=1e-12)


def test_full_count_is_the_chain_rule_and_counts_truncate():
    rng = np.random.default_rng(5)
    V, gamma = 40, 5
    for _ in range(30):
        logits = rng.standard_normal((gamma + 1, V)) * 2
        q = rng.dirichlet(np.ones(V), size=gamma)
        d = [int(rng.integers(V)) for _ in range(gamma)]
        u = rng.random(gamma + 1)
        T = float(rng.uniform(0.2, 1.5))
        full = so.verify_chain_varlen_sequence(logits, q, d, T, u, gamma)
        chain = so.verify_chain_sequence(logits, q, d, T, u)
        np.testing.assert_array_equal(full["tokens"], chain["tokens"])
        for gb in range(gamma + 1):
            r = so.verify_chain_varlen_sequence(logits, q, d, T, u, gb)
            assert 0 <= r["J"] <= gb
            assert (r["tokens"][gb + 1:] == -1).all()
            assert np.isnan(r["p_draft"][gb:]).all()
            # the first gb tests are the full round's own, with the same uniforms
            assert r["J"] == min(chain["J"], gb)
            np.testing.assert_array_equal(r["tokens"][:r["J"]], chain["tokens"][:r["J"]])


def test_out_of_range_count_is_an_error():
    logits = np.zeros((3, 5))
    q = np.full((2, 5), 0.2)
    for gb in (-1, 3):
        r = so.verify_chain_varlen_sequence(logits, q, [0, 1], 1.0, [0.5, 0.5, 0.5], gb)
        assert r["status"] == so.STATUS_BAD_TOKEN and r["J"] == -1 and (r["tokens"] == -1).all()
