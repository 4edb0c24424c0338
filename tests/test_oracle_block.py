"""Pins of the oracle's block verification (Art of Guessing, "Block verification").

The output law is integrated exactly over the uniforms (tests/exact_integration.py,
block_round_outcome_law), so every value below is a property of the oracle's decisions,
not a restatement of its formulas: the toy example's printed 11/9, the lossless output
law (the emitted tokens follow the target exactly, Sun et al.'s guarantee), the claim
that block verification never accepts fewer tokens than the token-wise rule, and the
reduction to greedy matching for a one-hot target.
"""
import itertools

import numpy as np
import pytest

from oracle import specdec_oracle as so
from exact_integration import (bigram_round_law, block_round_outcome_law, first_two_tokens_law,
                               round_outcome_law)
from golden import read_fixture


def _fr(xs):
    return np.array([float(x) for x in xs])


def block_rows(p_rows, q_rows, drafts, u):
    """Adapter: probabilities -> logits log p at T = 1; emitted tokens as a tuple."""
    with np.errstate(divide="ignore"):
        logits = np.log(np.asarray(p_rows, dtype=np.float64))
    r = so.verify_block_sequence(logits, np.asarray(q_rows), drafts, 1.0, u)
    assert r["status"] & so.STATUS_ERROR_MASK == 0, r["status"]
    t = r["tokens"]
    return tuple(int(x) for x in t[t >= 0])


def chain_rows(p_rows, q_rows, drafts, u):
    with np.errstate(divide="ignore"):
        logits = np.log(np.asarray(p_rows, dtype=np.float64))
    r = so.verify_chain_sequence(logits, np.asarray(q_rows), drafts, 1.0, u)
    t = r["tokens"]
    return tuple(int(x) for x in t[t >= 0])


def _expected_accepted(rows_fn, law_fn, p_rows_of, q_rows_of, q_of, V, gamma):
    """E[accepted drafts] with drafts drawn from q (q_of(drafts) = their probability)."""
    total = 0.0
    for drafts in itertools.product(range(V), repeat=gamma):
        w = q_of(drafts)
        if w == 0.0:
            continue
        pr, qr = p_rows_of(drafts), q_rows_of(drafts)
        law = law_fn(lambda d, u: rows_fn(pr, qr, d, u), list(drafts), gamma)
        total += w * sum(m * (len(out) - 1) for out, m in law.items())
    return total


def test_toy_example_block_value():
    """The page's toy: p = (1/3, 2/3), q = (2/3, 1/3) at every position, gamma = 2;
    block verification accepts 11/9 tokens per round (token-wise: 10/9)."""
    fx = read_fixture("block_verify_toy.txt")
    p, q, gamma = _fr(fx["p"]), _fr(fx["q"]), int(fx["gamma"][0])
    rows_p = np.stack([p] * (gamma + 1))
    rows_q = np.stack([q] * gamma)
    q_of = lambda d: float(np.prod([q[x] for x in d]))
    block = _expected_accepted(block_rows, block_round_outcome_law, lambda d: rows_p, lambda d: rows_q, q_of,
                               len(p), gamma)
    token = _expected_accepted(chain_rows, round_outcome_law, lambda d: rows_p, lambda d: rows_q, q_of,
                               len(p), gamma)
    assert block == pytest.approx(_fr(fx["block_accepted"])[0], abs=1e-12)
    assert token == pytest.approx(_fr(fx["tokenwise_accepted"])[0], abs=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_block_output_law_is_the_target(seed):
    """Lossless: under a bigram target and drafter, the first two generated tokens of
    block verification follow the target's own joint law exactly."""
    rng = np.random.default_rng(seed)
    V, gamma = 3, 2
    P = rng.dirichlet(np.ones(V), size=V)
    Q = rng.dirichlet(np.ones(V) * 0.7, size=V)
    start = 1
    joint = first_two_tokens_law(block_rows, P, Q, start, gamma, round_law=block_round_outcome_law)
    want = P[start][:, None] * P
    np.testing.assert_allclose(joint, want, atol=1e-12)


@pytest.mark.parametrize("seed", [3, 4, 5, 6])
def test_block_accepts_at_least_as_many_as_tokenwise(seed):
    """Sun et al. (as the page states): for a given draft distribution block
    verification maximises the expected accepted length among lossless rules, so it is
    never below the token-wise rule; here on random per-position distributions."""
    rng = np.random.default_rng(seed)
    V, gamma = 3, 3
    rows_p = rng.dirichlet(np.ones(V), size=gamma + 1)
    rows_q = rng.dirichlet(np.ones(V), size=gamma)
    q_of = lambda d: float(np.prod([rows_q[i][x] for i, x in enumerate(d)]))
    block = _expected_accepted(block_rows, block_round_outcome_law, lambda d: rows_p, lambda d: rows_q, q_of,
                               V, gamma)
    token = _expected_accepted(chain_rows, round_outcome_law, lambda d: rows_p, lambda d: rows_q, q_of, V,
                               gamma)
    assert block >= token - 1e-12


def test_one_hot_target_reduces_to_greedy_matching():
    """With a one-hot target the block rule keeps drafts while they are the argmax and
    emits the argmax after them: the same tokens as greedy verification."""
    rng = np.random.default_rng(7)
    V, gamma = 5, 4
    for _ in range(20):
        logits = rng.standard_normal((gamma + 1, V))
        z = logits.argmax(axis=1)
        drafts = [int(z[i]) if rng.random() < 0.7 else int((z[i] + 1) % V) for i in range(gamma)]
        q = rng.dirichlet(np.ones(V), size=gamma)
        u = rng.random(gamma + 1)
        onehot = np.full((gamma + 1, V), -np.inf)
        onehot[np.arange(gamma + 1), z] = 0.0
        sampled = so.verify_block_sequence(onehot, q, drafts, 1.0, u)
        greedy = so.verify_block_sequence(logits, q, drafts, 0.0, u)
        chain = so.verify_chain_sequence(logits, q, drafts, 0.0, u)
        np.testing.assert_array_equal(sampled["tokens"], greedy["tokens"])
        np.testing.assert_array_equal(greedy["tokens"], chain["tokens"])


def test_block_status_reads_every_position():
    V, gamma = 6, 3
    logits = np.zeros((gamma + 1, V))
    q = np.full((gamma, V), 1.0 / V)
    u = np.full(gamma + 1, 0.5)
    d = [0, 1, 2]
    assert so.verify_block_sequence(logits, q, d, 1.0, u)["status"] == 0
    bad = logits.copy(); bad[gamma, 2] = np.nan
    assert so.verify_block_sequence(bad, q, d, 1.0, u)["status"] & so.STATUS_BAD_LOGIT
    qb = q.copy(); qb[gamma - 1, 5] = -1.0  # far from the drafts: the whole row is read
    r = so.verify_block_sequence(logits, qb, d, 1.0, u)
    assert r["status"] & so.STATUS_BAD_PROB and r["J"] == -1 and (r["tokens"] == -1).all()
    ub = u.copy(); ub[gamma - 1] = 1.0
    assert so.verify_block_sequence(logits, q, d, 1.0, ub)["status"] & so.STATUS_BAD_UNIFORM
    assert so.verify_block_sequence(logits, q, [0, 9, 2], 1.0, u)["status"] & so.STATUS_BAD_TOKEN
    assert so.verify_block_sequence(logits, q, d, np.nan, u)["status"] == so.STATUS_BAD_TEMPERATURE
    # greedy sequences ignore q and u
    assert so.verify_block_sequence(logits, qb, d, 0.0, ub)["status"] == 0
