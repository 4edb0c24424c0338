"""Pins of the oracle's recursive rejection with children drawn without replacement
(Sequoia, Chen et al.; SD 20.5, the paragraph after the proof of "Recursive rejection at a
node with several children": each rejected token is zeroed in q, which is renormalised
before the next try).

The output law is integrated exactly over the uniforms (tests/exact_integration.py,
tree_rr_outcome_law) and averaged over every ordered draw of distinct children, each with
its probability prod_i q(s_i) / (1 - sum_{j<i} q(s_j)).  Pins: the emitted token follows p
(the box's theorem, which holds try by try when try i draws from q_i); the chance that some
child is accepted equals a recursion over the draws written from the rule's acceptance
probabilities (no uniforms); for a peaked drafter that disagrees with the target,
drawing without replacement accepts some child more often than i.i.d. children (the
page's reason for the variant); one child is the i.i.d. rule; duplicate siblings are an
input error.  Four plausible mistakes, planted in a one-node copy of the rule that
first reproduces the oracle, each move the emitted law away from p.
"""
import itertools

import numpy as np
import pytest

from oracle import specdec_oracle as so
from exact_integration import tree_rr_outcome_law


def _log(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, dtype=np.float64))


def _emitted(r):
    t, pth = r["tokens"], r["path"]
    return tuple(int(x) for x in t[t >= 0]), tuple(int(x) for x in pth[pth >= 0])


def _wor_draws(q, k):
    """Every ordered draw of k distinct tokens from q without replacement, with its
    probability."""
    V = len(q)
    for toks in itertools.permutations(range(V), k):
        w, left = 1.0, 1.0
        for t in toks:
            if left <= 0.0:
                w = 0.0
                break
            w *= q[t] / left
            left -= q[t]
        if w > 0.0:
            yield toks, w


def _iid_draws(q, k):
    for toks in itertools.product(range(len(q)), repeat=k):
        w = float(np.prod([q[t] for t in toks]))
        if w > 0.0:
            yield toks, w


def one_node_law(p, q, k, verify_one, draws):
    """Law of the first emitted token and P(some child accepted) at a root with k leaf
    children drawn by `draws`; verify_one(toks, u) -> (emitted, path)."""
    V = len(p)
    first = np.zeros(V)
    acc = 0.0
    parents = [-1] * k
    for toks, w in draws(q, k):
        law = tree_rr_outcome_law(lambda u, toks=toks: verify_one(toks, u), parents)
        for out, m in law.items():
            first[out[0]] += w * m
            if len(out) >= 2:
                acc += w * m
    return first, acc


def oracle_one(p, q, wor):
    V = len(p)

    def verify_one(toks, u):
        k = len(toks)
        logits = np.vstack([_log(p)] + [np.zeros(V)] * k)
        qrows = np.vstack([q] + [np.full(V, 1.0 / V)] * k)
        r = so.verify_tree_rr_sequence(logits, qrows, list(toks), [-1] * k, 1.0, u, 2, without_replacement=wor)
        assert r["status"] & so.STATUS_ERROR_MASK == 0, r["status"]
        return _emitted(r)
    return verify_one


def wor_acceptance(R, q, k):
    """P(some child accepted), k children drawn without replacement from q, target R: try
    one draws s from q and accepts with probability min(1, R(s)/q(s)); a rejection of s
    leaves R' = (R - q)+ normalised and q' = q without s, renormalised."""
    if k == 0:
        return 0.0
    total = 0.0
    r = np.maximum(R - q, 0.0)
    Rn = r / r.sum() if r.sum() > 0.0 else R
    for s in range(len(q)):
        if q[s] <= 0.0:
            continue
        a = min(1.0, R[s] / q[s])
        total += q[s] * a
        if a < 1.0:
            qn = q.copy()
            qn[s] = 0.0
            if qn.sum() <= 0.0:
                continue
            total += q[s] * (1.0 - a) * wor_acceptance(Rn, qn / qn.sum(), k - 1)
    return total


@pytest.mark.parametrize("k", [1, 2, 3])
@pytest.mark.parametrize("seed", [0, 1, None])
def test_output_is_p_and_acceptance_follows_the_draws(k, seed):
    if seed is None:  # a first residual that keeps several tokens, so every try matters
        p = np.array([0.10, 0.40, 0.30, 0.20])
        q = np.array([0.40, 0.30, 0.20, 0.10])
    else:
        rng = np.random.default_rng(seed)
        p = rng.dirichlet(np.ones(4))
        q = rng.dirichlet(np.ones(4) * 0.8)
    first, acc = one_node_law(p, q, k, oracle_one(p, q, True), _wor_draws)
    np.testing.assert_allclose(first, p, atol=1e-12)
    assert acc == pytest.approx(wor_acceptance(p, q, k), abs=1e-12)


def test_without_replacement_beats_iid_for_a_peaked_drafter():
    # the drafter is sure of a token the target rarely wants: i.i.d. children keep
    # proposing it, children without replacement move on to other tokens
    p = np.array([0.10, 0.40, 0.30, 0.20])
    q = np.array([0.85, 0.05, 0.05, 0.05])
    for k in (2, 3):
        f_wor, a_wor = one_node_law(p, q, k, oracle_one(p, q, True), _wor_draws)
        f_iid, a_iid = one_node_law(p, q, k, oracle_one(p, q, False), _iid_draws)
        np.testing.assert_allclose(f_wor, p, atol=1e-12)
        np.testing.assert_allclose(f_iid, p, atol=1e-12)
        assert a_wor > a_iid + 0.05, (k, a_wor, a_iid)
    # one child: the same rule
    _, a1w = one_node_law(p, q, 1, oracle_one(p, q, True), _wor_draws)
    _, a1i = one_node_law(p, q, 1, oracle_one(p, q, False), _iid_draws)
    assert a1w == pytest.approx(a1i, abs=1e-15)
    assert a1i == pytest.approx(np.minimum(p, q).sum(), abs=1e-12)


def test_one_child_equals_the_iid_rule_on_random_trees():
    rng = np.random.default_rng(3)
    V, N = 9, 12
    parents = [-1] + list(range(N - 1))  # a path: every node is its parent's only child
    for _ in range(40):
        logits = rng.standard_normal((N + 1, V))
        q = rng.dirichlet(np.ones(V), size=N + 1)
        toks = [int(t) for t in rng.integers(0, V, size=N)]
        u = rng.random(N + 1)
        a = so.verify_tree_rr_sequence(logits, q, toks, parents, 0.8, u, N + 1, without_replacement=True)
        b = so.verify_tree_rr_sequence(logits, q, toks, parents, 0.8, u, N + 1)
        assert a["status"] == b["status"]
        np.testing.assert_array_equal(a["tokens"], b["tokens"])
        np.testing.assert_array_equal(a["path"], b["path"])


def test_duplicate_siblings_are_an_input_error_only_without_replacement():
    V = 6
    logits = np.zeros((4, V))
    q = np.full((4, V), 1.0 / V)
    parents = [-1, -1, 0]
    u = np.full(4, 0.5)
    dup = so.verify_tree_rr_sequence(logits, q, [2, 2, 2], parents, 1.0, u, 3, without_replacement=True)
    assert dup["status"] == so.STATUS_BAD_TREE and dup["n_accepted"] == -1
    assert (dup["tokens"] == -1).all()
    # the same tokens under different parents are fine; i.i.d. children may repeat
    ok = so.verify_tree_rr_sequence(logits, q, [2, 3, 2], parents, 1.0, u, 3, without_replacement=True)
    assert ok["status"] & so.STATUS_ERROR_MASK == 0
    iid = so.verify_tree_rr_sequence(logits, q, [2, 2, 2], parents, 1.0, u, 3)
    assert iid["status"] & so.STATUS_ERROR_MASK == 0


def test_used_up_draft_mass_follows_the_zero_q_rule():
    # q is one-hot on token 0; after token 0 is rejected no mass is left, so the next
    # child (token 1, q = 0) is accepted iff the residual gives it mass
    p = np.array([0.2, 0.5, 0.3, 0.0])
    q = np.array([1.0, 0.0, 0.0, 0.0])
    logits = np.vstack([_log(p), np.zeros((2, 4))])
    qrows = np.vstack([q, np.full((2, 4), 0.25)])
    u = np.array([0.5, 0.9, 0.5])  # u[1] = 0.9 > p(0)/q(0) = 0.2: token 0 rejected
    r = so.verify_tree_rr_sequence(logits, qrows, [0, 1], [-1, -1], 1.0, u, 2, without_replacement=True)
    assert r["status"] & so.STATUS_ZERO_Q
    assert r["n_accepted"] == 1 and r["path"][0] == 1 and r["tokens"][0] == 1


# ---- planted mistakes ------------------------------------------------------------------

def _one_node_variant(p, q, toks, u, mistake=None):
    """The rule at one node with leaf children, written out again, with an optional
    planted mistake: 'iid' (q as given in test and residual: the i.i.d. rule applied to
    children drawn without replacement), 'renorm_test_only' (q_i in the test, q in the
    residual), 'renorm_residual_only' (q in the test, q_i in the residual),
    'zero_current' (the tried token is removed from q before its own test).  Returns
    (emitted, path) like the oracle."""
    R = p.copy()
    rejected, Z = [], 1.0
    for j, s in enumerate(toks):
        qi = q / Z if Z > 0.0 else np.zeros_like(q)
        qi[rejected] = 0.0
        qt = q if mistake in ("iid", "renorm_residual_only") else qi.copy()
        if mistake == "zero_current":
            qt[s] = 0.0
        qr = q if mistake in ("iid", "renorm_test_only") else qi
        qs = qt[s]
        accept = R[s] > 0.0 if qs == 0.0 else u[1 + j] * qs < R[s]
        if accept:
            return (s, 0), (j,)
        r = np.maximum(R - qr, 0.0)
        if r.sum() > 0.0:
            R = r / r.sum()
        rejected.append(s)
        Z -= q[s]
    y, _, _ = so.inverse_cdf(R, u[0])
    return (y,), ()


def test_the_planted_copy_reproduces_the_oracle():
    rng = np.random.default_rng(7)
    V = 5
    for _ in range(300):
        p = rng.dirichlet(np.ones(V))
        q = rng.dirichlet(np.ones(V) * 0.7)
        k = int(rng.integers(1, 4))
        toks = [int(t) for t in rng.permutation(V)[:k]]
        u = rng.random(k + 1)
        want = oracle_one(p, q, True)(toks, list(u))
        got = _one_node_variant(p, q, toks, u)
        assert want[1] == got[1]
        assert want[0][0] == got[0][0]


@pytest.mark.parametrize("mistake", ["iid", "renorm_test_only", "renorm_residual_only", "zero_current"])
def test_planted_mistakes_break_the_output_law(mistake):
    # a target whose first residual keeps several tokens, so later tries matter
    p = np.array([0.10, 0.40, 0.30, 0.20])
    q = np.array([0.40, 0.30, 0.20, 0.10])
    worst = 0.0
    for k in (2, 3):
        first, _ = one_node_law(p, q, k, lambda toks, u: _one_node_variant(p, q, toks, u, mistake), _wor_draws)
        worst = max(worst, float(np.abs(first - p).max()))
    assert worst > 1e-3, (mistake, worst)
    # the unplanted copy gives p on the same draws
    first, _ = one_node_law(p, q, 3, lambda toks, u: _one_node_variant(p, q, toks, u), _wor_draws)
    np.testing.assert_allclose(first, p, atol=1e-12)
