"""Pins of the oracle's recursive-rejection tree verification (SD 20.5, box "Recursive
rejection at a node with several children").

The output law is integrated exactly over the uniforms (tests/exact_integration.py,
tree_rr_outcome_law) and averaged over children drafted i.i.d. from q, so the values
below are properties of the oracle's decisions: the emitted token follows p whatever the
number of children (the box's theorem), the chance that some child is accepted equals the
box's closed form 1 - prod(1 - sum min(R_i, q)), a two-level tree under a bigram target
emits the target's joint law, a path-shaped tree is the chain rule, and a one-hot target
is the greedy walk.
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


def one_node_first_token_law(p, q, k):
    """Law of the first emitted token and P(some child accepted) at a root with k children
    drafted i.i.d. from q (leaf children; their own rows are uniform)."""
    V = len(p)
    parents = [-1] * k
    logits = np.vstack([_log(p)] + [np.zeros(V)] * k)
    qrows = np.vstack([q] + [np.full(V, 1.0 / V)] * k)
    first = np.zeros(V)
    acc = 0.0
    for toks in itertools.product(range(V), repeat=k):
        w = float(np.prod([q[t] for t in toks]))
        if w == 0.0:
            continue

        def verify(u, toks=toks):
            r = so.verify_tree_rr_sequence(logits, qrows, list(toks), parents, 1.0, u, 2)
            assert r["status"] & so.STATUS_ERROR_MASK == 0
            return _emitted(r)

        for out, m in tree_rr_outcome_law(verify, parents).items():
            first[out[0]] += w * m
            if len(out) >= 2:
                acc += w * m
    return first, acc


def page_acceptance(p, q, k):
    """The box's closed form: 1 - prod_{i<=k} (1 - sum_x min(R_i(x), q(x))), R_1 = p,
    R_{i+1} = (R_i - q)+ normalised."""
    R = np.asarray(p, dtype=np.float64)
    keep = 1.0
    for _ in range(k):
        keep *= 1.0 - np.minimum(R, q).sum()
        r = np.maximum(R - q, 0.0)
        if r.sum() <= 0.0:
            break
        R = r / r.sum()
    return 1.0 - keep


@pytest.mark.parametrize("k", [1, 2, 3])
@pytest.mark.parametrize("seed", [0, 1])
def test_one_node_output_is_p_and_acceptance_is_the_closed_form(k, seed):
    rng = np.random.default_rng(seed)
    V = 4
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V) * 0.8)
    first, acc = one_node_first_token_law(p, q, k)
    np.testing.assert_allclose(first, p, atol=1e-12)
    assert acc == pytest.approx(page_acceptance(p, q, k), abs=1e-12)


def test_acceptance_grows_with_children():
    """More i.i.d. children never lower the chance that one is accepted."""
    rng = np.random.default_rng(5)
    p = rng.dirichlet(np.ones(4))
    q = rng.dirichlet(np.ones(4))
    accs = [one_node_first_token_law(p, q, k)[1] for k in (1, 2, 3)]
    assert accs[0] <= accs[1] + 1e-12 <= accs[2] + 2e-12
    assert accs[0] == pytest.approx(1.0 - so.total_variation(p, q), abs=1e-12)


def _two_level_round_law(P, Q, state):
    """Exact law of one round's emitted tokens from `state`: root children 0 and 1 drafted
    from Q[state], node 2 a child of node 0 drafted from Q[token of node 0]."""
    V = P.shape[0]
    parents = [-1, -1, 0]
    law = {}
    for t0, t1, t2 in itertools.product(range(V), repeat=3):
        w = Q[state][t0] * Q[state][t1] * Q[t0][t2]
        if w == 0.0:
            continue
        toks = [t0, t1, t2]
        logits = np.vstack([_log(P[state])] + [_log(P[t]) for t in toks])
        qrows = np.vstack([Q[state]] + [Q[t] for t in toks])

        def verify(u, toks=toks, logits=logits, qrows=qrows):
            r = so.verify_tree_rr_sequence(logits, qrows, toks, parents, 1.0, u, 2)
            assert r["status"] & so.STATUS_ERROR_MASK == 0
            return _emitted(r)

        for out, m in tree_rr_outcome_law(verify, parents).items():
            law[out] = law.get(out, 0.0) + w * m
    return law


@pytest.mark.parametrize("seed", [0, 1])
def test_two_level_tree_emits_the_target_joint_law(seed):
    """Lossless over a whole tree: the first two generated tokens follow P[start][a] *
    P[a][b] (a round that emits one token is followed by the next round)."""
    rng = np.random.default_rng(10 + seed)
    V = 3
    P = rng.dirichlet(np.ones(V), size=V)
    Q = rng.dirichlet(np.ones(V) * 0.7, size=V)
    start = 2
    joint = np.zeros((V, V))
    cache = {}
    for out, m in _two_level_round_law(P, Q, start).items():
        if len(out) >= 2:
            joint[out[0], out[1]] += m
        else:
            y = out[0]
            if y not in cache:
                cache[y] = _two_level_round_law(P, Q, y)
            for out2, m2 in cache[y].items():
                joint[y, out2[0]] += m * m2
    np.testing.assert_allclose(joint, P[start][:, None] * P, atol=1e-12)


def test_path_shaped_tree_is_the_chain_rule():
    """One child per node: recursive rejection is the chain rule, uniform for uniform
    (tree u[1+i] is the chain's u[i], tree u[0] the chain's extra-token uniform)."""
    rng = np.random.default_rng(3)
    V, gamma = 50, 5
    for _ in range(40):
        logits = rng.standard_normal((gamma + 1, V)) * 2.0
        q = rng.dirichlet(np.ones(V), size=gamma + 1)
        drafts = [int(rng.integers(V)) for _ in range(gamma)]
        u = rng.random(gamma + 1)
        T = float(rng.uniform(0.3, 1.5))
        chain = so.verify_chain_sequence(logits, q[:gamma], drafts, T, u)
        tu = np.concatenate([[u[gamma]], u[:gamma]])
        tree = so.verify_tree_rr_sequence(logits, q, drafts, list(range(-1, gamma - 1)), T, tu, gamma)
        assert tree["n_accepted"] == chain["J"]
        np.testing.assert_array_equal(tree["tokens"], chain["tokens"])
        assert tree["status"] == chain["status"]


def test_one_hot_target_is_the_greedy_walk():
    rng = np.random.default_rng(4)
    V = 6
    parents = [-1, -1, -1, 0, 0, 3, 1]
    N = len(parents)
    for _ in range(30):
        logits = rng.standard_normal((N + 1, V))
        z = logits.argmax(axis=1)
        toks = [int(z[0 if a < 0 else 1 + a]) if rng.random() < 0.5 else int(rng.integers(V)) for a in parents]
        hot = np.full((N + 1, V), -np.inf)
        hot[np.arange(N + 1), z] = 0.0
        q = rng.dirichlet(np.ones(V), size=N + 1)
        u = rng.random(N + 1)
        sampled = so.verify_tree_rr_sequence(hot, q, toks, parents, 1.0, u, 4)
        greedy = so.verify_tree_rr_sequence(logits, q, toks, parents, 0.0, u, 4)
        walk = so.verify_tree_sequence(logits, toks, parents, 0.0, u, 4)
        np.testing.assert_array_equal(sampled["tokens"], greedy["tokens"])
        np.testing.assert_array_equal(greedy["tokens"], walk["tokens"])
        np.testing.assert_array_equal(greedy["path"], walk["path"])


def test_status_follows_the_walk():
    V = 8
    parents = [-1, -1, 0]
    logits = np.zeros((4, V))
    logits[0, 3] = 5.0  # the root target prefers token 3
    q = np.full((4, V), 1.0 / V)
    u = np.full(4, 0.5)
    ok = so.verify_tree_rr_sequence(logits, q, [3, 1, 2], parents, 1.0, u, 3)
    assert ok["status"] == 0 and ok["path"][0] == 0
    # node 1 is never tried when node 0 is accepted, so a bad q elsewhere in the root
    # row is not read
    qb = q.copy(); qb[0, 6] = np.nan
    assert so.verify_tree_rr_sequence(logits, qb, [3, 1, 2], parents, 1.0, u, 3)["status"] == 0
    # after a rejection the residual reads the whole row
    r = so.verify_tree_rr_sequence(logits, qb, [5, 1, 2], parents, 1.0, np.full(4, 0.99), 3)
    assert r["status"] & so.STATUS_BAD_PROB and r["n_accepted"] == -1
    assert so.verify_tree_rr_sequence(logits, q, [3, 9, 2], parents, 1.0, u, 3)["status"] & so.STATUS_BAD_TOKEN
    assert so.verify_tree_rr_sequence(logits, q, [3, 1, 2], [-1, 5, 0], 1.0, u, 3)["status"] & so.STATUS_BAD_TREE
    assert so.verify_tree_rr_sequence(logits, q, [3, 1, 2], parents, 1.0, u, 1)["status"] & so.STATUS_BAD_TREE
    ub = u.copy(); ub[2] = 1.0
    assert so.verify_tree_rr_sequence(logits, q, [3, 1, 2], parents, 1.0, ub, 3)["status"] & so.STATUS_BAD_UNIFORM
    assert so.verify_tree_rr_sequence(logits, q, [3, 1, 2], parents, np.inf, u, 3)["status"] == so.STATUS_BAD_TEMPERATURE
    lb = logits.copy(); lb[1, 2] = np.nan  # node 0's row, visited after its acceptance
    assert so.verify_tree_rr_sequence(lb, q, [3, 1, 2], parents, 1.0, u, 3)["status"] & so.STATUS_BAD_LOGIT
