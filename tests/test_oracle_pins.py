"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against a value printed on the pages (cited fixtures under
tests/golden/), a closed form, an identity, a library routine in a special case, or an
exact integration of its own output over the uniforms (tests/exact_integration.py).
"""
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import specdec_oracle as so
from exact_integration import (bigram_round_law, first_two_tokens_law, round_outcome_law,
                               step_function_masses)
from golden import read_fixture


def _f(xs):
    return np.array([float(x) for x in xs])


def oracle_rows(p_rows, q_rows, drafts, u):
    """Adapter: probabilities -> logits log p at T = 1, emitted tokens as a tuple."""
    with np.errstate(divide="ignore"):
        logits = np.log(np.asarray(p_rows, dtype=np.float64))
    r = so.verify_chain_sequence(logits, np.asarray(q_rows), drafts, 1.0, u)
    assert r["status"] & so.STATUS_ERROR_MASK == 0, r["status"]
    t = r["tokens"]
    return tuple(int(x) for x in t[t >= 0])


# ------------------------------------------------------------------ worked example

def test_worked_example_three_tokens():
    fx = read_fixture("worked_example_3token.txt")
    p, q = _f(fx["p"]), _f(fx["q"])
    assert so.acceptance_rate(p, q) == pytest.approx(float(fx["acceptance"][0]), abs=1e-15)
    assert so.total_variation(p, q) == pytest.approx(float(fx["total_variation"][0]), abs=1e-15)
    r = so.residual_distribution(p, q)
    assert np.allclose(r / r.sum(), _f(fx["residual_normalised"]), atol=1e-15)
    # naive rule's agreement sum_x p q, as a check on the example's numbers
    assert float((p * q).sum()) == pytest.approx(float(fx["naive_agreement"][0]), abs=1e-15)

    # keep probabilities, measured on the oracle: accept threshold in u for each draft
    for x, keep in enumerate(_f(fx["keep_probability"])):
        def accepted(uu, x=x):
            return len(oracle_rows(np.stack([p, p]), q[None], [x], [uu, 0.5])) > 1
        t = step_function_masses(accepted).get(True, 0.0)
        assert t == pytest.approx(keep, abs=1e-14)

    # exact law of the emitted token of a gamma = 1 round: output == p
    law = np.zeros(3)
    for x in range(3):
        sub = round_outcome_law(lambda d, u: oracle_rows(np.stack([p, p]), q[None], d, u), [x], 1)
        for out, m in sub.items():
            law[out[0]] += q[x] * m
    assert np.allclose(law, _f(fx["output"]), atol=1e-13)


# ------------------------------------------------------------------ exactness, bigram

def _bigram(V, seed, noise):
    rng = np.random.default_rng(seed)
    P = rng.dirichlet(np.ones(V) * 0.7, size=V)
    Q = np.abs(P + noise * rng.standard_normal((V, V)))
    Q /= Q.sum(1, keepdims=True)
    return P, Q


@pytest.mark.parametrize("gamma", [1, 2, 3])
def test_first_token_law_equals_target_exactly(gamma):
    """SD 20.5, "Proof that a whole round is exact": the first token is ~ p(.|state)."""
    P, Q = _bigram(3, 7 + gamma, 0.2)
    law = bigram_round_law(oracle_rows, P, Q, 0, gamma)
    first = np.zeros(3)
    for out, m in law.items():
        first[out[0]] += m
    assert np.allclose(first, P[0], atol=1e-12)
    assert sum(law.values()) == pytest.approx(1.0, abs=1e-12)


def test_two_token_joint_equals_target_exactly():
    """The bigram experiment of SD 20.5 ("A broken sampler looks healthy on a speed
    dashboard") made exact: joint law of the first two tokens equals P(y1|0) P(y2|y1)."""
    P, Q = _bigram(4, 3, 0.25)
    joint = first_two_tokens_law(oracle_rows, P, Q, 0, 2)
    assert np.allclose(joint, P[0][:, None] * P, atol=1e-12)


def test_resample_from_p_bug_is_detected(monkeypatch):
    """SD 20.5, "Four ways to lose exactness": resampling from p after a rejection."""
    P, Q = _bigram(4, 3, 0.25)
    monkeypatch.setattr(so, "residual_distribution", lambda p, q: so.widen(p))
    joint = first_two_tokens_law(oracle_rows, P, Q, 0, 2)
    assert np.abs(joint - P[0][:, None] * P).sum() > 1e-2


def test_topk_acceptance_bug_is_detected(monkeypatch):
    """SD 20.5, "Four ways to lose exactness": accepting whenever the target ranks the
    draft in its top few is a different (lossy) sampler."""
    P, Q = _bigram(4, 3, 0.25)
    real = so.verify_chain_sequence

    def lossy(logits, q, drafts, T, u, want_cdf=False):
        top2 = [set(np.argsort(-np.asarray(l))[:2].tolist()) for l in logits]
        J = 0
        while J < len(drafts) and drafts[J] in top2[J]:
            J += 1
        if J == len(drafts):
            return real(logits, q, drafts, T, u, want_cdf)
        r = real(logits[J:], q[J:], drafts[J:], T, u[J:], want_cdf)
        r["tokens"] = np.concatenate([np.asarray(drafts[:J]), r["tokens"][: len(drafts) + 1 - J]])
        return r

    monkeypatch.setattr(so, "verify_chain_sequence", lossy)
    joint = first_two_tokens_law(oracle_rows, P, Q, 0, 2)
    assert np.abs(joint - P[0][:, None] * P).sum() > 1e-2


def test_wrong_q_bug_is_detected():
    """SD 20.5, "Four ways to lose exactness": using a q other than the one sampled."""
    P, Q = _bigram(3, 11, 0.3)
    Qwrong = np.roll(Q, 1, axis=1)
    law = np.zeros(3)
    for x in range(3):
        sub = round_outcome_law(
            lambda d, u: oracle_rows(np.stack([P[0], P[d[0]]]), Qwrong[0][None], d, u), [x], 1)
        for out, m in sub.items():
            law[out[0]] += Q[0][x] * m
    assert np.abs(law - P[0]).sum() > 1e-2


# ------------------------------------------------------------------ acceptance identities

def test_acceptance_is_one_minus_tv_and_matches_measured_acceptance():
    rng = np.random.default_rng(0)
    for _ in range(20):
        V = int(rng.integers(2, 7))
        p, q = rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V))
        a = so.acceptance_rate(p, q)
        assert a == pytest.approx(1.0 - so.total_variation(p, q), abs=1e-14)
        # measured on the verifier: P(J >= 1) integrated exactly over drafts and u
        meas = 0.0
        for x in range(V):
            sub = round_outcome_law(lambda d, u: oracle_rows(np.stack([p, p]), q[None], d, u), [x], 1)
            meas += q[x] * sum(m for out, m in sub.items() if len(out) == 2)
        assert meas == pytest.approx(a, abs=1e-12)


def _iid_J_law(p, q, gamma):
    """Exact law of J when every position has the same (p, q), measured on the oracle."""
    law = np.zeros(gamma + 1)
    V = len(p)
    rows_p = np.stack([p] * (gamma + 1))
    rows_q = np.stack([q] * gamma)
    import itertools
    for drafts in itertools.product(range(V), repeat=gamma):
        w = float(np.prod([q[x] for x in drafts]))
        if w == 0:
            continue
        sub = round_outcome_law(lambda d, u: oracle_rows(rows_p, rows_q, d, u), list(drafts), gamma)
        for out, m in sub.items():
            law[len(out) - 1] += w * m
    return law


def test_closed_forms_printed_on_pages():
    """Expected tokens per round: the pages' printed values, via the oracle's exact law
    of J with a deterministic draft accepted with probability alpha (SD 20.5,
    "A deterministic draft": q one-hot, accepted with probability p(x))."""
    fx = read_fixture("closed_forms.txt")
    for alpha, gamma, printed, dec in fx["case"]:
        alpha, gamma, printed, dec = float(alpha), int(gamma), float(printed), int(dec)
        p = np.array([alpha, 1 - alpha])
        q = np.array([1.0, 0.0])
        law = _iid_J_law(p, q, gamma)
        mean = float((np.arange(gamma + 1) + 1) @ law)
        assert round(mean, dec) == pytest.approx(printed, abs=1e-12)
        assert round(so.expected_tokens_iid(alpha, gamma), dec) == pytest.approx(printed, abs=1e-12)
        # capped geometric law of J (SD 20.5, "Expected tokens per round")
        for i in range(gamma):
            assert law[i] == pytest.approx(alpha ** i * (1 - alpha), abs=1e-12)
        assert law[gamma] == pytest.approx(alpha ** gamma, abs=1e-12)


def test_iid_law_with_spread_distributions():
    """Same closed form with a non-degenerate q (alpha = 0.7 of the worked example)."""
    p = np.array([0.5, 0.3, 0.2])
    q = np.array([0.2, 0.6, 0.2])
    law = _iid_J_law(p, q, 3)
    mean = float((np.arange(4) + 1) @ law)
    assert mean == pytest.approx((1 - 0.7 ** 4) / 0.3, abs=1e-12)


def test_block_verify_toy_tokenwise_value():
    """Art of Guessing, "Block verification": token-wise verification of the toy
    accepts 10/9 tokens per round on average (the page's printed value)."""
    fx = read_fixture("block_verify_toy.txt")
    p, q, gamma = _f(fx["p"]), _f(fx["q"]), int(fx["gamma"][0])
    law = _iid_J_law(p, q, gamma)
    assert float(np.arange(gamma + 1) @ law) == pytest.approx(float(fx["tokenwise_accepted"][0]), abs=1e-12)


# ------------------------------------------------------------------ greedy

def test_greedy_speculation_reproduces_greedy_decoding():
    """SD 20.5, "Greedy speculation keeps the target's own choices" and the exercise
    "Greedy speculative generation, with call counting"."""
    rng = np.random.default_rng(5)
    V, gamma, n_new = 12, 4, 40
    target = rng.standard_normal((V, V)) * 2
    draft = target + rng.standard_normal((V, V)) * 1.5
    # plain greedy decoding with numpy argmax
    plain = [3]
    for _ in range(n_new):
        plain.append(int(np.argmax(target[plain[-1]])))
    toks, calls = [3], 0
    while len(toks) < n_new + 1:
        drafts, s = [], toks[-1]
        for _ in range(gamma):
            s = int(np.argmax(draft[s]))
            drafts.append(s)
        rows = np.stack([target[t] for t in [toks[-1]] + drafts])
        r = so.verify_greedy_sequence(rows, drafts)
        calls += 1
        emitted = r["tokens"][: r["J"] + 1]
        toks.extend(int(t) for t in emitted)
    assert toks[: n_new + 1] == plain
    assert calls < n_new


def test_lowest_index_argmax_ties():
    assert so.lowest_argmax([1.0, 3.0, 3.0, 2.0]) == 1
    assert so.lowest_argmax([-np.inf, -np.inf, 0.0, 0.0]) == 2
    rng = np.random.default_rng(1)
    for _ in range(50):
        l = rng.integers(0, 4, size=9).astype(np.float64)
        assert so.lowest_argmax(l) == int(np.argmax(l))  # numpy returns the first maximum


def test_greedy_rows_ignore_q_and_u():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((4, 10))
    drafts = [int(np.argmax(logits[0])), int(np.argmax(logits[1])), 0]
    r1 = so.verify_chain_sequence(logits, rng.random((3, 10)), drafts, 0.0, rng.random(4))
    r2 = so.verify_chain_sequence(logits, None, drafts, 5e-4, np.zeros(4))
    assert np.array_equal(r1["tokens"], r2["tokens"]) and r1["J"] == r2["J"] >= 2


# ------------------------------------------------------------------ library special cases

def test_target_distribution_is_softmax_at_temperature():
    rng = np.random.default_rng(3)
    for T in [0.25, 0.8, 1.0, 1.7]:
        l = rng.standard_normal(50) * 3
        assert np.allclose(so.target_distribution(l, T), scipy.special.softmax(l / T), atol=1e-15)
    l = np.array([0.0, -np.inf, 1.0])
    p = so.target_distribution(l, 1.0)
    assert p[1] == 0.0 and p.sum() == pytest.approx(1.0)


def test_inverse_cdf_matches_searchsorted_and_skips_zero_weights():
    rng = np.random.default_rng(4)
    for _ in range(200):
        w = rng.random(9) * (rng.random(9) < 0.6)
        if w.sum() == 0:
            continue
        u = rng.random()
        k, C, S = so.inverse_cdf(w, u)
        assert k == int(np.searchsorted(np.cumsum(w), u * w.sum(), side="right"))
        assert w[k] > 0


def test_bonus_token_when_all_accepted_is_drawn_from_last_row():
    """When every draft is accepted, the extra token comes from p_{gamma+1}."""
    p0 = np.array([0.0, 1.0, 0.0])          # draft 1 always accepted
    p1 = np.array([0.2, 0.3, 0.5])
    q = np.array([[0.0, 1.0, 0.0]])
    law = round_outcome_law(lambda d, u: oracle_rows(np.stack([p0, p1]), q, d, u), [1], 1)
    bonus = np.zeros(3)
    for out, m in law.items():
        assert out[0] == 1 and len(out) == 2
        bonus[out[1]] += m
    assert np.allclose(bonus, p1, atol=1e-14)


# ------------------------------------------------------------------ status / degenerate

def test_status_flags_and_degenerate_cases():
    l = np.zeros((2, 4))
    q = np.full((1, 4), 0.25)
    r = so.verify_chain_sequence(np.where(np.eye(2, 4) > 0, np.nan, l), q, [0], 1.0, [0.1, 0.1])
    assert r["status"] & so.STATUS_BAD_LOGIT and r["J"] == -1 and (r["tokens"] == -1).all()
    r = so.verify_chain_sequence(np.full((2, 4), -np.inf), q, [0], 1.0, [0.1, 0.1])
    assert r["status"] & so.STATUS_EMPTY_ROW
    r = so.verify_chain_sequence(l, q, [4], 1.0, [0.1, 0.1])
    assert r["status"] & so.STATUS_BAD_TOKEN
    r = so.verify_chain_sequence(l, q, [1], 1.0, [1.0, 0.1])
    assert r["status"] & so.STATUS_BAD_UNIFORM
    r = so.verify_chain_sequence(l, -q, [1], 1.0, [0.5, 0.1])
    assert r["status"] & so.STATUS_BAD_PROB
    # q(x) = 0: warning, accepted because p(x) > 0
    q0 = np.array([[0.0, 0.5, 0.5, 0.0]])
    r = so.verify_chain_sequence(l, q0, [0], 1.0, [0.99, 0.1])
    assert r["status"] == so.STATUS_ZERO_Q and r["J"] == 1
    # p == q exactly: always accepted (SD 20.5: "When p = q every draft is accepted")
    r = so.verify_chain_sequence(l, q, [2], 1.0, [np.nextafter(1.0, 0.0), 0.3])
    assert r["J"] == 1 and r["status"] == 0


def test_positions_after_the_first_rejection_are_not_evaluated():
    """SD 20.5, "A whole round of speculative sampling": drafts are tested in order and
    the round ends at the first rejected one, so later positions are never examined."""
    l = np.array([[0.0, 0.0], [np.nan, 0.0], [0.0, 0.0]])
    q = np.array([[1.0, 0.0], [0.5, 0.5]])
    r = so.verify_chain_sequence(l, q, [0, 99], 1.0, [0.9, 0.5, 0.25])
    assert r["status"] == 0 and r["J"] == 0 and r["tokens"][0] == 1
    assert r["p_draft"][0] == pytest.approx(0.5) and np.isnan(r["p_draft"][1])
    r = so.verify_chain_sequence(l, q, [0, 99], 1.0, [0.1, 0.5, 0.25])
    assert r["status"] == so.STATUS_BAD_LOGIT and r["J"] == -1 and np.isnan(r["p_draft"]).all()
    # greedy: position 0 rejected (argmax is token 0 on ties), row 1 never read
    r = so.verify_chain_sequence(l, None, [1, 99], 0.0, np.zeros(3))
    assert r["status"] == 0 and r["J"] == 0 and list(r["tokens"]) == [0, -1, -1]


def test_zero_residual_falls_back_to_p():
    # p slightly below q at the draft so it can be rejected, yet (p - q)+ == 0
    # everywhere is impossible in exact arithmetic; force it through q >= p elementwise.
    l = np.log(np.array([[0.5, 0.5], [0.5, 0.5]]))
    q = np.array([[0.5, 0.6]])
    r = so.verify_chain_sequence(l, q, [1], 1.0, [0.95, 0.3])
    assert r["J"] == 0 and r["status"] == so.STATUS_ZERO_RESIDUAL
    assert r["tokens"][0] == 0  # inverse CDF of p = (0.5, 0.5) at u = 0.3


# ------------------------------------------------------------------ trees

def test_tree_mask_worked_example():
    fx = read_fixture("tree_mask_6node.txt")
    parents = [int(x) for x in fx["parents"]]
    block = np.array([[int(x) for x in row] for row in fx["mask_row"]], dtype=bool)
    P = 5
    mask, pos, depth = so.build_tree_mask(parents, P)
    assert mask.shape == (6, P + 6)
    assert mask[:, :P].all()
    assert np.array_equal(mask[:, P:], block)
    assert list(depth) == [int(x) for x in fx["depth"]]
    assert list(pos) == [P + int(x) for x in fx["depth"]]


def test_chain_tree_gives_causal_mask():
    """SD 20.5: a chain par(i) = i - 1 gives the bottom-right causal mask."""
    n, P = 7, 3
    mask, pos, _ = so.build_tree_mask(list(range(-1, n - 1)), P)
    assert np.array_equal(mask, np.tril(np.ones((n, P + n), dtype=bool), k=P))
    assert list(pos) == list(range(P, P + n))


def test_bad_parents_rejected():
    with pytest.raises(ValueError):
        so.tree_depths([-1, 1])
    with pytest.raises(ValueError):
        so.tree_depths([-2])


def test_medusa_cartesian_counts():
    fx = read_fixture("medusa_counts.txt")
    tops = [int(x) for x in fx["tops"]]
    nodes, paths = so.cartesian_tree_counts(tops)
    assert nodes == int(fx["tokens"][0]) and paths == int(fx["paths"][0])
    # the greedy builder with an unlimited budget returns the full product tree
    acc = [[Fraction(1, 2 + i + k) for i in range(8)] for k in range(4)]
    parents, paths_, _ = so.medusa_sparse_tree(acc, 10 ** 6)
    assert len(parents) == int(fx["tokens"][0])
    n_children = np.bincount([p for p in parents if p >= 0], minlength=len(parents))
    assert int((n_children == 0).sum()) == int(fx["paths"][0])


def test_medusa_sparse_tree_is_greedy_optimal_and_closed():
    acc = [[f"{0.6 * 0.75 ** (i - 1) * 0.85 ** (k - 1):.12g}" for i in range(1, 11)] for k in range(1, 5)]
    acc_exact = [[Fraction(3, 5) * Fraction(3, 4) ** (i - 1) * Fraction(17, 20) ** (k - 1)
                  for i in range(1, 11)] for k in range(1, 5)]
    parents, paths, values = so.medusa_sparse_tree(acc_exact, 64)
    assert len(parents) == 64
    assert all(-1 <= a < i for i, a in enumerate(parents))
    # every node outside the tree is worth no more than every node inside it
    import itertools
    chosen = set(paths)
    vmin = min(values)
    for m in range(1, 5):
        for path in itertools.product(range(10), repeat=m):
            if path not in chosen:
                v = Fraction(1)
                for j, r in enumerate(path):
                    v *= acc_exact[j][r]
                assert v <= vmin
    # E[L] of the full product tree factorises: sum_m prod_{j<=m} sum_i a_j^(i)
    small = [[Fraction(1, 3), Fraction(1, 5)], [Fraction(1, 4), Fraction(1, 7)]]
    _, _, vals = so.medusa_sparse_tree(small, 10)
    s1, s2 = sum(small[0]), sum(small[1])
    assert so.medusa_expected_length(vals) == s1 + s1 * s2
    assert acc  # decimal-string accuracies parse as well
    assert len(so.medusa_sparse_tree(acc, 64)[0]) == 64


def _brute_force_greedy_walk(logits, node_tokens, parents):
    """Longest root path whose every token equals the argmax of its parent's row
    (enumerating every node's root path)."""
    n = len(parents)
    best = []
    for i in range(n):
        path, a = [], i
        while a != -1:
            path.append(a)
            a = parents[a]
        path = path[::-1]
        ok, row = True, 0
        for node in path:
            z = int(np.argmax(logits[row]))
            # READING: equal-token siblings resolve to the lowest node index
            first = min(j for j in range(n) if parents[j] == parents[node] and node_tokens[j] == node_tokens[node])
            if node_tokens[node] != z or node != first:
                ok = False
                break
            row = 1 + node
        if ok and len(path) > len(best):
            best = path
    return best


def test_greedy_tree_walk_matches_brute_force():
    rng = np.random.default_rng(9)
    fx_parents = [-1, -1, 0, 0, 1, 2, 2, 5]
    n, V = len(fx_parents), 5
    for _ in range(200):
        logits = rng.integers(0, 3, size=(n + 1, V)).astype(np.float64) + rng.random((n + 1, V)) * 0.5
        toks = rng.integers(0, V, size=n)
        r = so.verify_tree_sequence(logits, toks, fx_parents, 0.0, np.zeros(5), 4)
        best = _brute_force_greedy_walk(logits, toks, fx_parents)
        assert r["n_accepted"] == len(best)
        assert list(r["path"][: len(best)]) == best
        last_row = 0 if not best else 1 + best[-1]
        assert r["tokens"][len(best)] == int(np.argmax(logits[last_row]))


def test_sampled_tree_walk_emits_target_samples():
    """Every emitted token of the walk is a target sample (Medusa notes, "Attention
    Tree"): the first token's law is p_root, integrated exactly over u_0."""
    rng = np.random.default_rng(10)
    parents = [-1, -1, 0, 1]
    V = 4
    logits = rng.standard_normal((5, V))
    toks = [2, 1, 3, 0]
    T = 0.7

    def first(u0):
        return int(so.verify_tree_sequence(logits, toks, parents, T, [u0, 0.5, 0.5], 2)["tokens"][0])

    law = step_function_masses(first)
    p_root = scipy.special.softmax(logits[0] / T)
    for k in range(V):
        assert law.get(k, 0.0) == pytest.approx(p_root[k], abs=1e-13)

    # second token after descending into node 0 (token 2) follows the row of node 0
    def second(u1):
        u0 = 0.5 * (p_root[:2].sum() + p_root[:3].sum())  # inside token 2's interval
        return int(so.verify_tree_sequence(logits, toks, parents, T, [u0, u1, 0.5], 2)["tokens"][1])

    law2 = step_function_masses(second)
    p_node0 = scipy.special.softmax(logits[1] / T)
    for k in range(V):
        assert law2.get(k, 0.0) == pytest.approx(p_node0[k], abs=1e-13)


def test_tree_status():
    logits = np.zeros((3, 4))
    r = so.verify_tree_sequence(logits, [1, 2], [-1, 1], 0.0, np.zeros(3), 2)
    assert r["status"] & so.STATUS_BAD_TREE
    r = so.verify_tree_sequence(logits, [1, 9], [-1, 0], 0.0, np.zeros(3), 2)
    assert r["status"] & so.STATUS_BAD_TOKEN
    r = so.verify_tree_sequence(logits, [1, 2], [-1, 0], 0.0, np.zeros(2), 1)
    assert r["status"] & so.STATUS_BAD_TREE  # depth 2 exceeds max_depth 1


def test_public_namespace():
    assert oracle.GREEDY_T == 1e-3
    assert oracle.STATUS_ERROR_MASK & oracle.STATUS_ZERO_Q == 0
