"""Exact integration of a verifier's output distribution over its uniforms.

The verifier is treated as a black box f(drafts, u) -> emitted tokens.  For fixed
drafts, its output is piecewise constant in each uniform: the acceptance test of
position i is a threshold in u_i, and the extra-token draw is a non-decreasing step
function of u_gamma.  The breakpoints are located by bisection on the verifier itself
(to float64 resolution), so the probability of every outcome is a product of interval
lengths -- no formula of the method is restated here.  This is how the oracle's output
law is pinned to the target distribution exactly (SD 20.5, "The speculative sampling
rule": the emitted token is distributed exactly as p whatever q is).
"""
from __future__ import annotations

from collections import defaultdict
import itertools

import numpy as np

_BISECT_STEPS = 64


def _last_u_with(fn, lo: float, value) -> float:
    """Smallest b > lo such that fn(u) != value for u just at/after b (fn constant on [lo, b)).

    fn must be piecewise constant and, on [lo, 1), equal to value on an interval
    starting at lo.  Returns 1.0 if fn stays equal up to 1.
    """
    top = np.nextafter(1.0, 0.0)
    if fn(top) == value:
        return 1.0
    a, b = lo, top
    for _ in range(_BISECT_STEPS):
        mid = 0.5 * (a + b)
        if mid <= a or mid >= b:
            break
        if fn(mid) == value:
            a = mid
        else:
            b = mid
    return b


def step_function_masses(fn) -> dict:
    """Masses of the values of a left-to-right step function of one uniform on [0, 1)."""
    out = defaultdict(float)
    lo = 0.0
    while lo < 1.0:
        v = fn(lo)
        hi = _last_u_with(fn, lo, v)
        out[v] += hi - lo
        lo = hi
    return dict(out)


def round_outcome_law(verify, drafts, gamma: int) -> dict:
    """Law of the emitted token tuple of one verification round with fixed drafts.

    verify(drafts, u) -> tuple of emitted tokens (u has gamma + 1 entries: u[i] decides
    position i, u[gamma] drives the extra token).  The recursion walks the accept
    thresholds position by position, holding the already-decided uniforms at interior
    points of their intervals, then integrates the final draw over u[gamma].
    """
    law = defaultdict(float)

    def n_emitted_accepts(u):
        return len(verify(drafts, u)) - 1

    def recurse(prefix_u, weight):
        i = len(prefix_u)
        if i == gamma:
            def tok(x):
                return verify(drafts, list(prefix_u) + [x])
            for out, m in step_function_masses(tok).items():
                law[out] += weight * m
            return

        def accepted_here(x):
            u = list(prefix_u) + [x] + [0.5] * (gamma - i)
            return n_emitted_accepts(u) > i

        # acceptance is a threshold: accept on [0, t), reject on [t, 1)
        if accepted_here(0.0):
            t = _last_u_with(accepted_here, 0.0, True)
        else:
            t = 0.0
        if t > 0.0:
            recurse(prefix_u + [0.5 * t], weight * t)
        if t < 1.0:
            mid = 0.5 * (t + 1.0)
            # rejected at position i: the round ends; integrate the final draw
            def tok(x, mid=mid):
                u = list(prefix_u) + [mid] + [0.5] * (gamma - i - 1) + [x]
                return verify(drafts, u)
            for out, m in step_function_masses(tok).items():
                law[out] += weight * (1.0 - t) * m

    recurse([], 1.0)
    return dict(law)


def block_round_outcome_law(verify, drafts, gamma: int) -> dict:
    """Law of the emitted tuple of one block-verification round with fixed drafts.

    Structure assumed of the verifier (a wrong verifier then yields a wrong law, which
    the pins catch): prefix length k survives iff its own uniform u[k-1] lies below a
    threshold, the round keeps the longest surviving prefix, and the extra token is a
    step function of u[gamma].  Each threshold is located by bisection on the verifier
    with every other prefix's uniform near 1.
    """
    hi = np.nextafter(1.0, 0.0)

    def n_of(u):
        return len(verify(drafts, u)) - 1

    t = {}
    for k in range(1, gamma + 1):
        def survives(x, k=k):
            u = [hi] * gamma + [0.5]
            u[k - 1] = x
            return n_of(u) >= k
        t[k] = _last_u_with(survives, 0.0, True) if survives(0.0) else 0.0
    law = defaultdict(float)
    for n in range(gamma + 1):
        pn = t[n] if n >= 1 else 1.0
        for j in range(n + 1, gamma + 1):
            pn *= 1.0 - t[j]
        if pn <= 0.0:
            continue
        base = [0.5] * gamma
        if n >= 1:
            base[n - 1] = 0.5 * t[n]
        for j in range(n + 1, gamma + 1):
            base[j - 1] = 0.5 * (1.0 + t[j])

        def tok(x, base=base):
            return verify(drafts, base + [x])
        for out, m in step_function_masses(tok).items():
            law[out] += pn * m
    return dict(law)


def bigram_round_law(verify_rows, P, Q, state: int, gamma: int, round_law=None) -> dict:
    """Exact law of the tokens one round emits from `state` under bigram models.

    P[s], Q[s] are the target's and draft's next-token distributions after token s.
    Drafts are enumerated with their probabilities prod_i Q(x_i | x_{i-1}); each draft
    sequence's target rows p_i = P[x_{i-1}] (p_0 = P[state]) are passed to
    verify_rows(p_rows, q_rows, drafts, u) -> emitted tuple.
    """
    V = P.shape[0]
    law = defaultdict(float)
    for drafts in itertools.product(range(V), repeat=gamma):
        prev = [state] + list(drafts[:-1])
        w = 1.0
        for x, s in zip(drafts, prev):
            w *= Q[s][x]
        if w == 0.0:
            continue
        p_rows = np.stack([P[s] for s in [state] + list(drafts)])
        q_rows = np.stack([Q[s] for s in prev])

        def verify(d, u, p_rows=p_rows, q_rows=q_rows):
            return verify_rows(p_rows, q_rows, d, u)

        for out, m in (round_law or round_outcome_law)(verify, list(drafts), gamma).items():
            law[out] += w * m
    return dict(law)


def first_two_tokens_law(verify_rows, P, Q, start: int, gamma: int, round_law=None) -> np.ndarray:
    """Exact joint law of the first two generated tokens (several rounds if needed)."""
    V = P.shape[0]
    joint = np.zeros((V, V))
    first_round = bigram_round_law(verify_rows, P, Q, start, gamma, round_law)
    cache = {}
    for out, m in first_round.items():
        if len(out) >= 2:
            joint[out[0], out[1]] += m
        else:
            y1 = out[0]
            if y1 not in cache:
                cache[y1] = bigram_round_law(verify_rows, P, Q, y1, gamma, round_law)
            for out2, m2 in cache[y1].items():
                joint[y1, out2[0]] += m * m2
    return joint


def tree_rr_outcome_law(verify, parents) -> dict:
    """Law of the emitted token tuple of one tree round with fixed node tokens.

    verify(u) -> (emitted tokens, accepted path), both tuples; u has N + 1 entries: u[1+j]
    tests node j when the walk tries it, u[0] drives the final draw.  Structure assumed
    of the verifier (a wrong verifier then yields a wrong law, which the pins catch): at
    a node the children are tried in index order; child j is accepted on [0, t_j) of
    u[1+j] given the decisions before it, and the walk then continues below j; when every
    child is rejected the emitted token is a step function of u[0].  Each t_j is located
    by bisection on the verifier, with the decided uniforms held inside their intervals.
    """
    N = len(parents)
    law = defaultdict(float)

    def uniforms(fixed, slot=None, x=None):
        uu = [0.5] * (N + 1)
        for k, v in fixed.items():
            uu[k] = v
        if slot is not None:
            uu[slot] = x
        return uu

    def recurse(fixed, node, weight):
        fixed = dict(fixed)
        for j in [j for j in range(N) if parents[j] == node]:
            def accepted(x, j=j, fixed=dict(fixed)):
                return j in verify(uniforms(fixed, 1 + j, x))[1]
            t = _last_u_with(accepted, 0.0, True) if accepted(0.0) else 0.0
            if t > 0.0:
                recurse({**fixed, 1 + j: 0.5 * t}, j, weight * t)
            if t >= 1.0:
                return
            fixed[1 + j] = 0.5 * (1.0 + t)
            weight *= 1.0 - t

        def tok(x, fixed=fixed):
            return verify(uniforms(fixed, 0, x))[0]
        for out, m in step_function_masses(tok).items():
            law[out] += weight * m

    recurse({}, -1, 1.0)
    return dict(law)
