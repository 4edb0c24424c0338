"""Reference oracle for speculative-decoding verification -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 CPU statement of what the verification step computes.  Only the
test suite (``tests/``), ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import or call it.  The product path (the CUDA library and its
Python binding) never does, and this module imports nothing from the product.

Sources (cited by page title and section throughout):

* "Speculative decoding" (zerotofrontier.app, Chapter 20, Section 20.5) -- below "SD 20.5".
* "Speculative-Decoding / Medusa" (s1mplewind.github.io) -- below "Medusa notes".
* "Speculative Decoding: The Art of Guessing Well" (astralord.github.io) -- below "Art of Guessing".

Every floating-point input is widened exactly to float64 (bf16 and fp32 values are
exactly representable) and all arithmetic is float64.  Readings taken where the pages
are silent or disagree are marked READING.

Parity status: every public function here is pinned (``tests/test_oracle_*.py``: worked
examples, closed forms, identities, exact integration over the uniforms, and the Philox
generator's published known-answer vectors); none is "parity unpinned".
"""
from __future__ import annotations

from fractions import Fraction
import itertools

import numpy as np

# READING: a temperature below this threshold selects greedy (argmax) verification for
# that sequence; the pages treat tau = 0 as greedy decoding (SD 20.5, "Acceptance rate
# and temperature" exercise) and the workloads also use T < 1e-3.
GREEDY_T = 1e-3

# Per-sequence status bits.  These values are the interface documented for the
# library's status output; the oracle states them independently.
STATUS_BAD_LOGIT = 1        # a NaN or +inf logit in a row the verifier reads (error)
STATUS_EMPTY_ROW = 2        # a row with no finite logit, i.e. all -inf (error)
STATUS_BAD_TOKEN = 4        # a draft / node token outside [0, V) (error)
STATUS_BAD_PROB = 8         # a draft probability that is NaN, inf or negative (error)
STATUS_BAD_UNIFORM = 16     # a uniform outside [0, 1) on a sampled sequence (error)
STATUS_BAD_TREE = 32        # parent not in [-1, i) or a tree deeper than max_depth (error)
STATUS_BAD_TEMPERATURE = 64 # a NaN or infinite temperature (error)
STATUS_ZERO_Q = 256         # q_i(x_i) == 0 for a drafted token (warning)
STATUS_ZERO_RESIDUAL = 512  # residual mass was 0; the draw fell back to p (warning)
STATUS_ERROR_MASK = 0xFF


def widen(a) -> np.ndarray:
    """Exact widening of bf16 / fp32 / int inputs to float64."""
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------------------
# Distributions and their elementary statistics
# ---------------------------------------------------------------------------------------

def target_distribution(logits_row, T: float) -> np.ndarray:
    """p = softmax(l / T) over the vocabulary, in float64.

    SD 20.5, "When the target samples, keep a guess with probability p over q": p is the
    distribution the target really samples from, after temperature.  The maximum is
    subtracted first (a shift that leaves the softmax unchanged); a -inf logit gets
    probability exactly 0.
    """
    l = widen(logits_row)
    m = l.max()
    e = np.exp((l - m) / np.float64(T))
    return e / e.sum()


def lowest_argmax(logits_row) -> int:
    """Greedy choice z = argmax_x l(x), the smallest index among equal maxima.

    SD 20.5, "A round of greedy speculative decoding" (the target's own choice z_i).
    READING: ties resolve to the lowest token id.
    """
    l = widen(logits_row)
    return int(np.flatnonzero(l == l.max())[0])


def total_variation(p, q) -> float:
    """TV(p, q) = 1/2 sum_x |p(x) - q(x)|  (SD 20.5, "Acceptance rate and temperature")."""
    return 0.5 * float(np.abs(widen(p) - widen(q)).sum())


def acceptance_rate(p, q) -> float:
    """alpha = sum_x min(p(x), q(x)), the probability one draft is kept.

    SD 20.5, "The speculative sampling rule"; Art of Guessing, "Speculative sampling".
    """
    return float(np.minimum(widen(p), widen(q)).sum())


def residual_distribution(p, q) -> np.ndarray:
    """Unnormalised residual (p - q)+ (SD 20.5, "The speculative sampling rule")."""
    return np.maximum(0.0, widen(p) - widen(q))


def expected_tokens_iid(alpha: float, gamma: int) -> float:
    """E[J + 1] = (1 - alpha^(gamma+1)) / (1 - alpha) under i.i.d. acceptance.

    SD 20.5, "Expected tokens per round"; Art of Guessing, "How many tokens do we get?".
    """
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def inverse_cdf(weights, u: float):
    """Smallest k with C_k > u * S, C the running sum of the weights and S their total.

    The extra token of a round is one categorical draw (SD 20.5, "Verify one round of
    speculative sampling" uses one rng.choice); READING: the draw is the inverse CDF of
    the caller's uniform.  Zero-weight entries are never chosen.  If rounding leaves no
    qualifying k, the last entry with positive weight is taken.  Returns (k, C, S).
    """
    w = widen(weights)
    C = np.cumsum(w)
    S = C[-1]
    hits = np.flatnonzero(C > u * S)
    if hits.size:
        k = int(hits[0])
    else:
        k = int(np.flatnonzero(w > 0)[-1])
    return k, C, S


def _row_status(logits_row) -> int:
    l = widen(logits_row)
    if np.isnan(l).any() or np.isposinf(l).any():
        return STATUS_BAD_LOGIT
    if not np.isfinite(l).any():
        return STATUS_EMPTY_ROW
    return 0


# ---------------------------------------------------------------------------------------
# Chain verification (one round, one sequence)
# ---------------------------------------------------------------------------------------

def verify_chain_sequence(logits, q, drafts, T: float, u, want_cdf: bool = False) -> dict:
    """One round of speculative-sampling verification for one sequence.

    Follows SD 20.5, "A round of speculative sampling" (Leviathan et al. Alg. 1 /
    Chen et al. Alg. 2) and the exercise "Verify one round of speculative sampling",
    cross-read with Art of Guessing, "Speculative sampling" (the JAX verify):

      p_i = softmax(l_i / T) for i = 0..gamma        (rows are the target's distributions)
      accept draft i  iff  u_i < p_i(x_i) / q_i(x_i), evaluated as u_i * q_i(x_i) < p_i(x_i)
      J = number of leading accepted drafts
      extra token y ~ (p_J - q_J)+ normalised, with q_gamma == 0 (bonus from p_gamma)
      emit x_0 .. x_{J-1}, y

    The positions are evaluated in order and evaluation ends at the first rejected
    draft (SD 20.5, "A whole round of speculative sampling": the drafts are tested one
    after another and the round ends at the first one rejected, dropping the rest).  READING: only what is evaluated is validated -- row i, draft i,
    q_i(x_i) and u_i for i <= J, u_gamma and the q row of the draw -- and p_draft is NaN
    after J.

    A sequence with T < GREEDY_T is verified greedily (SD 20.5, "A round of greedy
    speculative decoding", and the special case "A greedy target" of the rule):
    accept while x_i == z_i = lowest argmax of row i, then emit z_J; q and u are unused.

    Arguments: logits [gamma+1, V]; q [gamma, V] (used as given, READING: no
    renormalisation); drafts [gamma] ints; T scalar; u [gamma+1] with u[i] the test
    uniform of position i and u[gamma] the uniform of the extra token (READING).

    Returns a dict: tokens [gamma+1] (-1 padded), J, status, p_draft [gamma] (p_i(x_i),
    NaN where unevaluated), q_draft [gamma], margins [gamma] (|u_i - p_i(x_i)/q_i(x_i)|,
    the distance of the test to its decision boundary), and for a sampled draw 'y_u'
    (u * S) plus, when want_cdf, 'cdf' and 'S' of the weights the draw used and 'pcdf',
    the CDF of p_J itself.
    """
    logits = np.asarray(logits)
    g1, V = logits.shape
    gamma = g1 - 1
    drafts = [int(x) for x in np.asarray(drafts).reshape(-1)]
    assert len(drafts) == gamma
    u = widen(u).reshape(-1)
    greedy = bool(T < GREEDY_T)   # READING: NaN is not >= the threshold; flagged below
    if np.isnan(T):
        greedy = True
    out = {
        "tokens": np.full(gamma + 1, -1, dtype=np.int64),
        "J": -1,
        "status": 0,
        "p_draft": np.full(gamma, np.nan),
        "q_draft": np.full(gamma, np.nan),
        "margins": np.full(gamma, np.inf),
        "greedy": greedy,
    }

    def error(bits):
        out["status"] = bits
        out["p_draft"][:] = np.nan
        return out

    status = 0
    if not np.isfinite(T):
        return error(STATUS_BAD_TEMPERATURE)

    # Checks of one position, in order: its logits row, then its draft token, then (when
    # sampled) its draft probability and uniform together; the first failing check ends
    # the round with that error.
    p = {}
    J = gamma
    for i in range(g1):
        rs = _row_status(logits[i])
        if rs:
            return error(status | rs)
        if i == gamma:
            break
        x = drafts[i]
        if not (0 <= x < V):
            return error(status | STATUS_BAD_TOKEN)
        if greedy:
            ok = x == lowest_argmax(logits[i])
        else:
            qx = float(widen(q[i][x]))
            bad = 0
            if not np.isfinite(qx) or qx < 0.0:
                bad |= STATUS_BAD_PROB
            if not (0.0 <= u[i] < 1.0):
                bad |= STATUS_BAD_UNIFORM
            if bad:
                return error(status | bad)
            p[i] = target_distribution(logits[i], T)
            px = p[i][x]
            out["p_draft"][i] = px
            out["q_draft"][i] = qx
            if qx == 0.0:
                # READING: a draft the drafter could not have produced; SD 20.5 notes the
                # ratio is then never needed.  Accept iff p(x) > 0 and warn.
                status |= STATUS_ZERO_Q
                ok = px > 0.0
            else:
                ok = u[i] * qx < px
                out["margins"][i] = abs(u[i] - px / qx)
        if not ok:
            J = i
            break

    if greedy:
        out["tokens"][:J] = drafts[:J]
        out["tokens"][J] = lowest_argmax(logits[J])
        out["J"] = J
        out["status"] = status
        return out

    if not (0.0 <= u[gamma] < 1.0):
        return error(status | STATUS_BAD_UNIFORM)
    if J not in p:
        p[J] = target_distribution(logits[J], T)
    if J < gamma:
        qJ = widen(q[J])
        if np.isnan(qJ).any() or np.isinf(qJ).any() or (qJ < 0).any():
            return error(status | STATUS_BAD_PROB)
        w = residual_distribution(p[J], qJ)
    else:
        # q_{gamma+1} == 0: the residual of the bonus row is p itself
        # (SD 20.5, "Speculative verification in PyTorch"; Art of Guessing, JAX verify).
        w = p[gamma].copy()
    if not (w.sum() > 0.0):
        # READING: possible only through rounding (p == q is always accepted); draw from p.
        status |= STATUS_ZERO_RESIDUAL
        w = p[J].copy()
    y, C, S = inverse_cdf(w, u[gamma])
    out["tokens"][:J] = drafts[:J]
    out["tokens"][J] = y
    out["J"] = J
    out["status"] = status
    out["y_u"] = u[gamma] * S
    if want_cdf:
        out["cdf"] = C
        out["S"] = S
        out["pcdf"] = np.cumsum(p[J])  # the target row's own CDF (the zero-residual fallback)
    return out


def verify_chain(logits, q, drafts, T, u) -> dict:
    """Batched chain verification: a Python loop of verify_chain_sequence over B.

    Shapes: logits [B, gamma+1, V], q [B, gamma, V], drafts [B, gamma], T [B],
    u [B, gamma+1].  Returns stacked tokens [B, gamma+1], J [B], status [B],
    p_draft [B, gamma].
    """
    B = np.asarray(logits).shape[0]
    res = [verify_chain_sequence(logits[b], q[b], drafts[b], float(T[b]), u[b]) for b in range(B)]
    return {
        "tokens": np.stack([r["tokens"] for r in res]),
        "J": np.array([r["J"] for r in res]),
        "status": np.array([r["status"] for r in res]),
        "p_draft": np.stack([r["p_draft"] for r in res]),
        "per_seq": res,
    }


# ---------------------------------------------------------------------------------------
# Block verification (one round, one sequence)
# ---------------------------------------------------------------------------------------

def verify_chain_varlen_sequence(logits, q, drafts, T: float, u, gamma_b: int, want_cdf: bool = False) -> dict:
    """One chain round that verifies only the first gamma_b drafts of a padded draft.

    SD 20.5, "Choosing how much to verify at every step" (adaptive verification): a step
    verifies l_r drafts of request r and the rest of its draft is dropped.  The round is the
    chain rule on the first gamma_b + 1 rows: drafts 0..gamma_b-1 are tested with
    u[0..gamma_b-1], and the extra token comes from row gamma_b (a rejection's residual, or
    the bonus row p_{gamma_b} with q = 0) with uniform u[gamma_b].  READINGS: the extra
    token's uniform sits at slot gamma_b of the padded [gamma+1] uniforms; gamma_b = 0
    samples row 0 directly; gamma_b outside [0, gamma] is an input error reported as
    STATUS_BAD_TOKEN (the count of drafts to verify is out of range).  Exactness needs
    gamma_b chosen without looking at the drafts it decides on (the page's
    non-anticipating requirement); the verifier cannot check that.
    Returns the chain result padded to gamma + 1 tokens and gamma p_draft entries."""
    logits = np.asarray(logits)
    g1, V = logits.shape
    gamma = g1 - 1
    gb = int(gamma_b)
    if not (0 <= gb <= gamma):
        return {"tokens": np.full(g1, -1, dtype=np.int64), "J": -1, "status": STATUS_BAD_TOKEN,
                "p_draft": np.full(gamma, np.nan), "margins": np.full(gamma, np.inf), "greedy": False}
    qq = None if q is None else np.asarray(q)[:gb]
    r = verify_chain_sequence(logits[:gb + 1], qq, list(np.asarray(drafts).reshape(-1)[:gb]), T,
                              widen(u).reshape(-1)[:gb + 1], want_cdf=want_cdf)
    tokens = np.full(g1, -1, dtype=np.int64)
    tokens[:gb + 1] = r["tokens"]
    p_draft = np.full(gamma, np.nan)
    p_draft[:gb] = r["p_draft"]
    margins = np.full(gamma, np.inf)
    margins[:gb] = r["margins"]
    return {**r, "tokens": tokens, "p_draft": p_draft, "margins": margins}


def verify_block_sequence(logits, q, drafts, T: float, u, want_cdf: bool = False) -> dict:
    """One round of block verification for one sequence.

    Art of Guessing, "Block verification" (Sun et al., 2024): the draft is judged jointly
    rather than token by token.  With p_k = softmax(l_k / T) the target's and q_k the
    drafter's distribution at draft position k (0-based here: row k predicts draft k):

      w_0 = 1,  w_{k+1} = min(1, w_k * p_k(x_k) / q_k(x_k))           (running weight)
      mass_k = sum_x (w_k p_k(x) - q_k(x))+  for k < gamma,   mass_gamma = w_gamma
      survival_k = mass_k / (mass_k + 1 - w_k)  if w_k < 1, else 1
      prefix length k (1..gamma) survives iff u[k-1] <= survival_k
      n = the longest surviving prefix (0 if none survives)
      extra token y ~ (w_n p_n - q_n)+ normalised, q_gamma == 0 (the bonus row)
      emit x_0 .. x_{n-1}, y

    READINGS: the survival test is `uniform <= survival`, as the page's block_verify
    writes it; the extra token is the inverse-CDF draw of u[gamma], as for the chain rule;
    a ratio with q_k(x_k) = 0 is +inf (p > 0) or 0 (p = 0) and 0 * inf = 0 in the weight
    recursion, with the ZERO_Q warning; a residual that sums to 0 (rounding only) falls
    back to p_n with the ZERO_RESIDUAL warning.  Every row, draft token, whole q row and
    uniform is read by the rule, so all of them are validated and every error found is
    reported (bits OR'd).  A sequence with T < GREEDY_T is verified greedily, exactly as
    verify_chain_sequence does: with a one-hot target the block rule reduces to it (the
    weights are 1 while x_k is the argmax and 0 after, and the residual is one-hot).

    Returns tokens [gamma+1] (-1 padded), J (= n), status, p_draft [gamma] (p_k(x_k)),
    w [gamma+1], survival [gamma+1], margins [gamma] (|u[k-1] - survival_k| for k =
    1..gamma), and for a sampled draw 'y_u' plus, when want_cdf, 'cdf', 'S' and 'pcdf'
    (the CDF of p_n itself).
    """
    logits = np.asarray(logits)
    g1, V = logits.shape
    gamma = g1 - 1
    drafts = [int(x) for x in np.asarray(drafts).reshape(-1)]
    assert len(drafts) == gamma
    u = widen(u).reshape(-1)
    greedy = bool(T < GREEDY_T) or bool(np.isnan(T))
    out = {
        "tokens": np.full(gamma + 1, -1, dtype=np.int64),
        "J": -1,
        "status": 0,
        "p_draft": np.full(gamma, np.nan),
        "w": np.full(gamma + 1, np.nan),
        "survival": np.full(gamma + 1, np.nan),
        "margins": np.full(gamma, np.inf),
        "greedy": greedy,
    }
    if not np.isfinite(T):
        out["status"] = STATUS_BAD_TEMPERATURE
        return out
    err = 0
    for i in range(g1):
        err |= _row_status(logits[i])
    for i in range(gamma):
        if not (0 <= drafts[i] < V):
            err |= STATUS_BAD_TOKEN
    if not greedy:
        qq = widen(q).reshape(gamma, V)
        if np.isnan(qq).any() or np.isinf(qq).any() or (qq < 0).any():
            err |= STATUS_BAD_PROB
        if not ((0.0 <= u) & (u < 1.0)).all():
            err |= STATUS_BAD_UNIFORM
    if err:
        out["status"] = err
        return out

    if greedy:
        J = gamma
        for i in range(gamma):
            if drafts[i] != lowest_argmax(logits[i]):
                J = i
                break
        out["tokens"][:J] = drafts[:J]
        out["tokens"][J] = lowest_argmax(logits[J])
        out["J"] = J
        return out

    status = 0
    p = [target_distribution(logits[k], T) for k in range(g1)]
    w = np.ones(g1)
    for k in range(gamma):
        px, qx = p[k][drafts[k]], qq[k][drafts[k]]
        out["p_draft"][k] = px
        if qx == 0.0:
            status |= STATUS_ZERO_Q
            ratio = np.inf if px > 0.0 else 0.0
        else:
            ratio = px / qx
        w[k + 1] = 0.0 if w[k] == 0.0 else min(1.0, w[k] * ratio)
    mass = np.empty(g1)
    for k in range(gamma):
        mass[k] = np.maximum(w[k] * p[k] - qq[k], 0.0).sum()
    mass[gamma] = w[gamma]
    with np.errstate(invalid="ignore", divide="ignore"):
        surv = np.where(w < 1.0, mass / (mass + 1.0 - w), 1.0)
    out["w"], out["survival"] = w, surv
    n = 0
    for k in range(1, gamma + 1):
        out["margins"][k - 1] = abs(u[k - 1] - surv[k])
        if u[k - 1] <= surv[k]:
            n = k
    qn = qq[n] if n < gamma else np.zeros(V)
    r = np.maximum(w[n] * p[n] - qn, 0.0)
    if not (r.sum() > 0.0):
        status |= STATUS_ZERO_RESIDUAL
        r = p[n].copy()
    y, C, S = inverse_cdf(r, u[gamma])
    out["tokens"][:n] = drafts[:n]
    out["tokens"][n] = y
    out["J"] = n
    out["status"] = status
    out["y_u"] = u[gamma] * S
    if want_cdf:
        out["cdf"] = C
        out["S"] = S
        out["pcdf"] = np.cumsum(p[n])  # the target row's own CDF (the zero-residual fallback)
    return out


def verify_block(logits, q, drafts, T, u) -> dict:
    """Batched block verification: a Python loop of verify_block_sequence over B."""
    B = np.asarray(logits).shape[0]
    res = [verify_block_sequence(logits[b], q[b], drafts[b], float(T[b]), u[b]) for b in range(B)]
    return {
        "tokens": np.stack([r["tokens"] for r in res]),
        "J": np.array([r["J"] for r in res]),
        "status": np.array([r["status"] for r in res]),
        "p_draft": np.stack([r["p_draft"] for r in res]),
        "per_seq": res,
    }


# ---------------------------------------------------------------------------------
# Gumbel coupling (Art of Guessing, "Speculative sampling" -> the Gumbel-max trick and
# "Gumbel coupling", Daliri et al.): the drafter and the target use the same noise g_k at
# position k; the drafter proposes argmax(log q_k + g_k), the target samples
# argmax(log p_k + g_k), and the round keeps the drafts up to the first position where the
# two differ, then emits the target's sample there.
#
# The noise is not an input: both sides generate it with Philox4x32-10 (Salmon, Moraes,
# Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011), written here from
# that definition.  READINGS (the page leaves the generator open): the uniforms of
# vocabulary entries 4j..4j+3 at row k of sequence b are the four outputs of counter
# (j, k, b, 0) under key (seed mod 2^32, seed div 2^32); a 32-bit output x gives
# u = ((x >> 9) + 0.5) / 2^23, exactly representable in float32 and inside (0, 1); the
# race is run in log2 units, score_i = a_i - log2(xi_i) with xi_i = -ln(u_i) = -log1p(u_i - 1)
# (argmax(a_i / ln 2 + g_i) with g = -ln(xi) is the same argmax), a_i = l_i * log2(e) / T
# for the target and log2(q_i) for the drafter; ties go to the lowest index.  The scores
# are float64 from the float32 uniforms.
# ---------------------------------------------------------------------------------
LOG2E = 1.0 / np.log(2.0)
PHILOX_M = (0xD2511F53, 0xCD9E8D57)   # round multipliers
PHILOX_W = (0x9E3779B9, 0xBB67AE85)   # key increments (golden ratio, sqrt(3) - 1)
_MASK32 = 0xFFFFFFFF


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Ten Philox4x32 rounds on counters (arrays of values < 2^32) under key (k0, k1).
    A round: (c0, c1, c2, c3) -> (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1,
    lo(M0 c0)); the key grows by (W0, W1) between rounds.  Returns four uint32 arrays."""
    c = [np.asarray(x, dtype=np.uint64) & _MASK32 for x in (c0, c1, c2, c3)]
    c = np.broadcast_arrays(*c)
    c = [x.copy() for x in c]
    k0, k1 = int(k0) & _MASK32, int(k1) & _MASK32
    for r in range(10):
        if r:
            k0 = (k0 + PHILOX_W[0]) & _MASK32
            k1 = (k1 + PHILOX_W[1]) & _MASK32
        p0 = np.uint64(PHILOX_M[0]) * c[0]
        p1 = np.uint64(PHILOX_M[1]) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(_MASK32)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(_MASK32)
        c = [hi1 ^ c[1] ^ np.uint64(k0), lo1, hi0 ^ c[3] ^ np.uint64(k1), lo0]
    return [x.astype(np.uint32) for x in c]


def gumbel_uniforms(seed: int, b, k, V: int) -> np.ndarray:
    """float32 uniforms of row k of sequence b (b, k scalars or broadcastable arrays):
    shape broadcast(b, k) + (V,)."""
    seed = int(seed)
    b = np.asarray(b, dtype=np.uint64)[..., None]
    k = np.asarray(k, dtype=np.uint64)[..., None]
    j = np.arange((V + 3) // 4, dtype=np.uint64)
    outs = philox4x32_10(j, k, b, np.uint64(0), seed & _MASK32, (seed >> 32) & _MASK32)
    x = np.stack(outs, axis=-1).reshape(np.broadcast_shapes(b.shape, k.shape)[:-1] + (-1,))[..., :V]
    return ((x >> np.uint32(9)).astype(np.float32) + np.float32(0.5)) * np.float32(2.0 ** -23)


def gumbel_scores(a, u32) -> np.ndarray:
    """The race in log2 units, in float64: a - log2(xi), xi = -ln(u), from the float32
    uniforms u (widened exactly) and the scores' first terms a (float64)."""
    a = np.asarray(a, dtype=np.float64)
    u = np.asarray(u32, dtype=np.float32).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        xi = -np.log1p(u - 1.0)
        return a - np.log2(xi)


def _lowest_argmax_score(s) -> int:
    """Lowest index of the largest score; a NaN score (a NaN or negative q) never wins;
    -1 when no score is a number."""
    s = np.asarray(s)
    ok = ~np.isnan(s)
    if not ok.any():
        return -1
    return int(np.flatnonzero(ok & (s == s[ok].max()))[0])


def _top2_gap(s) -> float:
    s = np.sort(np.asarray(s, dtype=np.float64)[np.isfinite(s)])
    return float(s[-1] - s[-2]) if len(s) >= 2 else np.inf


def gumbel_draft_sequence(q, seed: int, b: int) -> dict:
    """The drafter's side: x_k = argmax_i (log2 q_k(i) - log2 xi_{k,i}) for k < gamma.
    Returns drafts and each row's top-two score gap (for the parity flag rule)."""
    q = widen(q)
    gamma, V = q.shape
    u = gumbel_uniforms(seed, b, np.arange(gamma), V)
    with np.errstate(divide="ignore", invalid="ignore"):
        a = np.log2(q)
    drafts, gaps = [], []
    for kk in range(gamma):
        s = gumbel_scores(a[kk], u[kk])
        drafts.append(_lowest_argmax_score(s))
        gaps.append(_top2_gap(s))
    return {"drafts": np.array(drafts, dtype=np.int64), "gaps": np.array(gaps)}


def gumbel_target_token(logits_row, T: float, seed: int, b: int, k: int) -> tuple[int, float]:
    """The target's Gumbel-max sample at row k: argmax_i (l_i * c - log2 xi_i), c =
    log2(e) / T, in float64; returns (token, top-two score gap)."""
    c = LOG2E / float(T)
    a = widen(logits_row) * c
    s = gumbel_scores(a, gumbel_uniforms(seed, b, k, len(a)))
    return _lowest_argmax_score(s), _top2_gap(s)


def verify_gumbel_sequence(logits, drafts, T: float, seed: int, b: int) -> dict:
    """One round of Gumbel-coupled verification for sequence b.

    Art of Guessing, "Gumbel coupling": t_k = the target's Gumbel-max sample at row k with
    the shared noise; n = the first k < gamma with x_k != t_k (gamma if none); emit
    x_0..x_{n-1}, t_n.  The output is what the target alone samples with that noise,
    whatever the drafter.  Rows are evaluated left to right and the round stops at n, so
    rows after n are neither read nor validated (the chain rule's reading).  A greedy
    sequence (T < GREEDY_T) uses the plain argmax (T -> 0 of the race).  Returns tokens,
    J, status, targets (t_k of the rows evaluated, -1 after) and gaps (each evaluated
    row's top-two score gap)."""
    logits = np.asarray(logits)
    g1, V = logits.shape
    gamma = g1 - 1
    drafts = [int(x) for x in np.asarray(drafts).reshape(-1)]
    greedy = bool(T < GREEDY_T) or bool(np.isnan(T))
    out = {"tokens": np.full(g1, -1, dtype=np.int64), "J": -1, "status": 0,
           "targets": np.full(g1, -1, dtype=np.int64), "gaps": np.full(g1, np.inf), "greedy": greedy}
    if not np.isfinite(T):
        out["status"] = STATUS_BAD_TEMPERATURE
        return out
    for k in range(g1):
        rs = _row_status(logits[k])
        if rs:
            out["status"] = rs
            out["targets"][:] = -1
            return out
        if k < gamma and not (0 <= drafts[k] < V):
            out["status"] = STATUS_BAD_TOKEN
            out["targets"][:] = -1
            return out
        if greedy:
            t, gap = lowest_argmax(logits[k]), np.inf
        else:
            t, gap = gumbel_target_token(logits[k], T, seed, b, k)
        out["targets"][k], out["gaps"][k] = t, gap
        if k == gamma or drafts[k] != t:
            out["tokens"][:k] = drafts[:k]
            out["tokens"][k] = t
            out["J"] = k
            return out
    raise AssertionError("unreachable")


def verify_greedy_sequence(logits, drafts) -> dict:
    """Greedy verification only (SD 20.5, "A round of greedy speculative decoding";
    Art of Guessing, "Draft and verify"): J = longest prefix with x_i == z_i, emit z_J."""
    g1 = np.asarray(logits).shape[0]
    return verify_chain_sequence(logits, None, drafts, 0.0, np.zeros(g1))


# ---------------------------------------------------------------------------------------
# Token trees
# ---------------------------------------------------------------------------------------

def tree_depths(parents) -> np.ndarray:
    """depth(i) = number of ancestors of node i (a node whose parent is the prefix: 0).

    SD 20.5, "Token tree and tree attention".  Parents must satisfy par(i) in [-1, i).
    """
    parents = [int(x) for x in parents]
    depth = np.zeros(len(parents), dtype=np.int64)
    for i, a in enumerate(parents):
        if not (-1 <= a < i):
            raise ValueError(f"parent of node {i} is {a}, not in [-1, {i})")
        depth[i] = 0 if a == -1 else depth[a] + 1
    return depth


def build_tree_mask(parents, prefix_len: int):
    """Tree-attention mask M [n, P+n] (bool) and position ids P + depth (int64).

    SD 20.5, "Token tree and tree attention": node i attends to all P prefix positions,
    to its own ancestors and to itself, and to no other node; its position id is
    P + depth(i).  Plain ancestor
    walk.  Returns (mask, position_ids, depth).
    """
    parents = [int(x) for x in parents]
    n = len(parents)
    depth = tree_depths(parents)
    mask = np.zeros((n, prefix_len + n), dtype=bool)
    mask[:, :prefix_len] = True
    for i in range(n):
        a = i
        while a != -1:
            mask[i, prefix_len + a] = True
            a = parents[a]
    return mask, prefix_len + depth, depth


def verify_tree_sequence(logits, node_tokens, parents, T: float, u, max_depth: int) -> dict:
    """Medusa-style walk of a candidate tree for one sequence.

    Medusa notes, section "Attention Tree" (the target samples a token at the current
    node -- argmax when greedy -- and verification descends into the child carrying
    that token, stopping when none does); SD 20.5 states the greedy walk after the
    exercise "The tree attention mask".

    Row 0 of logits is the root (the distribution after the committed prefix); row
    1 + i is the distribution after node i.  The draw at depth d uses uniform u[d]
    (inverse CDF of softmax(l / T)).  READING: among children with equal tokens the
    lowest node index is taken.  Returns tokens [max_depth+1] (-1 padded), path
    [max_depth] (node ids, -1 padded), n_accepted and status.
    """
    logits = np.asarray(logits)
    n1, V = logits.shape
    n = n1 - 1
    parents = [int(x) for x in parents]
    node_tokens = [int(x) for x in node_tokens]
    u = widen(u).reshape(-1)
    greedy = bool(T < GREEDY_T) or bool(np.isnan(T))
    out = {
        "tokens": np.full(max_depth + 1, -1, dtype=np.int64),
        "path": np.full(max_depth, -1, dtype=np.int64),
        "n_accepted": -1,
        "status": 0,
    }
    status = 0 if np.isfinite(T) else STATUS_BAD_TEMPERATURE
    try:
        depth = tree_depths(parents)
        if n and depth.max() + 1 > max_depth:
            status |= STATUS_BAD_TREE
    except ValueError:
        status |= STATUS_BAD_TREE
    for t in node_tokens:
        if not (0 <= t < V):
            status |= STATUS_BAD_TOKEN
    if not greedy and not np.all((u >= 0.0) & (u < 1.0)):
        status |= STATUS_BAD_UNIFORM
    if status & STATUS_ERROR_MASK:
        out["status"] = status
        return out

    node, d = -1, 0
    while True:
        row = logits[0 if node == -1 else 1 + node]
        rs = _row_status(row)
        if rs:
            out = {**out, "tokens": np.full(max_depth + 1, -1, dtype=np.int64),
                   "path": np.full(max_depth, -1, dtype=np.int64), "status": status | rs}
            return out
        if greedy:
            y = lowest_argmax(row)
        else:
            y, _, _ = inverse_cdf(target_distribution(row, T), u[d])
        out["tokens"][d] = y
        child = next((j for j in range(n) if parents[j] == node and node_tokens[j] == y), None)
        if child is None:
            break
        out["path"][d] = child
        node, d = child, d + 1
    out["n_accepted"] = d
    out["status"] = status
    return out


def verify_tree_rr_sequence(logits, q, node_tokens, parents, T: float, u, max_depth: int,
                            want_cdf: bool = False, without_replacement: bool = False) -> dict:
    """Sampled verification of a token tree by recursive rejection, for one sequence.

    SD 20.5, box "Recursive rejection at a node with several children" (the multi-step
    speculative sampling of Miao et al., SpecInfer): at the current node, whose children
    s_1..s_k were drafted independently from q, start from R_1 = p (the target at the
    node).  Try the children in turn: accept s_i when a uniform falls below
    R_i(s_i) / q(s_i), and the walk moves to s_i's node; otherwise replace the target by
    R_{i+1} = max(0, R_i - q) / sum max(0, R_i - q) and try the next child.  When every
    child is rejected -- or the node has no children -- the extra token is drawn from the
    last R and the walk ends.  The argument for a chain applies level by level.

    logits [N+1, V]: row 0 is the target after the committed prefix (the root), row 1+i
    after node i.  q [N+1, V]: row 0 is the distribution the root's children were drafted
    from, row 1+i node i's children's.  u [N+1]: u[1+j] tests node j when it is tried,
    u[0] drives the final draw.

    READINGS: children are tried in node-index order; the test is `u * q(s) < R(s)` (the
    chain rule's strict test, so q(s) = 0 accepts iff R(s) > 0, with the ZERO_Q warning);
    the final draw is the inverse CDF of u[0] over R; a residual that sums to 0 after
    rounding (R_i = q) keeps R_i, with the ZERO_RESIDUAL warning.  A greedy sequence
    (T < GREEDY_T) descends into the lowest-index child carrying the argmax and emits the
    argmax where none does (a one-hot target reduces the rule to it).  Validation: the
    tree, every node token, T and (sampled) every uniform up front, as the Medusa walk
    does; then, in walk order, the logits row of every visited node, q(s) of every tried
    child, and the whole q row of a node at its first rejection (when the residual needs
    it).  An error gives n_accepted -1 and -1 outputs.

    without_replacement: Sequoia's variant (Chen et al.; SD 20.5, the paragraph after the
    box's proof): a node's children were drawn without replacement, so each try has its
    own draft distribution q_i -- q with the tokens of the children already rejected at the
    node set to zero, renormalised -- used both in the test (u * q_i(s_i) < R_i(s_i)) and
    in the residual (R_{i+1} = max(0, R_i - q_i) normalised).  READINGS: q_1 = q as given
    (as everywhere else) and q_i = q / Z_i off the rejected tokens with
    Z_i = 1 - sum of q at them (the renormaliser of a q that sums to 1); when Z_i <= 0
    (q's mass is used up) q_i is zero, so the try follows the q(s) = 0 rule and a rejection
    leaves R_i as it is; children drawn without replacement carry distinct tokens, so two
    children of one node with the same token are an input error (BAD_TREE).

    Returns tokens [max_depth+1] (-1 padded), path [max_depth], n_accepted, status,
    margins [N] (|u[1+j] - R(s_j)/q(s_j)| for every tried child j, inf otherwise) and,
    for a sampled final draw, 'y_u' and (want_cdf) 'cdf', 'S'.
    """
    logits = np.asarray(logits)
    n1, V = logits.shape
    n = n1 - 1
    parents = [int(x) for x in parents]
    node_tokens = [int(x) for x in node_tokens]
    u = widen(u).reshape(-1)
    greedy = bool(T < GREEDY_T) or bool(np.isnan(T))
    out = {
        "tokens": np.full(max_depth + 1, -1, dtype=np.int64),
        "path": np.full(max_depth, -1, dtype=np.int64),
        "n_accepted": -1,
        "status": 0,
        "margins": np.full(n, np.inf),
        "greedy": greedy,
    }
    status = 0 if np.isfinite(T) else STATUS_BAD_TEMPERATURE
    try:
        depth = tree_depths(parents)
        if n and depth.max() + 1 > max_depth:
            status |= STATUS_BAD_TREE
    except ValueError:
        status |= STATUS_BAD_TREE
    for t in node_tokens:
        if not (0 <= t < V):
            status |= STATUS_BAD_TOKEN
    if without_replacement and not status & STATUS_BAD_TREE:
        seen = set()
        for j in range(n):
            if (parents[j], node_tokens[j]) in seen:
                status |= STATUS_BAD_TREE
            seen.add((parents[j], node_tokens[j]))
    if not greedy and not np.all((u >= 0.0) & (u < 1.0)):
        status |= STATUS_BAD_UNIFORM
    if status & STATUS_ERROR_MASK:
        out["status"] = status
        return out

    def fail(bits):  # an error reports error bits only (warnings describe a clean round)
        out["tokens"][:] = -1
        out["path"][:] = -1
        out["n_accepted"] = -1
        out["status"] = (status | bits) & STATUS_ERROR_MASK
        return out

    node, d = -1, 0
    while True:
        row = 0 if node == -1 else 1 + node
        rs = _row_status(logits[row])
        if rs:
            return fail(rs)
        children = [j for j in range(n) if parents[j] == node]
        if greedy:
            y = lowest_argmax(logits[row])
            child = next((j for j in children if node_tokens[j] == y), None)
        else:
            R = target_distribution(logits[row], T)
            qn = widen(q[row]) if children else None
            q_checked = False
            child = None
            rejected, Zi = [], 1.0  # without replacement: tokens rejected here, q's mass left
            for j in children:
                s = node_tokens[j]
                qs = qn[s]
                if not (np.isfinite(qs) and qs >= 0.0):
                    return fail(STATUS_BAD_PROB)
                if without_replacement:  # q_i(s): children are distinct, so s is not rejected yet
                    qs = qs / Zi if Zi > 0.0 else 0.0
                if qs == 0.0:
                    status |= STATUS_ZERO_Q
                    out["margins"][j] = np.inf
                    accept = R[s] > 0.0
                else:
                    out["margins"][j] = abs(u[1 + j] - R[s] / qs)
                    accept = u[1 + j] * qs < R[s]
                if accept:
                    child = j
                    break
                if not q_checked:  # the residual reads the whole row
                    if not np.all(np.isfinite(qn) & (qn >= 0.0)):
                        return fail(STATUS_BAD_PROB)
                    q_checked = True
                if without_replacement:
                    qi = np.zeros_like(qn)
                    if Zi > 0.0:
                        qi = qn / Zi
                        qi[rejected] = 0.0
                    rejected.append(s)
                    Zi -= qn[s]
                else:
                    qi = qn
                r = np.maximum(R - qi, 0.0)
                if r.sum() > 0.0:
                    R = r / r.sum()
                else:
                    status |= STATUS_ZERO_RESIDUAL
            if child is None:
                y, C, S = inverse_cdf(R, u[0])
                out["y_u"] = u[0] * S
                if want_cdf:
                    out["cdf"], out["S"] = C, S
        if child is None:
            out["tokens"][d] = y
            break
        out["tokens"][d] = node_tokens[child]
        out["path"][d] = child
        node, d = child, d + 1
    out["n_accepted"] = d
    out["status"] = status
    return out


def verify_tree_rr(logits, q, node_tokens, parents, T, u, max_depth: int,
                   without_replacement: bool = False) -> dict:
    """Batched recursive-rejection tree verification: a loop of verify_tree_rr_sequence."""
    B = np.asarray(logits).shape[0]
    res = [verify_tree_rr_sequence(logits[b], q[b], node_tokens[b], parents, float(T[b]), u[b], max_depth,
                                   without_replacement=without_replacement)
           for b in range(B)]
    return {
        "tokens": np.stack([r["tokens"] for r in res]),
        "path": np.stack([r["path"] for r in res]),
        "n_accepted": np.array([r["n_accepted"] for r in res]),
        "status": np.array([r["status"] for r in res]),
    }


def verify_tree(logits, node_tokens, parents, T, u, max_depth: int) -> dict:
    """Batched tree verification: loop of verify_tree_sequence over the batch."""
    B = np.asarray(logits).shape[0]
    res = [verify_tree_sequence(logits[b], node_tokens[b], parents, float(T[b]), u[b], max_depth)
           for b in range(B)]
    return {
        "tokens": np.stack([r["tokens"] for r in res]),
        "path": np.stack([r["path"] for r in res]),
        "n_accepted": np.array([r["n_accepted"] for r in res]),
        "status": np.array([r["status"] for r in res]),
    }


def compact_kv(cache, prefix_len, path, num_accepted, block_table=None, block_size: int = 0):
    """Accepted-branch compaction of a KV cache after a tree round (SD 20.5, "Keeping the
    caches consistent after a rejection": the accepted branch's entries, scattered among
    discarded siblings, are gathered into consecutive slots; a chain only moves a length).

    cache [B, S, W] (contiguous) or [num_blocks, block_size, W] with block_table [B, max
    blocks] (paged: logical slot s of sequence b lives in block block_table[b, s //
    block_size], row s % block_size).  Node i of sequence b's tree sits at logical slot
    prefix_len[b] + i; after the round the entry of path[b, d] moves to slot prefix_len[b] + d
    for d < num_accepted[b].  Returns (new cache, new lengths prefix_len + num_accepted, status
    per sequence).  The definition gathers from the cache as it was before the round.
    READINGS: a path must climb the tree (path[d] >= d and strictly increasing, as node ids
    along a root path do), else the sequence is left alone with STATUS_BAD_TREE; a sequence
    with num_accepted < 0 (a failed round) is left alone and keeps its length."""
    src = np.asarray(cache)
    out = src.copy()
    B = len(prefix_len)
    new_len = np.array([int(prefix_len[b]) + max(int(num_accepted[b]), 0) for b in range(B)])
    status = np.zeros(B, dtype=np.int64)

    def at(b, s):
        if block_table is None:
            return (b, s)
        return (int(block_table[b][s // block_size]), s % block_size)

    for b in range(B):
        J = int(num_accepted[b])
        if J < 0:
            new_len[b] = int(prefix_len[b])
            continue
        pth = [int(x) for x in np.asarray(path[b])[:J]]
        if any(pth[d] < d for d in range(J)) or any(pth[d + 1] <= pth[d] for d in range(J - 1)):
            status[b] = STATUS_BAD_TREE
            new_len[b] = int(prefix_len[b])
            continue
        P0 = int(prefix_len[b])
        for d in range(J):
            out[at(b, P0 + d)] = src[at(b, P0 + pth[d])]
    return out, new_len, status


def cartesian_tree_counts(tops) -> tuple[int, int]:
    """(nodes, paths) of the full Cartesian candidate tree with s_i candidates at depth i.

    Medusa notes, "Attention Tree": depth i holds prod_{j<=i} s_j nodes, so the tree has
    sum_i prod_{j<=i} s_j tokens and prod_i s_i root-to-leaf paths.  Counted here by
    enumerating the tree itself.
    """
    nodes = 0
    level = [()]
    for s in tops:
        level = [path + (r,) for path in level for r in range(s)]
        nodes += len(level)
    return nodes, len(level)


def medusa_sparse_tree(accuracy, n_nodes: int):
    """Greedy sparse candidate tree from per-head top-k accuracies.

    Medusa notes, section "OPTIMIZED TREE CONSTRUCTION": with a_k^(i) the accuracy of
    head k's i-th candidate, a node reached by the path (i_1..i_m) is accepted with
    probability prod_j a_j^(i_j) (accuracies assumed independent), and the expected
    accepted length is the sum of these products over the tree's nodes; the tree is
    grown by repeatedly adding the node of largest product.

    accuracy[k][i] must be exact decimal strings or Fractions (READING: products are
    compared exactly, so mathematically equal products tie exactly).  Because every
    accuracy is <= 1, a child never outranks its parent, so the n_nodes largest
    products form a tree; READING: ties resolve by (depth, lexicographic path).
    Nodes are emitted ordered by (depth, lexicographic path), parents before children.

    Returns (parents [n], paths list of tuples of 0-based ranks, values list of Fraction).
    """
    acc = [[Fraction(a) for a in head] for head in accuracy]
    K = len(acc)
    cand = []
    for m in range(1, K + 1):
        for path in itertools.product(*[range(len(acc[j])) for j in range(m)]):
            v = Fraction(1)
            for j, r in enumerate(path):
                v *= acc[j][r]
            cand.append((v, path))
    cand.sort(key=lambda vp: (-vp[0], len(vp[1]), vp[1]))
    chosen = cand[:n_nodes]
    chosen.sort(key=lambda vp: (len(vp[1]), vp[1]))
    index = {path: i for i, (_, path) in enumerate(chosen)}
    parents = []
    for _, path in chosen:
        if len(path) == 1:
            parents.append(-1)
        else:
            if path[:-1] not in index:
                raise ValueError("selected nodes are not closed under parents")
            parents.append(index[path[:-1]])
    return parents, [p for _, p in chosen], [v for v, _ in chosen]


def medusa_expected_length(values) -> Fraction:
    """E[L] = sum over the tree's nodes of their path products (Medusa notes,
    "OPTIMIZED TREE CONSTRUCTION"); the tree version of 1 + sum_i a_i counts the
    extra token separately (Art of Guessing, "Token trees")."""
    return sum(values, Fraction(0))
