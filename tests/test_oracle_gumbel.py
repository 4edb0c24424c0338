"""Pins of the oracle's Gumbel-coupled verification (Art of Guessing, the Gumbel-max trick
and "Gumbel coupling").

The race and the coupling are checked against what the page states about them, on the
oracle's own noise: the race samples softmax(l / T) (the exponential-clocks argument), the
drafter and the target agree with the page's closed-form probability
sum_j 1 / sum_i max(p_i / p_j, q_i / q_j) (and with sum_i p_i q_i when the noise is not
shared), the emitted tokens are the target's own samples whatever the drafter
(drafter invariance), and T -> 0 is greedy matching.  The statistical pins use 4-5 sigma
bounds on fixed seeds.
"""
import numpy as np
import pytest
from scipy import stats

from oracle import specdec_oracle as so


def _race(a, seed, n, k=0):
    """Argmax of the race over n independent sequences b = 0..n-1 at row k."""
    u = so.gumbel_uniforms(seed, np.arange(n), k, len(a))
    s = so.gumbel_scores(np.asarray(a, dtype=np.float32)[None, :], u)
    return s.argmax(axis=1)


def test_uniforms_are_uniform_and_on_the_grid():
    u = so.gumbel_uniforms(123, np.arange(256), 3, 1024).ravel()
    assert u.dtype == np.float32 and u.min() > 0.0 and u.max() < 1.0
    m = (u.astype(np.float64) * 2.0 ** 23) - 0.5
    np.testing.assert_array_equal(m, np.round(m))  # ((x >> 9) + 0.5) / 2^23 exactly
    counts = np.histogram(u, bins=64, range=(0.0, 1.0))[0]
    assert stats.chisquare(counts).pvalue > 1e-4
    # streams of different rows, sequences and seeds are unrelated
    a = so.gumbel_uniforms(123, 5, 0, 50000).astype(np.float64)
    for other in (so.gumbel_uniforms(123, 5, 1, 50000), so.gumbel_uniforms(123, 6, 0, 50000),
                  so.gumbel_uniforms(124, 5, 0, 50000)):
        assert abs(np.corrcoef(a, other.astype(np.float64))[0, 1]) < 0.02
    # neighbouring entries of one row too
    assert abs(np.corrcoef(a[:-1], a[1:])[0, 1]) < 0.02


@pytest.mark.parametrize("T", [0.5, 1.0, 1.7])
def test_race_samples_the_softmax(T):
    logits = np.array([1.2, -0.3, 0.4, 2.0, -1.5, 0.0])
    c = np.float32(np.float32(so.LOG2E) / np.float32(T))
    a = logits.astype(np.float32) * c
    n = 120000
    idx = _race(a, 99, n)
    counts = np.bincount(idx, minlength=len(logits))
    p = so.target_distribution(logits, T)
    assert stats.chisquare(counts, p * n).pvalue > 1e-4


def _match_closed_form(p, q):
    return sum(1.0 / np.sum(np.maximum(p / p[j], q / q[j])) for j in range(len(p)))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_shared_noise_match_probability_is_the_closed_form(seed):
    rng = np.random.default_rng(seed)
    V = 5
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    n = 100000
    tgt = _race(np.log2(p).astype(np.float32), 7 + seed, n)
    dft = _race(np.log2(q).astype(np.float32), 7 + seed, n)        # shared noise
    ind = _race(np.log2(q).astype(np.float32), 1000 + seed, n)     # independent noise
    want = _match_closed_form(p, q)
    got = np.mean(tgt == dft)
    sd = np.sqrt(want * (1 - want) / n)
    assert abs(got - want) < 5 * sd
    tv = so.total_variation(p, q)
    assert want >= (1 - tv) / (1 + tv) - 1e-12
    want_ind = float(np.sum(p * q))
    assert abs(np.mean(tgt == ind) - want_ind) < 5 * np.sqrt(want_ind * (1 - want_ind) / n)


def test_output_is_drafter_invariant():
    """Whatever the drafter, the tokens a round emits are the target's own samples
    t_0..t_J under the shared noise."""
    rng = np.random.default_rng(3)
    V, gamma, T, seed = 300, 6, 0.9, 5
    for b in range(30):
        logits = rng.standard_normal((gamma + 1, V)) * 2.0
        own = [so.gumbel_target_token(logits[k], T, seed, b, k)[0] for k in range(gamma + 1)]
        for noise in (0.0, 0.5, 3.0):
            ql = logits[:gamma] / T + noise * rng.standard_normal((gamma, V))
            q = np.exp(ql - ql.max(axis=1, keepdims=True))
            q /= q.sum(axis=1, keepdims=True)
            d = so.gumbel_draft_sequence(q, seed, b)["drafts"]
            r = so.verify_gumbel_sequence(logits, d, T, seed, b)
            J = r["J"]
            assert list(r["tokens"][:J + 1]) == own[:J + 1]
            assert all(d[k] == own[k] for k in range(J))
            assert J == gamma or d[J] != own[J]


def test_drafter_with_the_target_distribution_is_always_accepted():
    rng = np.random.default_rng(4)
    V, gamma, seed = 200, 5, 9
    logits = rng.standard_normal((gamma + 1, V))
    p = np.stack([so.target_distribution(logits[k], 1.0) for k in range(gamma)])
    d = so.gumbel_draft_sequence(p, seed, 0)["drafts"]
    r = so.verify_gumbel_sequence(logits, d, 1.0, seed, 0)
    # log2 p and l * log2(e) differ by a constant per row, up to float32 rounding
    assert r["J"] == gamma or r["gaps"][r["J"]] < 1e-5


def test_low_temperature_is_greedy_matching():
    rng = np.random.default_rng(6)
    V, gamma = 100, 4
    for _ in range(20):
        logits = rng.standard_normal((gamma + 1, V)) * 3
        z = logits.argmax(axis=1)
        d = [int(z[i]) if rng.random() < 0.7 else int((z[i] + 1) % V) for i in range(gamma)]
        g = so.verify_greedy_sequence(logits, d)
        r0 = so.verify_gumbel_sequence(logits, d, 0.0, 1, 0)
        np.testing.assert_array_equal(r0["tokens"], g["tokens"])
        # a small positive temperature lets the logits dominate the noise
        r1 = so.verify_gumbel_sequence(logits, d, 0.002, 1, 0)
        np.testing.assert_array_equal(r1["tokens"], g["tokens"])


def test_status_follows_the_rows_read():
    V, gamma = 50, 3
    logits = np.zeros((gamma + 1, V))
    logits[:, 7] = 20.0  # every row's sample is 7 at T = 1
    d = [7, 7, 3]
    r = so.verify_gumbel_sequence(logits, d, 1.0, 0, 0)
    assert r["status"] == 0 and r["J"] == 2 and list(r["tokens"]) == [7, 7, 7, -1]
    bad = logits.copy(); bad[3, 1] = np.nan  # the bonus row is never reached
    assert so.verify_gumbel_sequence(bad, d, 1.0, 0, 0)["status"] == 0
    bad = logits.copy(); bad[1, 1] = np.nan
    r = so.verify_gumbel_sequence(bad, d, 1.0, 0, 0)
    assert r["status"] == so.STATUS_BAD_LOGIT and r["J"] == -1
    assert so.verify_gumbel_sequence(logits, [7, 99, 3], 1.0, 0, 0)["status"] == so.STATUS_BAD_TOKEN
    assert so.verify_gumbel_sequence(logits, d, np.inf, 0, 0)["status"] == so.STATUS_BAD_TEMPERATURE


def test_target_sample_follows_softmax_at_temperature():
    """The oracle's own target sampler (the one verification uses) draws softmax(l / T)."""
    logits = np.array([0.7, -0.2, 1.5, 0.1])
    T = 0.6
    n = 40000
    toks = np.array([so.gumbel_target_token(logits, T, 21, b, 2)[0] for b in range(n)])
    counts = np.bincount(toks, minlength=len(logits))
    assert stats.chisquare(counts, so.target_distribution(logits, T) * n).pvalue > 1e-4


def _kat_vectors():
    from pathlib import Path
    rows = []
    for line in (Path(__file__).resolve().parent / "golden" / "philox4x32_10_kat.txt").read_text().splitlines():
        line = line.strip()
        if line.startswith("kat ="):
            w = [int(t, 16) for t in line.split("=", 1)[1].split()]
            rows.append((w[:4], w[4:6], w[6:10]))
    assert len(rows) == 3
    return rows


def test_philox_matches_the_published_known_answers():
    """Philox4x32-10 against the generator's published known-answer vectors (Random123,
    Salmon et al., SC 2011): counter, key -> four output words, bit for bit."""
    for ctr, key, want in _kat_vectors():
        got = [int(x) for x in so.philox4x32_10(*ctr, *key)]
        assert got == want, ([hex(v) for v in got], [hex(v) for v in want])


def _philox_variant(ctr, key, *, swap_hilo=False, bump_first=False, swap_mult=False, rounds=10,
                    swap_key_words=False):
    """Philox4x32 with one plausible mistake planted (the KAT test must reject each)."""
    M = (0xD2511F53, 0xCD9E8D57)
    W = (0x9E3779B9, 0xBB67AE85)
    m0, m1 = (M[1], M[0]) if swap_mult else M
    c = list(ctr)
    k0, k1 = (key[1], key[0]) if swap_key_words else key
    for r in range(rounds):
        if r or bump_first:
            k0, k1 = (k0 + W[0]) & 0xFFFFFFFF, (k1 + W[1]) & 0xFFFFFFFF
        p0, p1 = m0 * c[0], m1 * c[2]
        hi0, lo0, hi1, lo1 = p0 >> 32, p0 & 0xFFFFFFFF, p1 >> 32, p1 & 0xFFFFFFFF
        if swap_hilo:
            hi0, lo0, hi1, lo1 = lo0, hi0, lo1, hi1
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return c


@pytest.mark.parametrize("mistake", [dict(swap_hilo=True), dict(bump_first=True), dict(swap_mult=True),
                                     dict(rounds=7), dict(swap_key_words=True)])
def test_planted_philox_mistakes_fail_the_known_answers(mistake):
    kats = _kat_vectors()
    # the unmodified variant reproduces every vector (the variant itself is faithful) ...
    for ctr, key, want in kats:
        assert _philox_variant(ctr, key) == want
    # ... and each planted mistake misses at least one of them
    assert any(_philox_variant(ctr, key, **mistake) != want for ctr, key, want in kats)
