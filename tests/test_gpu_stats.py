"""Statistical exactness of the CUDA path (SD 20.5: test a speculative sampler by its
output distribution over many samples, never by speed).

10^6 seeded rounds on a small vocabulary: the first emitted token must follow p_1, the
accepted length must follow the survival law P(J >= i) = prod_{j<i} alpha_j with
alpha_j = sum_x min(p_j, q_j), and the extra token given J must follow the normalised
residual (p_J - q_J)+ (or p_gamma for the bonus).  Pearson chi-square, p-value > 1e-3.
"""
import numpy as np
import pytest
import scipy.stats
import torch

from golden import read_fixture
from oracle import specdec_oracle as so

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ROUNDS = 1_000_000
BATCH = 50_000


@pytest.fixture(scope="module")
def sd(built_library):
    import speculative_decoding_token_temperature_gb300 as m
    m.load_library()
    return m


def _chi2(counts, probs):
    counts = np.asarray(counts, dtype=np.float64)
    probs = np.asarray(probs, dtype=np.float64)
    keep = probs > 0
    assert counts[~keep].sum() == 0, "a zero-probability outcome occurred"
    if keep.sum() == 1:  # a one-point law: every count in that cell is the whole test
        return 1.0
    exp = probs[keep] / probs[keep].sum() * counts.sum()
    return scipy.stats.chisquare(counts[keep], exp).pvalue


@pytest.mark.parametrize("dtype,V", [("fp32", 6), ("bf16", 6), ("fp32", 8), ("bf16", 8)])
def test_chain_output_law(sd, dtype, V):
    """V = 6 rows are not 16-byte aligned (scalar-load kernels); V = 8 rows (32 bytes in
    fp32, 16 in bf16) take the left-to-right kernel."""
    gamma, T = 3, 0.8
    rng = np.random.default_rng(21)
    logits = rng.standard_normal((gamma + 1, V)) * 1.5
    t = torch.tensor(logits, dtype=torch.float32)
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    lw = t.float().numpy().astype(np.float64)
    p = [so.target_distribution(lw[i], T) for i in range(gamma + 1)]
    q = rng.dirichlet(np.ones(V) * 2.0, size=gamma)
    qt = torch.tensor(q, dtype=torch.float32)
    qd = qt.double().numpy()
    alpha = [so.acceptance_rate(p[i], qd[i]) for i in range(gamma)]

    g = torch.Generator(device=DEV).manual_seed(5)
    first = np.zeros(V)
    J_hist = np.zeros(gamma + 1)
    y_given_J = np.zeros((gamma + 1, V))
    L = t.to(DEV).unsqueeze(0).expand(BATCH, gamma + 1, V).contiguous()
    Q = qt.to(DEV).unsqueeze(0).expand(BATCH, gamma, V).contiguous()
    Tt = torch.full((BATCH,), T, device=DEV)
    for _ in range(ROUNDS // BATCH):
        d = torch.multinomial(Q.view(-1, V), 1, replacement=True, generator=g).view(BATCH, gamma).to(torch.int32)
        u = torch.rand(BATCH, gamma + 1, generator=g, device=DEV)
        out = sd.verify_chain(L, Q, d, Tt, u)
        tok = out["tokens"].long()
        J = out["num_accepted"].long()
        assert (out["status"] == 0).all()
        first += torch.bincount(tok[:, 0], minlength=V).cpu().numpy()
        J_hist += torch.bincount(J, minlength=gamma + 1).cpu().numpy()
        y = tok.gather(1, J.view(-1, 1)).view(-1)
        y_given_J += torch.bincount(J * V + y, minlength=(gamma + 1) * V).view(gamma + 1, V).cpu().numpy()

    assert _chi2(first, p[0]) > 1e-3
    surv = np.cumprod([1.0] + alpha)               # P(J >= i), i = 0..gamma
    pJ = np.append(surv[:-1] - surv[1:], surv[-1])
    assert _chi2(J_hist, pJ) > 1e-3
    for j in range(gamma + 1):
        w = so.residual_distribution(p[j], qd[j]) if j < gamma else p[gamma]
        if y_given_J[j].sum() > 100:
            assert _chi2(y_given_J[j], w) > 1e-3, j


def test_tree_first_token_law(sd):
    V, T = 7, 0.6
    parents = torch.tensor([-1, -1, 0], dtype=torch.int32, device=DEV)
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((4, V)) * 1.2
    lt = torch.tensor(logits, dtype=torch.float32)
    p0 = so.target_distribution(lt.double().numpy()[0], T)
    p1 = so.target_distribution(lt.double().numpy()[1], T)
    toks = torch.tensor([2, 5, 1], dtype=torch.int32)
    g = torch.Generator(device=DEV).manual_seed(9)
    first = np.zeros(V)
    second_after_node0 = np.zeros(V)
    L = lt.to(DEV).unsqueeze(0).expand(BATCH, 4, V).contiguous()
    K = toks.to(DEV).unsqueeze(0).expand(BATCH, 3).contiguous()
    Tt = torch.full((BATCH,), T, device=DEV)
    for _ in range(ROUNDS // BATCH // 2):
        u = torch.rand(BATCH, 3, generator=g, device=DEV)
        out = sd.verify_tree(L, K, parents, Tt, u, 2)
        tok = out["tokens"].long()
        first += torch.bincount(tok[:, 0], minlength=V).cpu().numpy()
        via0 = out["path"][:, 0] == 0
        second_after_node0 += torch.bincount(tok[via0, 1], minlength=V).cpu().numpy()
    assert _chi2(first, p0) > 1e-3
    assert _chi2(second_after_node0, p1) > 1e-3


def _bigram_round(sd, LP, QQ, ctx, g):
    """One verification round (gamma = 1) of the toy bigram model from contexts ctx: the
    drafter proposes d ~ q(. | ctx); target rows p(. | ctx) and p(. | d)."""
    n = ctx.numel()
    d = torch.multinomial(QQ[ctx], 1, generator=g).view(n)
    L = torch.stack([LP[ctx], LP[d]], 1).contiguous()
    Q = QQ[ctx].unsqueeze(1).contiguous()
    u = torch.rand(n, 2, generator=g, device=DEV)
    out = sd.verify_chain(L, Q, d.view(n, 1).to(torch.int32), torch.ones(n, device=DEV), u)
    assert (out["status"] == 0).all()
    return out["tokens"].long(), out["num_accepted"].long()


@pytest.mark.parametrize("V", [6, 8])
def test_bigram_two_token_joint_law(sd, V):
    """SD 20.5, "A broken sampler looks healthy on a speed dashboard": a toy bigram target
    and drafter over V tokens; rounds of gamma = 1 from a start token until every sequence
    has emitted two tokens; the joint law of (first, second) must be p(a | s) p(b | a) over
    all V^2 cells (chi-square; V = 6: the page's 36 cells, rows of 24 bytes for the
    scalar-load kernels; V = 8: 32-byte rows for the left-to-right kernel).  The
    resample-from-p mistake (the extra token after a rejection drawn from p instead of the
    residual), planted on the host in a copy of the outputs, must fail the same test."""
    s0 = 3
    rng = np.random.default_rng(11)
    P = rng.dirichlet(np.ones(V) * 1.2, size=V)
    Qd = rng.dirichlet(np.ones(V) * 1.2, size=V)
    LP = torch.tensor(np.log(P), dtype=torch.float32, device=DEV)
    QQ = torch.tensor(Qd, dtype=torch.float32, device=DEV)
    Pw = np.stack([so.target_distribution(LP[c].double().cpu().numpy(), 1.0) for c in range(V)])
    PW = torch.tensor(Pw, dtype=torch.float64, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(17)
    good, bad = np.zeros(V * V), np.zeros(V * V)
    for _ in range(ROUNDS // BATCH):
        ctx = torch.full((BATCH,), s0, dtype=torch.long, device=DEV)
        tok, J = _bigram_round(sd, LP, QQ, ctx, g)
        first, second = tok[:, 0], torch.where(J == 1, tok[:, 1], torch.full_like(J, -1))
        need = J == 0
        tok2, J2 = _bigram_round(sd, LP, QQ, first[need], g)
        second[need] = tok2[:, 0]
        good += torch.bincount(first * V + second, minlength=V * V).cpu().numpy()
        # the planted mistake: after a rejection the extra token comes from p, not the residual
        bf = torch.where(need, torch.multinomial(PW[ctx].float(), 1, generator=g).view(-1), first)
        bs = second.clone()
        rej2 = J2 == 0
        idx = torch.nonzero(need).view(-1)
        bs[idx[rej2]] = torch.multinomial(PW[first[need][rej2]].float(), 1, generator=g).view(-1)
        bad += torch.bincount(bf * V + bs, minlength=V * V).cpu().numpy()
    joint = (Pw[s0][:, None] * Pw).reshape(-1)
    assert _chi2(good, joint) > 1e-3
    assert _chi2(bad, joint) < 1e-6


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_accepted_length_iid_worked_example(sd, dtype):
    """SD 20.5, "How many tokens a round produces, and the speedup": the worked example's
    p and q (box "The rule by hand, three tokens") at every position, alpha = 0.7, gamma = 4:
    E[J + 1] = (1 - 0.7^5) / 0.3 = 2.77310 within 4 standard errors over 10^6 rounds, and J
    follows the capped geometric law.  The vocabulary is padded with zero-probability
    tokens (logit -inf, q = 0) to 16-byte rows, so the left-to-right kernel runs."""
    fx = read_fixture("worked_example_3token.txt")
    p = np.array([float(v) for v in fx["p"]])
    q = np.array([float(v) for v in fx["q"]])
    gamma, V = 4, (4 if dtype == "fp32" else 8)
    lrow = np.full(V, -np.inf)
    lrow[:3] = np.log(p)
    qrow = np.zeros(V)
    qrow[:3] = q
    lt = torch.tensor(lrow, dtype=torch.float32)
    if dtype == "bf16":
        lt = lt.to(torch.bfloat16)
    pw = so.target_distribution(lt.double().numpy(), 1.0)
    qt = torch.tensor(qrow, dtype=torch.float32)
    alpha = so.acceptance_rate(pw, qt.double().numpy())
    if dtype == "fp32":
        assert abs(alpha - 0.7) < 1e-6  # the page's alpha (bf16 logits round p slightly)
    L = lt.to(DEV).view(1, 1, V).expand(BATCH, gamma + 1, V).contiguous()
    Q = qt.to(DEV).view(1, 1, V).expand(BATCH, gamma, V).contiguous()
    Tt = torch.ones(BATCH, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(29)
    hist = np.zeros(gamma + 1)
    for _ in range(ROUNDS // BATCH):
        d = torch.multinomial(Q.view(-1, V), 1, replacement=True, generator=g).view(BATCH, gamma).to(torch.int32)
        u = torch.rand(BATCH, gamma + 1, generator=g, device=DEV)
        out = sd.verify_chain(L, Q, d, Tt, u)
        assert (out["status"] == 0).all()
        hist += torch.bincount(out["num_accepted"].long(), minlength=gamma + 1).cpu().numpy()
    law = np.array([alpha ** i * (1 - alpha) for i in range(gamma)] + [alpha ** gamma])
    n = hist.sum()
    mean = float((hist * np.arange(1, gamma + 2)).sum() / n)
    sd_ = float(np.sqrt((law * (np.arange(1, gamma + 2) - (law * np.arange(1, gamma + 2)).sum()) ** 2).sum()))
    expect = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(mean - expect) < 4 * sd_ / np.sqrt(n), (mean, expect)
    if dtype == "fp32":
        assert abs(expect - 2.77310) < 1e-5
    assert _chi2(hist, law) > 1e-3


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_tree_without_replacement_first_token_law(sd, dtype):
    """SD 20.5, the paragraph after the proof of "Recursive rejection at a node with
    several children" (Sequoia): with a node's children drawn without replacement, each
    rejected token zeroed in q and q renormalised, the emitted token still follows p.
    Three children at the root, drawn without replacement from q, 10^6 walks: the first
    token's law is p (chi-square); the i.i.d. rule applied to the same children is not
    (its error here is 0.05 on two tokens, found exactly in the oracle's pins)."""
    V, k = 8, 3
    p4 = np.array([0.10, 0.40, 0.30, 0.20])
    q4 = np.array([0.40, 0.30, 0.20, 0.10])
    lrow = np.full(V, -np.inf)
    lrow[:4] = np.log(p4)
    qrow = np.zeros(V)
    qrow[:4] = q4
    lt = torch.tensor(lrow, dtype=torch.float32)
    if dtype == "bf16":
        lt = lt.to(torch.bfloat16)
    pw = so.target_distribution(lt.double().numpy(), 1.0)
    L = lt.to(DEV).view(1, 1, V).expand(BATCH, k + 1, V).contiguous()
    Q = torch.tensor(qrow, dtype=torch.float32, device=DEV).view(1, 1, V).expand(BATCH, k + 1, V).contiguous()
    parents = torch.full((k,), -1, dtype=torch.int32, device=DEV)
    T = torch.ones(BATCH, device=DEV)
    qdraw = torch.tensor(qrow, dtype=torch.float64).view(1, V).expand(BATCH, V).contiguous()
    g_cpu = torch.Generator().manual_seed(31)  # sequential draws without replacement, in draw order
    g = torch.Generator(device=DEV).manual_seed(37)
    good, bad = np.zeros(V), np.zeros(V)
    for _ in range(ROUNDS // BATCH):
        toks = torch.multinomial(qdraw, k, replacement=False, generator=g_cpu).to(torch.int32).to(DEV)
        u = torch.rand(BATCH, k + 1, generator=g, device=DEV)
        out = sd.verify_tree_recursive(L, Q, toks, parents, T, u, 1, without_replacement=True)
        assert (out["status"] & 0xFF == 0).all()
        good += torch.bincount(out["tokens"][:, 0].long(), minlength=V).cpu().numpy()
        iid = sd.verify_tree_recursive(L, Q, toks, parents, T, u, 1)
        bad += torch.bincount(iid["tokens"][:, 0].long(), minlength=V).cpu().numpy()
    assert _chi2(good, pw) > 1e-3
    assert _chi2(bad, pw) < 1e-6
