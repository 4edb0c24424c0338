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
    """V = 6 rows are not 16-byte aligned (scalar-load kernels); V = 8 rows take the
    streaming bulk-copy kernels."""
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
