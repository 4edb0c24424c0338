"""A seeded random sweep of shapes and inputs for the chain, per-request-count (varlen),
block and greedy rules against the fp64 oracle, under the parity rules of tests/parity.py.

Batch sizes, draft counts, vocabularies (16-byte rows and not), logits dtypes, input
recipes, drafter noise and temperature mixes come from one seeded generator, so that a
size- or input-dependent mistake that the fixed shape lists miss still meets the oracle.
Each case stays small enough for the oracle (at most 3M logits per call)."""
import numpy as np
import pytest
import torch

import workloads
from parity import ParityReport, check_chain, run_oracle_chain

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KEYS = ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms")
MAX_ELEMS = 3_000_000


@pytest.fixture(scope="module")
def sd(built_library):
    import speculative_decoding_token_temperature_gb300 as m
    m.load_library()
    return m


def _np(t):
    return (t.float() if t.dtype == torch.bfloat16 else t).detach().cpu().numpy()


def _cases(seed, n):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        V = int([rng.integers(1, 64), rng.integers(64, 6000), rng.integers(6000, 70000)][rng.integers(0, 3)])
        if rng.random() < 0.5:
            V = max(8, V - V % 8)  # rows of whole 16-byte vectors in both dtypes
        g = int(rng.integers(1, 32))
        B = int(max(1, min(rng.integers(1, 64), MAX_ELEMS // ((g + 1) * V))))
        yield dict(B=B, gamma=g, V=V, dtype=["bf16", "fp32"][rng.integers(0, 2)],
                   recipe=["spikes", "zipf"][rng.integers(0, 2)], noise=float(rng.choice([0.3, 0.8, 1.5])),
                   temps=str(rng.choice(["const:1.0", "uniform:0.0:1.5", "half_greedy:0.8", "uniform:0.5:2.0"])),
                   seed=int(rng.integers(0, 2**31)))


def _inputs(c):
    return workloads.make_chain_inputs(c["B"], c["gamma"], c["V"], c["dtype"], seed=c["seed"], device=DEV,
                                       recipe=c["recipe"], scale=2.0, n_spikes=min(3, c["V"]), spike=4.0,
                                       noise=c["noise"], temps=c["temps"])


@pytest.mark.parametrize("rule", ["chain", "varlen", "block"])
def test_random_sweep(sd, rule):
    rep = ParityReport(f"random sweep, {rule}")
    for i, c in enumerate(_cases({"chain": 11, "varlen": 12, "block": 13}[rule], 16)):
        if rule in ("varlen", "block"):  # both need 16-byte rows (specdec.h)
            c["V"] = max(8, c["V"] - c["V"] % 8)
        x = _inputs(c)
        gammas = None
        if rule == "chain":
            out = sd.verify_chain(*(x[k] for k in KEYS))
        elif rule == "block":
            out = sd.verify_block(*(x[k] for k in KEYS))
        else:
            gen = np.random.default_rng(c["seed"])
            gammas = torch.from_numpy(gen.integers(0, c["gamma"] + 1, c["B"]).astype(np.int32)).to(DEV)
            out = sd.verify_chain_varlen(*(x[k] for k in KEYS), gammas)
        torch.cuda.synchronize()
        gpu = {k: _np(v) for k, v in out.items()}
        orc = run_oracle_chain(*(_np(x[k]) for k in KEYS), gpu["tokens"], gpu["num_accepted"], workers=1,
                               mode=rule, gammas=None if gammas is None else gammas.cpu().numpy())
        n0 = len(rep.failures)
        gm = None if gammas is None else gammas.cpu().numpy()
        check_chain(rep, gpu, orc, _np(x["uniforms"]), rule="block" if rule == "block" else "chain", extra_slot=gm)
        assert len(rep.failures) == n0, (i, c, rep.failures[n0:n0 + 3])
        if gm is not None:
            assert (gpu["num_accepted"] <= gm).all(), (i, c)
    assert not rep.failures


def test_random_sweep_greedy(sd):
    from oracle import specdec_oracle as so
    for c in _cases(14, 16):
        x = _inputs(c)
        out = sd.verify_greedy(x["logits"], x["draft_tokens"])
        torch.cuda.synchronize()
        L, d = _np(x["logits"]), _np(x["draft_tokens"])
        toks, J, st = _np(out["tokens"]), _np(out["num_accepted"]), _np(out["status"])
        for b in range(c["B"]):
            o = so.verify_greedy_sequence(L[b], d[b])
            assert int(J[b]) == o["J"] and int(st[b]) == o["status"], (c, b)
            assert np.array_equal(toks[b], o["tokens"]), (c, b)


def test_random_sweep_gumbel(sd):
    """Gumbel coupling over the same kind of random cases (the drafts from the oracle's
    shared-noise drafter, so that long agreeing prefixes occur), against the oracle's race."""
    from test_gpu_gumbel import Report as GumbelReport, check_rounds, oracle_drafts
    rep = GumbelReport("random sweep, gumbel")
    for i, c in enumerate(_cases(15, 12)):
        B = max(1, min(c["B"], 2_000_000 // ((c["gamma"] + 1) * c["V"])))
        c = dict(c, B=B)
        x = _inputs(c)
        seed = c["seed"] % (2**40)
        od = oracle_drafts(_np(x["draft_probs"]), seed, range(B))
        drafts = torch.tensor(np.stack([od[b]["drafts"] for b in range(B)]), dtype=torch.int32, device=DEV)
        out = sd.verify_gumbel(x["logits"], drafts, x["temperatures"], seed)
        torch.cuda.synchronize()
        n0 = len(rep.failures)
        check_rounds(rep, _np(x["logits"]), {b: od[b]["drafts"] for b in range(B)}, _np(x["temperatures"]), seed,
                     out, range(B))
        assert len(rep.failures) == n0, (i, {k: c[k] for k in ("B", "gamma", "V", "dtype")}, rep.failures[n0:n0 + 3])
    rep.finish()
