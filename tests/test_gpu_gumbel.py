"""GPU parity of Gumbel-coupled verification and of the drafter's shared-noise sampler
against the oracle (Art of Guessing, "Gumbel coupling"), through the C ABI.

Both sides regenerate the same Philox4x32-10 noise, so every uniform is bit-identical;
the oracle forms the scores in float64 and the kernels in float32, so two entries whose
scores lie within GAP_TOL of each other may swap.  Rules:
status bits and greedy rows bit-exact; a sampled token (draft or target) may differ only
where the oracle's top-two score gap at that row is below GAP_TOL (flagged); the round
then follows from the tokens.
"""
import json
import os

import numpy as np
import pytest
import torch

import workloads
from parity import assert_flag_budget

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GAP_TOL = 1e-4  # log2 units


@pytest.fixture(scope="module")
def sd(built_library):
    import speculative_decoding_token_temperature_gb300 as m
    m.load_library()
    return m


def _np(t):
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


class Report:
    def __init__(self, name):
        self.name, self.rows, self.flagged, self.failures, self.accepted, self.seqs = name, 0, 0, [], 0, 0

    def fail(self, msg):
        if len(self.failures) < 20:
            self.failures.append(msg)

    def finish(self):
        path = os.environ.get("SPECDEC_PARITY_REPORT")
        if path:
            with open(path, "a") as f:
                f.write(json.dumps({"workload": self.name, "rule": "gumbel", "rows": self.rows,
                                    "sequences": self.seqs, "mean_accepted": self.accepted / max(self.seqs, 1),
                                    "flagged": self.flagged, "hard_failures": len(self.failures)}) + "\n")
        assert not self.failures, self.failures[:10]


def oracle_drafts(q, seed, idx):
    from oracle import specdec_oracle as so
    return {b: so.gumbel_draft_sequence(q[b], seed, b) for b in idx}


def check_rounds(rep, L, drafts, T, seed, gpu, idx):
    from oracle import specdec_oracle as so
    g_t, g_J, g_s = (_np(gpu[k]) for k in ("tokens", "num_accepted", "status"))
    for b in idx:
        o = so.verify_gumbel_sequence(L[b], drafts[b], float(T[b]), seed, b)
        rep.seqs += 1
        rep.rows += len(o["tokens"])  # gamma + 1 rows per sequence, as in the chain rule
        if int(g_s[b]) != o["status"]:
            rep.fail(f"seq {b}: status gpu {int(g_s[b])} oracle {o['status']}")
            continue
        if o["status"]:
            if g_J[b] != -1 or (g_t[b] != -1).any():
                rep.fail(f"seq {b}: error sequence has outputs")
            continue
        rep.accepted += o["J"]
        if g_J[b] == o["J"] and np.array_equal(g_t[b], o["tokens"]):
            continue
        # the first row whose target token differs must be a near-tie in the oracle
        k = 0
        while k <= o["J"] and k < len(g_t[b]) and g_t[b][k] == o["tokens"][k]:
            k += 1
        if not o["greedy"] and k <= o["J"] and o["gaps"][k] < GAP_TOL:
            rep.flagged += 1
        else:
            rep.fail(f"seq {b}: gpu J={g_J[b]} {g_t[b]} oracle J={o['J']} {o['tokens']} gaps {o['gaps']}")


@pytest.mark.parametrize("B,gamma,V,dtype", [
    (6, 3, 1000, "fp32"), (4, 4, 32000, "bf16"), (3, 2, 1001, "bf16"), (5, 3, 7, "fp32"), (2, 5, 50000, "bf16"),
])
def test_gumbel_round_shapes(sd, B, gamma, V, dtype):
    rep = Report(f"gumbel B={B} g={gamma} V={V} {dtype}")
    for seed in range(3):
        x = workloads.make_chain_inputs(B, gamma, V, dtype, seed=seed, device=DEV, recipe="spikes", scale=2.0,
                                        n_spikes=min(3, V), spike=4.0, noise=0.4, temps="uniform:0.0:1.5")
        q = _np(x["draft_probs"])
        od = oracle_drafts(q, 77 + seed, range(B))
        drafts = torch.tensor(np.stack([od[b]["drafts"] for b in range(B)]), dtype=torch.int32, device=DEV)
        # the drafter's sampler on the GPU against the oracle's
        gd = _np(sd.gumbel_draft(x["draft_probs"], 77 + seed))
        for b in range(B):
            for k in range(gamma):
                if gd[b, k] != od[b]["drafts"][k] and not od[b]["gaps"][k] < GAP_TOL:
                    rep.fail(f"draft b={b} k={k}: gpu {gd[b, k]} oracle {od[b]['drafts'][k]}")
        out = sd.verify_gumbel(x["logits"], drafts, x["temperatures"], 77 + seed)
        torch.cuda.synchronize()
        check_rounds(rep, _np(x["logits"]), {b: od[b]["drafts"] for b in range(B)}, _np(x["temperatures"]),
                     77 + seed, out, range(B))
    rep.finish()
    assert rep.flagged <= 1


def test_gumbel_b256_v128256_full_round(sd):
    """A full-size launch; the oracle drafts and checks every sequence (the drafts the GPU
    verifies are the oracle's), and at most 1e-4 of the rows may be flagged."""
    rep = Report("gumbel chain_b256_v128256 (1 full round)")
    x = workloads.chain_workload("chain_b256_v128256", 0, DEV)
    seed = 2024
    idx = list(range(256))
    q = x["draft_probs"]
    od = oracle_drafts({b: _np(q[b]) for b in idx}, seed, idx)
    drafts = sd.gumbel_draft(q, seed).clone()
    for b in idx:
        drafts[b] = torch.tensor(od[b]["drafts"], dtype=torch.int32, device=DEV)
    out = sd.verify_gumbel(x["logits"], drafts, x["temperatures"], seed)
    torch.cuda.synchronize()
    L = _np(x["logits"][idx])
    Lfull = {b: L[i] for i, b in enumerate(idx)}
    T = _np(x["temperatures"])
    check_rounds(rep, Lfull, {b: od[b]["drafts"] for b in idx}, T, seed, out, idx)
    rep.finish()
    assert rep.accepted > 0
    assert_flag_budget(rep.flagged, rep.rows, (rep.flagged, rep.rows))


def test_gumbel_errors_follow_the_rows_read(sd):
    from oracle import specdec_oracle as so
    B, g, V = 8, 3, 256
    x = workloads.make_chain_inputs(B, g, V, "fp32", seed=4, device=DEV, temps="const:0.8")
    L = x["logits"].clone()
    T = x["temperatures"].clone()
    q = _np(x["draft_probs"])
    d = torch.tensor(np.stack([so.gumbel_draft_sequence(q[b], 5, b)["drafts"] for b in range(B)]),
                     dtype=torch.int32, device=DEV)
    L[0, 0, 3] = float("nan")
    L[1, 3, 3] = float("nan")      # the bonus row: read only if every draft is accepted
    L[2, 0, :] = float("-inf")
    d[3, 0] = V + 1
    d[4, 2] = -5                    # read only if drafts 0 and 1 are accepted
    T[5] = float("nan")
    T[6] = 0.0
    out = sd.verify_gumbel(L, d, T, 5)
    torch.cuda.synchronize()
    Ln, dn, Tn = _np(L), _np(d), _np(T)
    for b in range(B):
        o = so.verify_gumbel_sequence(Ln[b], dn[b], float(Tn[b]), 5, b)
        assert int(out["status"][b]) == o["status"], (b, int(out["status"][b]), o["status"])
        assert int(out["num_accepted"][b]) == o["J"], b
        if o["status"]:
            assert (out["tokens"][b] == -1).all()


def test_gumbel_drafter_invariance_on_gpu(sd):
    """Two drafters sharing the noise: each round emits the target's own samples, so the
    tokens agree wherever both rounds reached."""
    B, g, V = 16, 5, 32000
    x = workloads.make_chain_inputs(B, g, V, "bf16", seed=8, device=DEV, temps="const:1.0", noise=0.3)
    y = workloads.make_chain_inputs(B, g, V, "bf16", seed=9, device=DEV, temps="const:1.0", noise=2.0)
    d1 = sd.gumbel_draft(x["draft_probs"], 11)
    d2 = sd.gumbel_draft(y["draft_probs"], 11)
    o1 = sd.verify_gumbel(x["logits"], d1, x["temperatures"], 11)
    o2 = sd.verify_gumbel(x["logits"], d2, x["temperatures"], 11)
    torch.cuda.synchronize()
    for b in range(B):
        n = min(int(o1["num_accepted"][b]), int(o2["num_accepted"][b]))
        assert torch.equal(o1["tokens"][b, :n + 1], o2["tokens"][b, :n + 1])


def test_noise_matches_the_float64_definition(sd):
    """The library's noise against G = -log2(-log1p(u - 1)) in float64 on the same
    uniforms: every entry within 4e-6, two float32 ulps at |G| < 32 (the parity rule's tie
    band is 1e-4)."""
    from oracle import specdec_oracle as so
    B, R, V, seed = 3, 4, 262147, 99
    g = _np(sd.gumbel_noise(seed, B, R, V, device=DEV))
    worst = 0.0
    for b in range(B):
        u = so.gumbel_uniforms(seed, b, np.arange(R), V).astype(np.float64)
        want = -np.log2(-np.log1p(u - 1.0))
        worst = max(worst, float(np.max(np.abs(g[b] - want))))
    assert worst < 4e-6, worst


def test_gumbel_deterministic(sd):
    x = workloads.chain_workload("chain_b64_v32000", 2, DEV)
    d = sd.gumbel_draft(x["draft_probs"], 3)
    a = sd.verify_gumbel(x["logits"], d, x["temperatures"], 3)
    b = sd.verify_gumbel(x["logits"], d, x["temperatures"], 3)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k])
    assert torch.equal(d, sd.gumbel_draft(x["draft_probs"], 3))


def test_noise_at_the_zero_known_answer(sd):
    """Counter (0, 0, 0, 0) under key (0, 0) is the first published Philox4x32-10
    known-answer vector (Random123, Salmon et al., SC 2011): seed 0, sequence 0, row 0,
    entries 0..3 of the library's noise come from those four words."""
    from pathlib import Path
    line = next(l for l in (Path(__file__).resolve().parent / "golden" / "philox4x32_10_kat.txt")
                .read_text().splitlines() if l.startswith("kat = 00000000 00000000 00000000 00000000 00000000 00000000"))
    words = np.array([int(t, 16) for t in line.split("=", 1)[1].split()[6:10]], dtype=np.float64)
    u = (np.floor(words / 512.0) + 0.5) * 2.0 ** -23
    want = -np.log2(-np.log1p(u - 1.0))
    g = _np(sd.gumbel_noise(0, 1, 1, 4, device=DEV)).reshape(-1)
    assert np.max(np.abs(g - want)) < 4e-6, (g, want)
