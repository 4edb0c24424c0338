"""GPU parity of chain and greedy verification against the fp64 oracle (via the C ABI)."""
import json
import os

import numpy as np
import pytest
import torch

import workloads
from parity import FLAG_TOL, ParityReport, assert_flag_budget, check_chain, run_oracle_chain

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def sd(built_library):
    import speculative_decoding_token_temperature_gb300 as m
    m.load_library()
    return m


def _np(t):
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def _run_and_check(sd, report, x, sample=None, workers=None):
    out = sd.verify_chain(x["logits"], x["draft_probs"], x["draft_tokens"], x["temperatures"], x["uniforms"])
    torch.cuda.synchronize()
    idx = slice(None) if sample is None else sample
    gpu = {k: _np(v)[idx] for k, v in out.items()}
    orc = run_oracle_chain(_np(x["logits"])[idx], _np(x["draft_probs"])[idx], _np(x["draft_tokens"])[idx],
                           _np(x["temperatures"])[idx], _np(x["uniforms"])[idx],
                           gpu["tokens"], gpu["num_accepted"], workers=workers)
    check_chain(report, gpu, orc, _np(x["uniforms"])[idx])
    return out


def _record(report):
    path = os.environ.get("SPECDEC_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(report.summary()) + "\n")


def _finish(report, budget=True):
    """No hard failure; on a measured workload (budget) the stated flag bound as well."""
    _record(report)
    assert not report.failures, report.failures[:10]
    if budget:
        assert_flag_budget(report.flagged, report.rows, report.summary())


def test_chain_b1_v1000_all_rounds(sd):
    rep = ParityReport("chain_b1_v1000 (100 rounds)")
    for r in range(100):
        _run_and_check(sd, rep, workloads.chain_workload("chain_b1_v1000", r, DEV), workers=1)
    _finish(rep)


def test_chain_b64_v32000_all_rounds(sd):
    rep = ParityReport("chain_b64_v32000 (100 rounds)")
    for r in range(100):
        _run_and_check(sd, rep, workloads.chain_workload("chain_b64_v32000", r, DEV))
    _finish(rep)


def test_chain_b256_v128256_full_rounds(sd):
    """Five full-size launches of the benchmarked workload, every sequence checked: 10,240
    rows, enough for the 1e-4 bound on flagged rows to be measurable (it allows one)."""
    rep = ParityReport("chain_b256_v128256 (5 full rounds)")
    for r in range(5):
        x = workloads.chain_workload("chain_b256_v128256", r, DEV)
        _run_and_check(sd, rep, x)
        del x
    _finish(rep)


def test_chain_b256_v128256_sigma075_full_rounds(sd):
    rep = ParityReport("chain_b256_v128256_s075 (5 full rounds)")
    for r in range(5):
        x = workloads.chain_workload("chain_b256_v128256_s075", r, DEV)
        _run_and_check(sd, rep, x)
        del x
    _finish(rep)


def test_chain_b512_v152064_full_rounds(sd):
    """Three full-size launches of the B=512 fp32 workload, every sequence checked."""
    rep = ParityReport("chain_b512_v152064 (3 full rounds)")
    for r in range(3):
        x = workloads.chain_workload("chain_b512_v152064", r, DEV)
        _run_and_check(sd, rep, x)
        del x
        torch.cuda.empty_cache()
    _finish(rep)


@pytest.mark.parametrize("B,gamma,V,dtype", [
    (3, 1, 1, "fp32"), (2, 2, 7, "bf16"), (5, 3, 1001, "fp32"), (4, 4, 1001, "bf16"),
    (2, 16, 4099, "bf16"), (3, 2, 16384 + 8, "bf16"), (2, 3, 3 * 8192 + 4, "fp32"),
    (1, 1, 8, "fp32"), (7, 5, 50000, "bf16"), (2, 255, 64, "fp32"),
    (4, 31, 8192, "bf16"), (3, 31, 6144 + 4, "fp32"),  # the left-to-right kernel's longest chains
    (300, 2, 1024, "bf16"),                              # more sequences than teams
])
def test_chain_ragged_shapes(sd, B, gamma, V, dtype):
    rep = ParityReport(f"ragged B={B} g={gamma} V={V} {dtype}")
    for seed in range(3):
        x = workloads.make_chain_inputs(B, gamma, V, dtype, seed=seed, device=DEV,
                                        recipe="spikes", scale=2.0, n_spikes=min(3, V), spike=4.0,
                                        noise=0.7, temps="uniform:0.0:1.5")
        _run_and_check(sd, rep, x, workers=1)
    _finish(rep, budget=False)  # a few dozen rows per shape: flags reported, not bounded


def test_greedy_call_matches_oracle(sd):
    from oracle import specdec_oracle as so
    for dtype, V in [("bf16", 32000), ("fp32", 1001), ("bf16", 5)]:
        x = workloads.make_chain_inputs(16, 4, V, dtype, seed=3, device=DEV, scale=1.0, n_spikes=1,
                                        spike=3.0, noise=0.2, temps="const:0.0")
        out = sd.verify_greedy(x["logits"], x["draft_tokens"])
        torch.cuda.synchronize()
        L, d = _np(x["logits"]), _np(x["draft_tokens"])
        for b in range(16):
            o = so.verify_greedy_sequence(L[b], d[b])
            assert int(out["num_accepted"][b]) == o["J"]
            assert np.array_equal(_np(out["tokens"])[b], o["tokens"])
            assert int(out["status"][b]) == o["status"]


def test_greedy_ties_resolve_to_lowest_index(sd):
    V = 64
    logits = torch.zeros(2, 3, V, dtype=torch.bfloat16, device=DEV)
    logits[:, :, 5] = 2.0
    logits[:, :, 9] = 2.0
    logits[:, :, 40] = 2.0
    drafts = torch.tensor([[5, 5], [5, 9]], dtype=torch.int32, device=DEV)
    out = sd.verify_greedy(logits, drafts)
    assert out["num_accepted"].tolist() == [2, 1]
    assert out["tokens"].tolist() == [[5, 5, 5], [5, 5, -1]]


def test_degenerate_inputs_set_status(sd):
    from oracle import specdec_oracle as so
    B, g, V = 10, 3, 256
    x = workloads.make_chain_inputs(B, g, V, "fp32", seed=5, device=DEV, temps="const:0.9")
    L, q, d, T, u = (x[k].clone() for k in ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms"))
    L[0, 1, 17] = float("nan")
    L[1, 2, :] = float("-inf")
    L[2, 0, 3] = float("inf")
    d[3, 1] = V
    d[4, 0] = -2
    u[5, 2] = 1.0
    q[6, 0, int(d[6, 0])] = 0.0          # warning only
    q[7, 1, int(d[7, 1])] = -0.5
    T[8] = float("nan")
    T[9] = -1.0                            # greedy
    out = sd.verify_chain(L, q, d, T, u)
    torch.cuda.synchronize()
    for b in range(B):
        o = so.verify_chain_sequence(_np(L)[b], _np(q)[b], _np(d)[b], float(T[b]), _np(u)[b])
        assert int(out["status"][b]) & 0xFF == o["status"] & 0xFF, (b, int(out["status"][b]), o["status"])
        assert int(out["status"][b]) & 256 == o["status"] & 256
        if o["status"] & 0xFF:
            assert int(out["num_accepted"][b]) == -1 and (out["tokens"][b] == -1).all()
    # a NaN draft probability inside the drawn row is caught by the draw
    x2 = workloads.make_chain_inputs(1, 1, 64, "fp32", seed=1, device=DEV, temps="const:1.0")
    x2["uniforms"][0, 0] = 0.999999
    x2["draft_probs"][0, 0, 7] = float("nan")
    o2 = sd.verify_chain(x2["logits"], x2["draft_probs"], x2["draft_tokens"], x2["temperatures"], x2["uniforms"])
    r2 = so.verify_chain_sequence(_np(x2["logits"])[0], _np(x2["draft_probs"])[0], _np(x2["draft_tokens"])[0], 1.0,
                                  _np(x2["uniforms"])[0])
    assert int(o2["status"][0]) == r2["status"]
    assert int(o2["num_accepted"][0]) == r2["J"]


def test_p_equals_q_always_accepts(sd):
    B, g, V = 8, 4, 1000
    logits = torch.randn(B, g + 1, V, device=DEV) * 2
    q = torch.softmax(logits[:, :g], dim=-1)
    d = torch.multinomial(q.view(-1, V), 1).view(B, g).to(torch.int32)
    u = torch.rand(B, g + 1, device=DEV) * 0.999
    out = sd.verify_chain(logits, q.contiguous(), d, torch.ones(B, device=DEV), u)
    # u < p/q holds except when rounding puts p/q a hair below u very close to 1
    assert (out["num_accepted"] >= 0).all()
    assert (out["num_accepted"] == g).float().mean() > 0.95


def test_outputs_fully_written_and_deterministic(sd):
    x = workloads.chain_workload("chain_b64_v32000", 7, DEV)
    B, g1 = x["uniforms"].shape
    res = []
    for _ in range(3):
        out = {
            "tokens": torch.full((B, g1), 0x7F7F7F7F, dtype=torch.int32, device=DEV),
            "num_accepted": torch.full((B,), 0x7F7F7F7F, dtype=torch.int32, device=DEV),
            "status": torch.full((B,), 0x7F7F7F7F, dtype=torch.int32, device=DEV),
            "p_draft": torch.full((B, g1 - 1), 123.0, device=DEV),
        }
        sd.verify_chain(x["logits"], x["draft_probs"], x["draft_tokens"], x["temperatures"], x["uniforms"], out=out)
        torch.cuda.synchronize()
        assert not (out["tokens"] == 0x7F7F7F7F).any()
        assert not (out["num_accepted"] == 0x7F7F7F7F).any()
        assert not (out["status"] == 0x7F7F7F7F).any()
        assert not (out["p_draft"] == 123.0).any()
        res.append({k: v.clone() for k, v in out.items()})
    for r in res[1:]:
        for k in r:
            assert torch.equal(torch.nan_to_num(r[k].float(), nan=-7.0), torch.nan_to_num(res[0][k].float(), nan=-7.0)), k


def test_workspace_reuse_across_shapes(sd):
    xa = workloads.make_chain_inputs(6, 3, 20000, "bf16", seed=11, device=DEV, temps="const:1.0")
    xb = workloads.make_chain_inputs(40, 7, 3000, "fp32", seed=12, device=DEV, temps="const:0.7")
    ra = sd.verify_chain(*(xa[k] for k in ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms")))
    rb = sd.verify_chain(*(xb[k] for k in ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms")))
    ra2 = sd.verify_chain(*(xa[k] for k in ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms")))
    rb2 = sd.verify_chain(*(xb[k] for k in ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms")))
    torch.cuda.synchronize()
    assert torch.equal(ra["tokens"], ra2["tokens"]) and torch.equal(rb["tokens"], rb2["tokens"])


def test_host_tensors_round_trip(sd):
    x = workloads.chain_workload("chain_b1_v1000", 3, "cpu")
    x = {k: v.pin_memory() for k, v in x.items()}
    out = sd.verify_chain(x["logits"], x["draft_probs"], x["draft_tokens"], x["temperatures"], x["uniforms"])
    assert out["tokens"].device.type == "cpu"
    xd = {k: v.to(DEV) for k, v in x.items()}
    out2 = sd.verify_chain(xd["logits"], xd["draft_probs"], xd["draft_tokens"], xd["temperatures"], xd["uniforms"])
    assert torch.equal(out["tokens"], out2["tokens"].cpu())


def test_flag_tolerance_constant():
    assert FLAG_TOL == 1e-5
