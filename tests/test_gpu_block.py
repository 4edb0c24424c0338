"""GPU parity of block verification (Art of Guessing, "Block verification") against the
fp64 oracle, through the C ABI.  The comparison rules are tests/parity.py's, with the
block rule's flag: two accepted lengths may differ only where the survival test of the
longer one lies within FLAG_TOL of its boundary."""
import json
import os

import numpy as np
import pytest
import torch

import workloads
from parity import ParityReport, assert_flag_budget, check_chain, run_oracle_chain

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
KEYS = ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms")


@pytest.fixture(scope="module")
def sd(built_library):
    import speculative_decoding_token_temperature_gb300 as m
    m.load_library()
    return m


@pytest.fixture(params=["one_launch", "two_pass"], autouse=True)
def block_path(request, sd):
    """Every test runs on both implementations: the single launch that reads each row
    once (default) and the statistics + mass kernels (the library's test hook)."""
    with sd.test_hooks(block_two_pass=int(request.param == "two_pass")):
        yield request.param


def _np(t):
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def _run_and_check(sd, report, x, sample=None, workers=None):
    path = "two_pass" if sd.get_test_hook(sd.HOOK_BLOCK_TWO_PASS) else "one_launch"
    report.name = report.name.split(" [")[0] + f" [{path}]"
    out = sd.verify_block(*(x[k] for k in KEYS))
    torch.cuda.synchronize()
    idx = slice(None) if sample is None else sample
    gpu = {k: _np(v)[idx] for k, v in out.items()}
    orc = run_oracle_chain(*(_np(x[k])[idx] for k in KEYS), gpu["tokens"], gpu["num_accepted"],
                           workers=workers, mode="block")
    check_chain(report, gpu, orc, _np(x["uniforms"])[idx], rule="block")
    return out


def _finish(report, budget=True):
    """No hard failure; on a measured workload (budget) the stated flag bound as well."""
    path = os.environ.get("SPECDEC_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(dict(report.summary(), rule="block")) + "\n")
    assert not report.failures, report.failures[:10]
    if budget:
        assert_flag_budget(report.flagged, report.rows, report.summary())


def test_block_b1_v1000_all_rounds(sd):
    rep = ParityReport("block chain_b1_v1000 (100 rounds)")
    for r in range(100):
        _run_and_check(sd, rep, workloads.chain_workload("chain_b1_v1000", r, DEV), workers=1)
    _finish(rep)


def test_block_b64_v32000_all_rounds(sd):
    rep = ParityReport("block chain_b64_v32000 (40 rounds)")
    for r in range(40):
        _run_and_check(sd, rep, workloads.chain_workload("chain_b64_v32000", r, DEV))
    _finish(rep)


def test_block_b256_v128256_full_rounds(sd):
    """Two full-size launches, every sequence checked."""
    rep = ParityReport("block chain_b256_v128256 (2 full rounds)")
    for r in range(2):
        x = workloads.chain_workload("chain_b256_v128256", r, DEV)
        _run_and_check(sd, rep, x)
        del x
    _finish(rep)


def test_block_b512_v152064_fp32_full_round(sd):
    rep = ParityReport("block chain_b512_v152064 (1 full round)")
    x = workloads.chain_workload("chain_b512_v152064", 0, DEV)
    _run_and_check(sd, rep, x)
    del x
    torch.cuda.empty_cache()
    _finish(rep)


@pytest.mark.parametrize("B,gamma,V,dtype", [
    (3, 1, 8, "fp32"), (2, 2, 16, "bf16"), (5, 3, 1004, "fp32"), (4, 4, 1000, "bf16"),
    (2, 16, 4104, "bf16"), (3, 2, 16384 + 8, "bf16"), (2, 3, 3 * 8192 + 4, "fp32"),
    (7, 5, 50000, "bf16"), (2, 31, 64, "fp32"),
])
def test_block_ragged_shapes(sd, B, gamma, V, dtype):
    rep = ParityReport(f"block ragged B={B} g={gamma} V={V} {dtype}")
    for seed in range(3):
        x = workloads.make_chain_inputs(B, gamma, V, dtype, seed=seed, device=DEV,
                                        recipe="spikes", scale=2.0, n_spikes=min(3, V), spike=4.0,
                                        noise=0.7, temps="uniform:0.0:1.5")
        _run_and_check(sd, rep, x, workers=1)
    _finish(rep, budget=False)  # a few dozen rows per shape: flags reported, not bounded


def test_block_unsupported_layouts_are_refused(sd):
    x = workloads.make_chain_inputs(2, 2, 7, "fp32", seed=0, device=DEV)   # 28-byte rows
    with pytest.raises(sd.SpecdecError, match="unsupported"):
        sd.verify_block(*(x[k] for k in KEYS))
    x = workloads.make_chain_inputs(1, 32, 64, "fp32", seed=0, device=DEV)  # g + 1 > 32
    with pytest.raises(sd.SpecdecError, match="unsupported"):
        sd.verify_block(*(x[k] for k in KEYS))


def test_block_errors_are_all_reported(sd):
    """The block rule reads every row, draft, q row and uniform: every error is found and
    the bits are OR'd, whatever the position."""
    from oracle import specdec_oracle as so
    B, g, V = 12, 3, 256
    x = workloads.make_chain_inputs(B, g, V, "fp32", seed=5, device=DEV, temps="const:0.9")
    L, q, d, T, u = (x[k].clone() for k in KEYS)
    L[0, 3, 17] = float("nan")            # the bonus row
    L[1, 2, :] = float("-inf")
    L[2, 0, 3] = float("inf")
    d[3, 2] = V
    d[4, 0] = -2
    u[5, 0] = 1.0
    q[6, 0, int(d[6, 0])] = 0.0          # warning only
    q[7, 2, 100] = -0.5                   # far from any draft
    T[8] = float("nan")
    T[9] = -1.0                           # greedy
    L[10, 3, 5] = float("nan")            # two errors in one sequence
    u[10, 1] = -0.25
    q[11, 1, 7] = float("inf")
    d[11, 0] = V + 3
    out = sd.verify_block(L, q, d, T, u)
    torch.cuda.synchronize()
    for b in range(B):
        o = so.verify_block_sequence(_np(L)[b], _np(q)[b], _np(d)[b], float(T[b]), _np(u)[b])
        assert int(out["status"][b]) & 0xFF == o["status"] & 0xFF, (b, int(out["status"][b]), o["status"])
        assert int(out["status"][b]) & 256 == o["status"] & 256, b
        if o["status"] & 0xFF:
            assert int(out["num_accepted"][b]) == -1 and (out["tokens"][b] == -1).all(), b
            assert torch.isnan(out["p_draft"][b]).all(), b


def test_one_hot_target_gives_greedy_tokens(sd):
    """A one-hot target (every logit -inf but the argmax) at T = 1 keeps the drafts while
    they are the argmax and emits the argmax after them, as greedy verification does."""
    B, g, V = 32, 5, 4096
    x = workloads.make_chain_inputs(B, g, V, "bf16", seed=9, device=DEV, temps="const:1.0")
    L = x["logits"].float()
    z = L.argmax(dim=-1)
    d = x["draft_tokens"].clone()
    keep = torch.rand(B, g, generator=torch.Generator(device=DEV).manual_seed(1), device=DEV) < 0.7
    d = torch.where(keep, z[:, :g].to(torch.int32), d)
    hot = torch.full_like(L, float("-inf"))
    hot.scatter_(2, z.unsqueeze(-1), 0.0)
    out = sd.verify_block(hot, x["draft_probs"], d, x["temperatures"], x["uniforms"])
    ref = sd.verify_greedy(x["logits"], d)
    torch.cuda.synchronize()
    assert torch.equal(out["tokens"], ref["tokens"])
    assert torch.equal(out["num_accepted"], ref["num_accepted"])


def test_block_outputs_fully_written_and_deterministic(sd):
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
        sd.verify_block(*(x[k] for k in KEYS), out=out)
        torch.cuda.synchronize()
        for k in ("tokens", "num_accepted", "status"):
            assert not (out[k] == 0x7F7F7F7F).any(), k
        assert not (out["p_draft"] == 123.0).any()
        res.append({k: v.clone() for k, v in out.items()})
    for r in res[1:]:
        for k in r:
            assert torch.equal(torch.nan_to_num(r[k].float(), nan=-7.0), torch.nan_to_num(res[0][k].float(), nan=-7.0)), k


def test_block_and_chain_share_a_workspace(sd):
    """Calls of both rules on one stream reuse the binding's workspace."""
    x = workloads.make_chain_inputs(6, 3, 20000, "bf16", seed=11, device=DEV, temps="const:1.0")
    a = sd.verify_block(*(x[k] for k in KEYS))
    c = sd.verify_chain(*(x[k] for k in KEYS))
    a2 = sd.verify_block(*(x[k] for k in KEYS))
    c2 = sd.verify_chain(*(x[k] for k in KEYS))
    torch.cuda.synchronize()
    assert torch.equal(a["tokens"], a2["tokens"]) and torch.equal(c["tokens"], c2["tokens"])
