"""The chain calls' other kernel paths and their bounded waits, through the C ABI.

- The all-rows streaming kernels (statistics, decision, draw, finish), which serve the
  chain and greedy calls under the library's test hook and, without it, shapes beyond the
  left-to-right kernel's vocabulary limit: parity with the fp64 oracle under the rules of
  tests/parity.py.
- A bounded wait that gives up: the test hook that loses queued draws makes the teams that
  wait for them give up after a short bound; every sequence then comes back either exact
  or marked SPECDEC_STATUS_TIMEOUT (J = -1, tokens -1, p_draft NaN), and the next call on
  the same context is exact again.
"""
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


def _np(t):
    return (t.float() if t.dtype == torch.bfloat16 else t).detach().cpu().numpy()


def _check(sd, rep, x, workers=None, idx=None):
    out = sd.verify_chain(*(x[k] for k in KEYS))
    torch.cuda.synchronize()
    sel = slice(None) if idx is None else idx
    gpu = {k: _np(v)[sel] for k, v in out.items()}
    orc = run_oracle_chain(*(_np(x[k])[sel] for k in KEYS), gpu["tokens"], gpu["num_accepted"], workers=workers)
    check_chain(rep, gpu, orc, _np(x["uniforms"])[sel])
    return out


def test_all_rows_path_matches_oracle(sd, hooks):
    hooks(chain_all_rows=1)
    rep = ParityReport("all-rows path chain_b64_v32000 (20 rounds)")
    for r in range(20):
        _check(sd, rep, workloads.chain_workload("chain_b64_v32000", r, DEV))
    assert not rep.failures, rep.failures[:5]
    rep2 = ParityReport("all-rows path chain_b256_v128256 (1 full round)")
    _check(sd, rep2, workloads.chain_workload("chain_b256_v128256", 0, DEV))
    assert not rep2.failures, rep2.failures[:5]
    assert_flag_budget(rep.flagged + rep2.flagged, rep.rows + rep2.rows, (rep.summary(), rep2.summary()))


def test_all_rows_path_greedy_call(sd, hooks):
    from oracle import specdec_oracle as so
    hooks(chain_all_rows=1)
    x = workloads.make_chain_inputs(16, 4, 32000, "bf16", seed=3, device=DEV, scale=1.0, n_spikes=1, spike=3.0,
                                    noise=0.2, temps="const:0.0")
    out = sd.verify_greedy(x["logits"], x["draft_tokens"])
    torch.cuda.synchronize()
    L, d = _np(x["logits"]), _np(x["draft_tokens"])
    for b in range(16):
        o = so.verify_greedy_sequence(L[b], d[b])
        assert int(out["num_accepted"][b]) == o["J"]
        assert np.array_equal(_np(out["tokens"])[b], o["tokens"])


@pytest.mark.parametrize("dtype,V", [("bf16", 1_048_576), ("fp32", 786_432)])
def test_vocabulary_at_the_left_to_right_limit(sd, dtype, V):
    """The largest vocabulary the left-to-right kernel takes (a full chunk table in both
    members): it runs that kernel, and matches the oracle."""
    rep = ParityReport(f"V={V} {dtype} (left-to-right limit)")
    for seed in range(2):
        x = workloads.make_chain_inputs(2, 2, V, dtype, seed=10 + seed, device=DEV, recipe="spikes", scale=2.0,
                                        n_spikes=4, spike=8.0, noise=0.5, temps="const:1.0")
        with sd.KernelTimer() as kt:
            _check(sd, rep, x, workers=1)
            launches = kt.read()
        assert launches["chain_seq"][1] == 1 and launches["chain_stats"][1] == 0, launches
    assert not rep.failures, rep.failures[:5]


@pytest.mark.parametrize("dtype,V", [("bf16", 1_048_576 + 1024), ("fp32", 786_432 + 512)])
def test_vocabulary_beyond_the_left_to_right_limit(sd, dtype, V):
    """One past the left-to-right kernel's chunk table: the all-rows kernels serve it."""
    rep = ParityReport(f"V={V} {dtype}")
    for seed in range(2):
        x = workloads.make_chain_inputs(2, 2, V, dtype, seed=seed, device=DEV, recipe="spikes", scale=2.0,
                                        n_spikes=4, spike=8.0, noise=0.5, temps="const:1.0")
        with sd.KernelTimer() as kt:
            _check(sd, rep, x, workers=1)
            launches = kt.read()
        assert launches["chain_seq"][1] == 0 and launches["chain_stats"][1] == 1, launches
    assert not rep.failures, rep.failures[:5]


def test_wait_that_gives_up_marks_unfinished_sequences(sd):
    x = workloads.chain_workload("chain_b256_v128256", 0, DEV)
    with sd.test_hooks(chain_drop_draws=1, queue_wait_us=300):
        out = sd.verify_chain(*(x[k] for k in KEYS))
        torch.cuda.synchronize()
    st, J, tok, pd = (_np(out[k]) for k in ("status", "num_accepted", "tokens", "p_draft"))
    timed = (st & 0xFF) == sd.STATUS_TIMEOUT
    assert timed.any() and not timed.all(), int(timed.sum())
    assert (J[timed] == -1).all() and (tok[timed] == -1).all() and np.isnan(pd[timed]).all()
    assert (st[timed] == sd.STATUS_TIMEOUT).all()
    # the sequences that finished are exact
    idx = np.flatnonzero(~timed)
    rep = ParityReport("finished sequences under lost draws")
    gpu = {k: _np(v)[idx] for k, v in out.items()}
    orc = run_oracle_chain(*(_np(x[k])[idx] for k in KEYS), gpu["tokens"], gpu["num_accepted"])
    check_chain(rep, gpu, orc, _np(x["uniforms"])[idx])
    assert not rep.failures, rep.failures[:5]
    # the context stays usable: the same call without the hook is exact for every sequence
    rep2 = ParityReport("after the hook")
    _check(sd, rep2, x)
    assert not rep2.failures, rep2.failures[:5]


def test_launch_beside_kernels_that_hold_sms(sd):
    """Kernels on other streams hold SMs for longer than the queue waits' bound (48 bounded
    clock spins of about 0.5 s, one CTA each, the bound shortened to 200 ms by the test
    hook), so part of the left-to-right launch cannot be resident until they end.  The
    teams that are resident must finish every sequence without waiting on the others: the
    outputs equal those of the call on an idle GPU, with no sequence timed out."""
    x = workloads.chain_workload("chain_b256_v128256", 1, DEV)
    ref = sd.verify_chain(*(x[k] for k in KEYS))
    torch.cuda.synchronize()
    sides = [torch.cuda.Stream() for _ in range(48)]
    with sd.test_hooks(queue_wait_us=200_000):
        for sdv in sides:
            with torch.cuda.stream(sdv):
                torch.cuda._sleep(1_000_000_000)  # ~0.5 s of clock cycles
        out = sd.verify_chain(*(x[k] for k in KEYS))
        torch.cuda.synchronize()
    st = _np(out["status"]).astype(np.int64)
    assert not ((st & 0xFF) == sd.STATUS_TIMEOUT).any(), int(((st & 0xFF) == sd.STATUS_TIMEOUT).sum())
    for k in ref:
        a, b = _np(ref[k]), _np(out[k])
        assert np.array_equal(np.nan_to_num(a, nan=-7.0), np.nan_to_num(b, nan=-7.0)), k


def test_two_calls_in_flight_on_two_streams(sd):
    """Two B=256 calls launched back to back on two streams (each with its own workspace)
    compete for SMs; each must equal the same call made alone."""
    xs = [workloads.chain_workload("chain_b256_v128256", r, DEV) for r in (0, 2)]
    refs = [sd.verify_chain(*(x[k] for k in KEYS)) for x in xs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.current_stream().synchronize()
    for rep in range(3):
        outs = [sd.verify_chain(*(x[k] for k in KEYS), stream=s) for x, s in zip(xs, streams)]
        torch.cuda.synchronize()
        for ref, out in zip(refs, outs):
            for k in ref:
                a, b = _np(ref[k]), _np(out[k])
                assert np.array_equal(np.nan_to_num(a, nan=-7.0), np.nan_to_num(b, nan=-7.0)), (rep, k)
